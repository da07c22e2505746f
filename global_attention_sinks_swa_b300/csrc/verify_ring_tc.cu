// MTP verify against the SWA ring buffer on the 5th-generation tensor cores
// (sm_103a), bf16 in/out, fp32 accumulation, D = 128.
//
// The step (release announcement "小米开源 MiMo-V2-Flash", figure "Multi-Token
// Prediction"; technical-report summary, section "MTP加速"): every request
// scores its real token and up to three drafts in one pass, draft t seeing the
// history and drafts 0..t; the SWA layers read a fixed-size cache (section
// "将效率推向极限") -- here a ring of R = W + q_max - 1 slots per (request,
// kv head), position p in slot p mod R.
//
// One CTA per (request, kv head).  Its q_len x G query rows (G = 8 heads of
// the kv group, q_len <= 4 tokens) meet the whole ring in one pass:
//   - the softmax warps copy Q (q_len tokens x 8 heads) into shared memory in
//     the 128-byte-swizzled layout a TMA box would have; TMA loads K and V of
//     all R slots as one box of 144 rows per D half (rows past the ring read 0);
//   - S = Q K^T is one tcgen05.mma group with M = 128: the A descriptor's
//     8-row-group stride is 256 bytes, so MMA rows 32t..32t+7 read token t's
//     8 heads (one 1 KB swizzle atom) and the other rows read unused data
//     whose results are ignored; token t's scores land in TMEM lane quarter t;
//   - warp t runs the softmax of token t's rows (thread = row = TMEM lane),
//     with the running max seeded by the sink logit, and writes P (bf16) over
//     the S columns;
//   - O = P V is a second tcgen05.mma group (P from TMEM, V from shared
//     memory); warp t normalises its rows and stores them.
// Mask: slot s holds position ring_slot_position_r0(s, L, R, L mod R); it is
// visible from query position i iff that position is in [max(0, i-W+1), i],
// i.e. iff s lies in one of the two intervals of ring_visible_slots().
#include "index_math.cuh"
#include "internal.h"
#include "ptx_sm103.cuh"
#include "tc_tile.cuh"

namespace attn {
namespace {
namespace vring {

using namespace tc;

constexpr int kMaxTokens = 4;                     // q_max supported by this kernel
constexpr int kG = 8;                             // query heads per kv head
constexpr int kN = kVerifyRingKeys;               // key rows per D half (R rounded up to 16)
constexpr int kKHalf = kN * kHalfRowBytes;        // 18 KB
constexpr int kQHalf = kMaxTokens * kG * kHalfRowBytes;  // 4 KB
constexpr int kThreads = 160;                     // warps 0-3 softmax/epilogue, warp 4 TMA + MMA
constexpr int kOCol = 96;                         // O accumulator column (P uses 0..71)
constexpr uint32_t kIdescPV = ptx::idesc_bf16(128, 128, false, true);
static_assert(kN % 16 == 0 && kN <= 256 && kOCol >= kN / 2 && kOCol + 128 <= 256, "TMEM layout");

struct __align__(1024) Smem {
    uint8_t q[2][kQHalf];   // [D half][token][head] rows of 128 B
    uint8_t k[2][kKHalf];   // [D half][slot] rows of 128 B
    uint8_t v[2][kKHalf];
    uint64_t q_ready, k_full, v_full, s_full, p_full, o_full, mma_done;
    uint32_t tmem_base;
    int abort;
};

__global__ void __launch_bounds__(kThreads, 2)
    verify_ring_tc_kernel(const __nv_bfloat16 *__restrict__ q,
                          const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tmv,
                          const int32_t *__restrict__ cu_q, const int32_t *__restrict__ seq_lens,
                          const float *__restrict__ sink, __nv_bfloat16 *__restrict__ o, int Hq,
                          int Hkv, int window, int R, int q_max, float scale, unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                         ~static_cast<uintptr_t>(1023));
    const int g = blockIdx.x, b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = cu_q[b], q_len = cu_q[b + 1] - r0, L = seq_lens[b];

    // ---- validate the request (uniform across the CTA)
    if (q_len <= 0) return;
    if (q_len > q_max || q_len > kMaxTokens) {
        if (threadIdx.x == 0 && g == 0) atomicOr(err, 0x4u);
        return;
    }
    if (L < q_len) {
        if (threadIdx.x == 0 && g == 0) atomicOr(err, 0x2u);
        return;
    }

    if (threadIdx.x == 0) {
        ptx::mbar_init(&sm.q_ready, 4);  // one arrival per softmax warp
        ptx::mbar_init(&sm.k_full, 1);
        ptx::mbar_init(&sm.v_full, 1);
        ptx::mbar_init(&sm.mma_done, 1);
        ptx::mbar_init(&sm.s_full, 1);
        ptx::mbar_init(&sm.p_full, 4);  // one arrival per softmax warp
        ptx::mbar_init(&sm.o_full, 1);
        sm.abort = ptx::prior_timeout(err) ? 1 : 0;
        ptx::fence_mbar_init();
    }
    if (warp == 4) {
        ptx::tmem_alloc(&sm.tmem_base, 256);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const bool skip = sm.abort != 0;  // an earlier launch timed out: do nothing

    if (warp == 4) {
        // ----------------------------------------------- TMA loads and MMAs
        if (lane == 0 && !skip) {
            bool ok = true, issued = false;
            ptx::prefetch_tmap(&tmk);
            ptx::prefetch_tmap(&tmv);
            ptx::mbar_arrive_expect_tx(&sm.k_full, 2 * kKHalf);
            for (int hf = 0; hf < 2; ++hf) ptx::tma_load_4d(sm.k[hf], &tmk, hf * 64, 0, g, b, &sm.k_full);
            ptx::mbar_arrive_expect_tx(&sm.v_full, 2 * kKHalf);
            for (int hf = 0; hf < 2; ++hf) ptx::tma_load_4d(sm.v[hf], &tmv, hf * 64, 0, g, b, &sm.v_full);
            // S = Q K^T: A rows 32t + j (j < 8) read token t, head j (8-row
            // group stride 256 B, i.e. group 4t starts at t's 1 KB atom)
            ok = ptx::mbar_wait(&sm.k_full, 0) && ptx::mbar_wait(&sm.q_ready, 0);
            if (ok) {
                ptx::tc_fence_after();
                const uint32_t idS = ptx::idesc_bf16(128, kN, false, false);
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad =
                        ptx::sdesc_sw128(ptx::smem_u32(sm.q[kk >> 2]) + (kk & 3) * 32, 16, 256);
                    ptx::mma_ss(tmem, ad, kmajor_desc(sm.k[kk >> 2], kk & 3), idS, kk > 0 ? 1u : 0u);
                }
                ptx::tc_commit(&sm.s_full);
                issued = true;
                ok = ptx::mbar_wait(&sm.v_full, 0) && ptx::mbar_wait(&sm.p_full, 0);
            }
            if (ok) {  // O = P V, P (bf16) in TMEM columns 0..kN/2-1
                ptx::tc_fence_after();
                for (int kk = 0; kk < kN / 16; ++kk)
                    ptx::mma_ts(tmem + kOCol, tmem + kk * 8, vmajor_desc(sm.v[0], kk, kKHalf), kIdescPV,
                                kk > 0 ? 1u : 0u);
                ptx::tc_commit(&sm.o_full);
            }
            if (!ok) atomicOr(err, kErrWait);
            // copies and MMAs in flight finish before the CTA may exit (bounded)
            ptx::mbar_wait(&sm.k_full, 0);
            ptx::mbar_wait(&sm.v_full, 0);
            if (issued) {
                ptx::tc_commit(&sm.mma_done);
                ptx::mbar_wait(&sm.mma_done, 0);
            }
        }
        __syncwarp();
    } else if (!skip) {
        // ------------------------------------- softmax and epilogue (warp t)
        // Thread = TMEM lane of quarter t; lanes 0..7 hold token t's 8 heads,
        // the other lanes take part in the warp-wide TMEM accesses only.
        const int t = warp, j = lane;
        const bool real = (j < kG) && (t < q_len);
        const uint32_t lane_off = static_cast<uint32_t>(t * 32) << 16;
        const uint32_t tS = tmem + lane_off, tO = tS + kOCol;
        const int qpos = L - q_len + t;
        const int h = g * kG + (j & (kG - 1));
        const float sig = sink[h];
        const float sl2 = scale * kLog2e;
        // Q rows t*8+hh -> shared memory, 128-byte swizzled like a TMA box
        for (int x = threadIdx.x; x < kMaxTokens * kG * 16; x += 4 * 32) {
            const int r = x >> 4, c = x & 15;  // row, 16-byte chunk of its 256 bytes
            const int tt = r / kG, hh = r % kG;
            if (tt < q_len)
                *reinterpret_cast<uint4 *>(sm.q[c >> 3] + r * kHalfRowBytes +
                                           (((c & 7) ^ (r & 7)) << 4)) =
                    *reinterpret_cast<const uint4 *>(
                        q + (static_cast<long>(r0 + tt) * Hq + g * kG + hh) * 128 + c * 8);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.q_ready);
        bool ok = ptx::mbar_wait_warp(&sm.s_full, 0);
        float mb = 0.f, l = 0.f;
        if (ok) {
            ptx::tc_fence_after();
            // visible slots: at most two intervals of slot indices
            const RingVisible vis = ring_visible_slots(L, R, window, qpos);
            auto visible = [&](int c) { return vis.contains(c); };
            // pass 1: masked row max of the raw scores (scale > 0), 48 columns at a time
            float mx = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < kN / 48; ++cc) {
                float x[48];
                tmem_load_row<48>(tS + 48 * cc, x);
#pragma unroll
                for (int i = 0; i < 48; ++i) mx = fmaxf(mx, visible(48 * cc + i) ? x[i] : -INFINITY);
            }
            // seeded with the sink logit; sigma = +inf gives m = +inf and every p = 0
            const float m = fmaxf(sig * kLog2e, mx * sl2);
            mb = (m == -INFINITY) ? 0.f : m;
            // pass 2: P = 2^(s*scale*log2e - m) as bf16 over the S columns (P
            // column c/2 <= S column c, already read)
            float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int cc = 0; cc < kN / 48; ++cc) {
                float x[48];
                tmem_load_row<48>(tS + 48 * cc, x);
#pragma unroll
                for (int i = 0; i < 48; ++i) {
                    x[i] = visible(48 * cc + i) ? ptx::exp2_approx(fmaf(x[i], sl2, -mb)) : 0.f;
                    l4[i & 3] += x[i];
                }
                tmem_store_p<48>(tS + 24 * cc, x);
            }
            ptx::tmem_st_wait();
            l = (l4[0] + l4[1]) + (l4[2] + l4[3]);
        }
        ptx::tc_fence_before();
        if (lane == 0) ptx::mbar_arrive(&sm.p_full);  // also on failure: the issuer stops by itself
        ok = ok && ptx::mbar_wait_warp(&sm.o_full, 0);
        if (ok) {
            ptx::tc_fence_after();
            const bool sink_all = isinf(sig) && sig > 0.f;
            if (!sink_all && !(isinf(sig) && sig < 0.f)) l += ptx::exp2_approx(sig * kLog2e - mb);
            const float inv = sink_all ? 0.f : 1.f / l;
            uint4 *dst = reinterpret_cast<uint4 *>(o + (static_cast<long>(r0 + t) * Hq + h) * 128);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float ov[64];
                tmem_load_row<64>(tO + 64 * hf, ov);
                if (real) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        uint32_t w[4];
#pragma unroll
                        for (int q2 = 0; q2 < 4; ++q2)
                            w[q2] = ptx::pack_bf16x2(ov[8 * i + 2 * q2] * inv, ov[8 * i + 2 * q2 + 1] * inv);
                        dst[8 * hf + i] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
        } else if (lane == 0) {
            atomicOr(err, kErrWait);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 256);
    }
}

}  // namespace vring
}  // namespace

int verify_ring_tc_supported(int G, int R, int q_max) {
    return G == vring::kG && R >= 1 && R <= vring::kN && q_max >= 1 && q_max <= vring::kMaxTokens;
}

cudaError_t launch_verify_ring_tc(const VerifyMaps &maps, const void *q, const int32_t *cu_q,
                                  const int32_t *seq_lens, const float *sink, void *o, int B,
                                  int Hq, int Hkv, int window, int R, int q_max, float scale,
                                  unsigned int *err, cudaStream_t s) {
    if (B == 0) return cudaSuccess;
    const size_t smem = sizeof(vring::Smem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(vring::verify_ring_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    vring::verify_ring_tc_kernel<<<dim3(Hkv, B), vring::kThreads, smem, s>>>(
        static_cast<const __nv_bfloat16 *>(q), maps.k, maps.v, cu_q, seq_lens, sink,
        static_cast<__nv_bfloat16 *>(o), Hq, Hkv, window, R, q_max, scale, err);
    return cudaGetLastError();
}

}  // namespace attn

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
//   - TMA loads Q (one box of 8 heads per token, q_len boxes) and K of all R
//     slots as one box of 144 rows per D half (rows past the ring read 0), and
//     V into the same buffer once S has read K, while the softmax runs -- 44 KB
//     of shared memory and <= 102 registers per thread let 4 CTAs share an SM,
//     so a 64-request x 8-kv-head batch runs in one wave;
//   - S = Q K^T is one tcgen05.mma group with M = 128: the A descriptor's
//     8-row-group stride is 256 bytes, so MMA rows 32t..32t+7 read token t's
//     8 heads (one 1 KB swizzle atom) and the other rows read unused data
//     whose results are ignored; token t's scores land in TMEM lane quarter t;
//   - warp t runs the softmax of token t's rows, four threads per row through
//     the 16-lane TMEM load/store shapes, with the max seeded by the sink
//     logit, and writes P (bf16) over the S columns;
//   - O = P V is a second tcgen05.mma group (P from TMEM, V from shared
//     memory); warp t normalises its rows and stores them.
// Mask: slot s holds position ring_slot_position_r0(s, L, R, L mod R); it is
// visible from query position i iff that position is in [max(0, i-W+1), i],
// i.e. iff s lies in one of the two intervals of ring_visible_slots().
#include "index_math.cuh"
#include "internal.h"
#include "ptx_sm103.cuh"
#include "tc_tile.cuh"

#include <type_traits>

namespace attn {
namespace {
namespace vring {

using namespace tc;

// Bits of the slots [a, a + n) that fall in the 32-slot word starting at base.
ATTN_DEV uint32_t interval_bits(int a, int n, int base) {
    const int lo = max(a - base, 0), hi = min(a + n - base, 32);
    if (hi <= lo) return 0u;
    const uint32_t span = (hi - lo == 32) ? 0xffffffffu : ((1u << (hi - lo)) - 1u);
    return span << lo;
}

constexpr int kMaxTokens = 4;                     // q_max supported by this kernel
constexpr int kG = 8;                             // query heads per kv head
constexpr int kN = kVerifyRingKeys;               // key rows per D half (R rounded up to 16)
constexpr int kKHalf = kN * kHalfRowBytes;        // 18 KB
constexpr int kQHalf = kMaxTokens * kG * kHalfRowBytes;  // 4 KB
constexpr int kThreads = 160;                     // warps 0-3 softmax/epilogue, warp 4 TMA + MMA
constexpr int kOCol = 96;                         // O accumulator column (P uses 0..71)
constexpr uint32_t kIdescPV = ptx::idesc_bf16(128, 128, false, true);
static_assert(kN % 16 == 0 && kN <= 256 && kOCol >= kN / 2 && kOCol + 128 <= 256, "TMEM layout");
static_assert(kN == 8 * (8 + 8 + 2), "the softmax walks 18 repetitions of 8 columns: x8, x8, x2");

struct __align__(1024) Smem {
    uint8_t q[2][kQHalf];   // [D half][token][head] rows of 128 B
    uint8_t kv[2][kKHalf];  // [D half][slot] rows of 128 B: K, then V
    uint64_t q_ready, k_full, v_full, s_full, s_done, p_full, o_full, mma_done;
    uint32_t tmem_base;
    int abort;
};

__global__ void __launch_bounds__(kThreads, 4)
    verify_ring_tc_kernel(const __grid_constant__ CUtensorMap tmq,
                          const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tmv,
                          const int32_t *__restrict__ cu_q, const int32_t *__restrict__ seq_lens,
                          const float *__restrict__ sink, __nv_bfloat16 *__restrict__ o, int Hq,
                          int Hkv, int window, int R, int q_max, int q_rows, float scale,
                          unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                         ~static_cast<uintptr_t>(1023));
    const int g = blockIdx.x, b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = cu_q[b], q_len = cu_q[b + 1] - r0, L = seq_lens[b];

    // ---- validate the request (uniform across the CTA)
    if (q_len <= 0) return;
    if (q_len > q_max || q_len > kMaxTokens || r0 < 0 || r0 + q_len > q_rows) {
        if (threadIdx.x == 0 && g == 0) atomicOr(err, 0x4u);
        return;
    }
    if (L < q_len) {
        if (threadIdx.x == 0 && g == 0) atomicOr(err, 0x2u);
        return;
    }

    if (threadIdx.x == 0) {
        ptx::mbar_init(&sm.q_ready, 1);
        ptx::mbar_init(&sm.k_full, 1);
        ptx::mbar_init(&sm.v_full, 1);
        ptx::mbar_init(&sm.mma_done, 1);
        ptx::mbar_init(&sm.s_full, 1);
        ptx::mbar_init(&sm.s_done, 1);
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
            ptx::prefetch_tmap(&tmq);
            ptx::prefetch_tmap(&tmk);
            ptx::prefetch_tmap(&tmv);
            // Q: token t's 8 heads (1 KB per D half) at row group t
            ptx::mbar_arrive_expect_tx(&sm.q_ready, 2 * q_len * kG * kHalfRowBytes);
            for (int tt = 0; tt < q_len; ++tt)
                for (int hf = 0; hf < 2; ++hf)
                    ptx::tma_load_3d(sm.q[hf] + tt * kG * kHalfRowBytes, &tmq, hf * 64, g * kG, r0 + tt,
                                     &sm.q_ready);
            ptx::mbar_arrive_expect_tx(&sm.k_full, 2 * kKHalf);
            for (int hf = 0; hf < 2; ++hf) ptx::tma_load_4d(sm.kv[hf], &tmk, hf * 64, 0, g, b, &sm.k_full);
            // S = Q K^T: A rows 32t + j (j < 8) read token t, head j (8-row
            // group stride 256 B, i.e. group 4t starts at t's 1 KB atom)
            ok = ptx::mbar_wait(&sm.k_full, 0) && ptx::mbar_wait(&sm.q_ready, 0);
            if (ok) {
                ptx::tc_fence_after();
                const uint32_t idS = ptx::idesc_bf16(128, kN, false, false);
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad =
                        ptx::sdesc_sw128(ptx::smem_u32(sm.q[kk >> 2]) + (kk & 3) * 32, 16, 256);
                    ptx::mma_ss(tmem, ad, kmajor_desc(sm.kv[kk >> 2], kk & 3), idS, kk > 0 ? 1u : 0u);
                }
                ptx::tc_commit(&sm.s_full);
                ptx::tc_commit(&sm.s_done);
                issued = true;
                // V replaces K once S has read it
                ok = ptx::mbar_wait(&sm.s_done, 0);
                if (ok) {
                    ptx::mbar_arrive_expect_tx(&sm.v_full, 2 * kKHalf);
                    for (int hf = 0; hf < 2; ++hf)
                        ptx::tma_load_4d(sm.kv[hf], &tmv, hf * 64, 0, g, b, &sm.v_full);
                }
                ok = ok && ptx::mbar_wait(&sm.v_full, 0) && ptx::mbar_wait(&sm.p_full, 0);
            }
            if (ok) {  // O = P V, P (bf16) in TMEM columns 0..kN/2-1
                ptx::tc_fence_after();
                for (int kk = 0; kk < kN / 16; ++kk)
                    ptx::mma_ts(tmem + kOCol, tmem + kk * 8, vmajor_desc(sm.kv[0], kk, kKHalf), kIdescPV,
                                kk > 0 ? 1u : 0u);
                ptx::tc_commit(&sm.o_full);
            }
            if (!ok) atomicOr(err, kErrWait);
            // copies and MMAs in flight finish before the CTA may exit (bounded)
            ptx::mbar_wait(&sm.q_ready, 0);
            ptx::mbar_wait(&sm.k_full, 0);
            if (issued) ptx::mbar_wait(&sm.v_full, 0);
            if (issued) {
                ptx::tc_commit(&sm.mma_done);
                ptx::mbar_wait(&sm.mma_done, 0);
            }
        }
        __syncwarp();
    } else if (!skip) {
        // ------------------------------------- softmax and epilogue (warp t)
        // Warp t handles token t, whose 8 heads are TMEM lanes 0..7 of quarter
        // t.  The 16-lane TMEM shapes give each row to a quad of threads:
        // thread 4q + r holds columns 8k + 2r and 8k + 2r + 1 (k = 0, 1, ..)
        // of row q (16x256b), and the bf16 pair of exactly those two keys is
        // P column 4k + r (16x128b).  Lanes 8..15 are read and written but
        // unused; lanes 16..31 are not touched.
        const int t = warp, qrow = lane >> 2, r = lane & 3;
        const bool real = t < q_len;
        const uint32_t lane_off = static_cast<uint32_t>(t * 32) << 16;
        const uint32_t tS = tmem + lane_off, tO = tS + kOCol;
        const int qpos = L - q_len + t;
        const int h = g * kG + qrow;
        const float sig = sink[h];
        const float sl2 = scale * kLog2e;
        bool ok = ptx::mbar_wait_warp(&sm.s_full, 0);
        float mb = 0.f, l = 0.f;
        if (ok) {
            ptx::tc_fence_after();
            // visible slots: at most two intervals, the same for the whole
            // warp; as bitmask words pre-shifted by 2r, the two keys of
            // repetition k are bits 8(k%4) and 8(k%4)+1 of word k/4
            const RingVisible vis = ring_visible_slots(L, R, window, qpos);
            uint32_t vm[kN / 32 + 1];
#pragma unroll
            for (int w = 0; w <= kN / 32; ++w)
                vm[w] = (interval_bits(vis.a1, vis.n1, 32 * w) | interval_bits(vis.a2, vis.n2, 32 * w)) >>
                        (2 * r);
            auto vis_bit = [&](int k, int e) { return ((vm[k >> 2] >> (8 * (k & 3) + e)) & 1u) != 0u; };
            // pass 1: masked max of the raw scores (scale > 0) over the quad
            float mx = -INFINITY;
            auto max_reps = [&](auto reps, int k0) {
                constexpr int NR = decltype(reps)::value;
                uint32_t v[4 * NR];
                if constexpr (NR == 8) ptx::tmem_ld_16x256b_x8(tS + 8 * k0, v);
                else ptx::tmem_ld_16x256b_x2(tS + 8 * k0, v);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                for (int k = 0; k < NR; ++k)
                    mx = fmax3(mx, vis_bit(k0 + k, 0) ? __uint_as_float(v[4 * k]) : -INFINITY,
                               vis_bit(k0 + k, 1) ? __uint_as_float(v[4 * k + 1]) : -INFINITY);
            };
            max_reps(std::integral_constant<int, 8>{}, 0);
            max_reps(std::integral_constant<int, 8>{}, 8);
            max_reps(std::integral_constant<int, 2>{}, 16);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            // seeded with the sink logit; sigma = +inf gives m = +inf and every p = 0
            const float m = fmaxf(sig * kLog2e, mx * sl2);
            mb = (m == -INFINITY) ? 0.f : m;
            // pass 2: P = 2^(s*scale*log2e - m); the pair of repetition k is P
            // column 4k + r (written over S columns already read)
            float ls = 0.f;
            auto p_reps = [&](auto reps, int k0) {
                constexpr int NR = decltype(reps)::value;
                uint32_t v[4 * NR], pw[2 * NR];
                if constexpr (NR == 8) ptx::tmem_ld_16x256b_x8(tS + 8 * k0, v);
                else ptx::tmem_ld_16x256b_x2(tS + 8 * k0, v);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                for (int k = 0; k < NR; ++k) {
                    const float p0 = vis_bit(k0 + k, 0)
                                         ? ptx::exp2_approx(fmaf(__uint_as_float(v[4 * k]), sl2, -mb))
                                         : 0.f;
                    const float p1 = vis_bit(k0 + k, 1)
                                         ? ptx::exp2_approx(fmaf(__uint_as_float(v[4 * k + 1]), sl2, -mb))
                                         : 0.f;
                    ls += p0 + p1;
                    pw[2 * k] = ptx::pack_bf16x2(p0, p1);
                    pw[2 * k + 1] = 0u;  // lane q + 8: unused row
                }
                if constexpr (NR == 8) ptx::tmem_st_16x128b_x8(tS + 4 * k0, pw);
                else ptx::tmem_st_16x128b_x2(tS + 4 * k0, pw);
            };
            p_reps(std::integral_constant<int, 8>{}, 0);
            p_reps(std::integral_constant<int, 8>{}, 8);
            p_reps(std::integral_constant<int, 2>{}, 16);
            ptx::tmem_st_wait();
            ls += __shfl_xor_sync(0xffffffffu, ls, 1);
            ls += __shfl_xor_sync(0xffffffffu, ls, 2);
            l = ls;
        }
        ptx::tc_fence_before();
        if (lane == 0) ptx::mbar_arrive(&sm.p_full);  // also on failure: the issuer stops by itself
        ok = ok && ptx::mbar_wait_warp(&sm.o_full, 0);
        if (ok) {
            ptx::tc_fence_after();
            const bool sink_all = isinf(sig) && sig > 0.f;
            if (!sink_all && !(isinf(sig) && sig < 0.f)) l += ptx::exp2_approx(sig * kLog2e - mb);
            const float inv = sink_all ? 0.f : 1.f / l;
            // O row q: thread 4q + r holds columns 8k + 2r, +1 and stores them
            // as one bf16 pair
            uint32_t *dst = reinterpret_cast<uint32_t *>(o + (static_cast<long>(r0 + t) * Hq + h) * 128) + r;
#pragma unroll
            for (int k0 = 0; k0 < 16; k0 += 8) {
                uint32_t v[32];
                ptx::tmem_ld_16x256b_x8(tO + 8 * k0, v);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                if (real) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        dst[4 * (k0 + k)] = ptx::pack_bf16x2(__uint_as_float(v[4 * k]) * inv,
                                                             __uint_as_float(v[4 * k + 1]) * inv);
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

cudaError_t launch_verify_ring_tc(const VerifyMaps &maps, const int32_t *cu_q,
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
        maps.q, maps.k, maps.v, cu_q, seq_lens, sink, static_cast<__nv_bfloat16 *>(o), Hq, Hkv,
        window, R, q_max, B * q_max, scale, err);
    return cudaGetLastError();
}

}  // namespace attn

// bf16 sink-attention prefill on the 5th-generation tensor cores (sm_103a).
//
// The kernel computes, for every query row, softmax over the visible scores
// plus one sink column per query head (no value), times V:
//   technical-report summary (fanfer.top, "MiMo-V2"), section "Hybrid Sliding
//   Window Attention Architecture" (learnable gpt-oss-style sink bias) and
//   section "MiMo-V2-Flash Model Architecture" (W = 128 SWA layers, 1-in-6
//   global-attention layers).
//
// Building blocks: TMA (cp.async.bulk.tensor) stages 128-byte-swizzled tiles
// of Q, K, V in shared memory; one thread issues tcgen05.mma (kind::f16, bf16
// operands, fp32 accumulators in tensor memory) for S = Q K^T from shared
// memory and for O += P V with P read from tensor memory; softmax warps own
// one row each (tensor-memory lane = row), load S with tcgen05.ld, run the
// online softmax in registers with the running max seeded by the sink logit
// and the running sum by the sink's own term, and write P back as bf16 with
// tcgen05.st over the S columns.
//
// GA tiling: a CTA owns two consecutive 128-row query tiles of one
// head and streams 128-key tiles of K and V through a two-stage ring; the two
// softmax warpgroups ping-pong so that one tile's exponentials overlap the
// other tile's MMAs.  Causal (and window) tile skipping comes from
// ga_key_tiles(); only tiles crossing the diagonal or window edge are masked.
// The running max is raised lazily (only when it grows by more than 2^8), so
// the O accumulator in tensor memory is rarely rescaled.
//
// The sliding-window layers with 8 query heads per kv head use the streaming
// kernel in prefill_swa.cu; this kernel serves every other window and head ratio.
#include "index_math.cuh"
#include "internal.h"
#include "ptx_sm103.cuh"
#include "tc_tile.cuh"

namespace attn {
namespace {

using namespace tc;

constexpr float kRescaleLog2 = 8.0f;   // lazy-rescale threshold (log2 units)

// Epilogue helper: this thread's output row (128 fp32 in TMEM at taddr) times
// inv -> bf16 -> two 128B-swizzled smem halves (row `row` of a 128-row tile).
ATTN_DEV void store_o_row_smem(uint32_t taddr, float inv, uint8_t *half0, uint8_t *half1,
                               int row) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        ptx::tmem_ld32(taddr + c * 32, r);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        reg_dep(r);
        uint8_t *half = (c < 2) ? half0 : half1;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {  // 4 chunks of 8 columns = 16 B each
            const int lc = (c & 1) * 4 + ch;  // logical 16-byte chunk within the 128-byte row
            uint4 v;
            v.x = ptx::pack_bf16x2(__uint_as_float(r[ch * 8 + 0]) * inv, __uint_as_float(r[ch * 8 + 1]) * inv);
            v.y = ptx::pack_bf16x2(__uint_as_float(r[ch * 8 + 2]) * inv, __uint_as_float(r[ch * 8 + 3]) * inv);
            v.z = ptx::pack_bf16x2(__uint_as_float(r[ch * 8 + 4]) * inv, __uint_as_float(r[ch * 8 + 5]) * inv);
            v.w = ptx::pack_bf16x2(__uint_as_float(r[ch * 8 + 6]) * inv, __uint_as_float(r[ch * 8 + 7]) * inv);
            *reinterpret_cast<uint4 *>(half + row * kHalfRowBytes + ((lc ^ (row & 7)) << 4)) = v;
        }
    }
}

// =========================================================== GA-tiled kernel
namespace ga {

constexpr int kThreads = 320;  // WG0, WG1 (softmax), warp 8 TMA, warp 9 MMA
constexpr int kTile = 128 * kHalfRowBytes;  // one 128-row D half: 16 KB
constexpr uint32_t kIdescS = ptx::idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescPV = ptx::idesc_bf16(128, 128, false, true);

struct __align__(1024) Smem {
    uint8_t q[2][2][kTile];  // [query tile][D half]; reused to stage O
    uint8_t k[2][2][kTile];  // [stage][D half]
    uint8_t v[2][2][kTile];
    uint64_t q_full;
    uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
    uint64_t s_full[2], p_full[2], o_full[2];
    uint32_t tmem_base;
    int abort;
};

__global__ void __launch_bounds__(kThreads, 1)
    prefill_ga_kernel(const __grid_constant__ CUtensorMap tmq,
                      const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv,
                      const __grid_constant__ CUtensorMap tmo, __nv_bfloat16 *__restrict__ out,
                      const float *__restrict__ sink, float *__restrict__ lse,
                      const int32_t *__restrict__ cu, int B, int T, int total, int Hq, int Hkv,
                      int window, float scale, float vscale, unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                         ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // block -> (pair, head, sequence) in ga_block_coords order: one kv head's
    // query heads together, heaviest (latest) pairs first.  T bounds every
    // sequence: pairs past a sequence's end exit.
    const int npairs = (T + 255) / 256;
    int pair, h, b;
    ga_block_coords(static_cast<int>(blockIdx.x), npairs, Hq, Hkv, &pair, &h, &b);
    const int g = h / (Hq / Hkv);
    const int q0 = pair * 256;
    const SeqSpan span = seq_span(cu, b, T, total);
    if (q0 >= span.len) {  // uniform over the block: nothing to do
        if (!span.ok && pair == npairs - 1 && h == 0 && threadIdx.x == 0) atomicOr(err, kErrSeqlens);
        return;
    }
    const int len = span.len, start = span.start;
    int first[2], last[2];
    bool live[2];
    for (int t = 0; t < 2; ++t) {
        live[t] = q0 + 128 * t < len;
        ga_key_tiles(q0 + 128 * t, len, window, &first[t], &last[t]);
    }
    if (!live[1]) { first[1] = first[0]; last[1] = first[0] - 1; }  // empty range
    const int jf = first[0];
    const int jl = live[1] ? (last[1] > last[0] ? last[1] : last[0]) : last[0];

    if (threadIdx.x == 0) {
        ptx::mbar_init(&sm.q_full, 1);
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&sm.k_full[i], 1);
            ptx::mbar_init(&sm.k_empty[i], 1);
            ptx::mbar_init(&sm.v_full[i], 1);
            ptx::mbar_init(&sm.v_empty[i], 1);
            ptx::mbar_init(&sm.s_full[i], 1);
            ptx::mbar_init(&sm.p_full[i], 128);
            ptx::mbar_init(&sm.o_full[i], 1);
        }
        sm.abort = ptx::prior_timeout(err) ? 1 : 0;
        ptx::fence_mbar_init();
    }
    if (warp == 9) {
        ptx::tmem_alloc(&sm.tmem_base, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const bool skip = sm.abort != 0;  // an earlier launch timed out: do nothing

    if (warp == 8) {
        // ------------------------------------------------------------ TMA
        if (lane == 0 && !skip) {
            bool ok = true;
            ptx::prefetch_tmap(&tmq);
            ptx::prefetch_tmap(&tmk);
            ptx::prefetch_tmap(&tmv);
            const int ntl = live[1] ? 2 : 1;
            ptx::mbar_arrive_expect_tx(&sm.q_full, 2 * ntl * kTile);
            for (int t = 0; t < ntl; ++t)
                for (int hf = 0; hf < 2; ++hf)
                    ptx::tma_load_3d(sm.q[t][hf], &tmq, hf * 64, h, start + q0 + 128 * t, &sm.q_full);
            for (int j = jf; ok && j <= jl; ++j) {
                const int n = j - jf, st = n & 1;
                if (n >= 2 && !ptx::mbar_wait(&sm.k_empty[st], ((n >> 1) - 1) & 1)) { ok = false; break; }
                ptx::mbar_arrive_expect_tx(&sm.k_full[st], 2 * kTile);
                for (int hf = 0; hf < 2; ++hf)
                    ptx::tma_load_3d(sm.k[st][hf], &tmk, hf * 64, g, start + j * 128, &sm.k_full[st]);
                if (n >= 2 && !ptx::mbar_wait(&sm.v_empty[st], ((n >> 1) - 1) & 1)) { ok = false; break; }
                ptx::mbar_arrive_expect_tx(&sm.v_full[st], 2 * kTile);
                for (int hf = 0; hf < 2; ++hf)
                    ptx::tma_load_3d(sm.v[st][hf], &tmv, hf * 64, g, start + j * 128, &sm.v_full[st]);
            }
            if (!ok) atomicOr(err, kErrWait);
        }
        __syncwarp();
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA
        if (lane == 0 && !skip) {
            const uint32_t tS[2] = {tmem, tmem + 256};
            const uint32_t tO[2] = {tmem + 128, tmem + 384};
            auto issue_s = [&](int t, int st) {
                for (int kk = 0; kk < 8; ++kk)
                    ptx::mma_ss(tS[t], kmajor_desc(sm.q[t][kk >> 2], kk & 3),
                                kmajor_desc(sm.k[st][kk >> 2], kk & 3), kIdescS, kk > 0);
                ptx::tc_commit(&sm.s_full[t]);
            };
            auto active = [&](int t, int j) { return live[t] && j >= first[t] && j <= last[t]; };
            bool ok = ptx::mbar_wait(&sm.q_full, 0) && ptx::mbar_wait(&sm.k_full[0], 0);
            if (ok) {
                ptx::tc_fence_after();
                for (int t = 0; t < 2; ++t)
                    if (active(t, jf)) issue_s(t, 0);
                ptx::tc_commit(&sm.k_empty[0]);
            }
            for (int j = jf; ok && j <= jl; ++j) {
                const int n = j - jf, st = n & 1;
                const bool more = j + 1 <= jl;
                const int st1 = (n + 1) & 1;
                ok = ptx::mbar_wait(&sm.v_full[st], (n >> 1) & 1) &&
                     (!more || ptx::mbar_wait(&sm.k_full[st1], ((n + 1) >> 1) & 1));
                for (int t = 0; ok && t < 2; ++t) {
                    if (active(t, j)) {
                        const int nt = j - first[t];
                        if (!ptx::mbar_wait(&sm.p_full[t], nt & 1)) { ok = false; break; }
                        ptx::tc_fence_after();
                        for (int kk = 0; kk < 8; ++kk)
                            ptx::mma_ts(tO[t], tS[t] + kk * 8, vmajor_desc(sm.v[st][0], kk, kTile),
                                        kIdescPV, (nt > 0 || kk > 0) ? 1u : 0u);
                        ptx::tc_commit(&sm.o_full[t]);
                    }
                    if (more && active(t, j + 1)) issue_s(t, st1);
                }
                if (ok) {
                    ptx::tc_commit(&sm.v_empty[st]);
                    if (more) ptx::tc_commit(&sm.k_empty[st1]);
                }
            }
            if (!ok) atomicOr(err, kErrWait);
        }
        __syncwarp();
    } else if (live[warp >> 2] && !skip) {
        // ------------------------------------------------ softmax warpgroups
        // Every failure decision is warp-uniform and the warpgroup's named
        // barrier is always reached, so an error unwinds without a hang.
        const int t = warp >> 2;               // query tile of this warpgroup
        const int row = threadIdx.x & 127;     // TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + 256 * t + lane_off, tO = tS + 128;
        const int qs = q0 + 128 * t, qpos = qs + row;
        const float sig = sink[h];
        const float sl2 = scale * kLog2e;
        float m = sig * kLog2e;                 // running max, log2 units
        float l = isinf(sig) && sig < 0.f ? 0.f : 1.f;  // running sum incl. the sink term
        bool ok = true;
        for (int j = first[t]; j <= last[t]; ++j) {
            const int nt = j - first[t];
            if (!ptx::mbar_wait_warp(&sm.s_full[t], nt & 1)) { ok = false; break; }
            ptx::tc_fence_after();
            float x[128];
            tmem_load_row<128>(tS, x);
            // row max of the raw scores (scale > 0 commutes with max), four
            // independent partial maxima; masked entries become -inf
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (ga_tile_needs_mask(qs, j, window)) {
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    x[c] = key_visible(qpos, j * 128 + c, window) ? x[c] : -INFINITY;
                    m4[c & 3] = fmaxf(m4[c & 3], x[c]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 128; ++c) m4[c & 3] = fmaxf(m4[c & 3], x[c]);
            }
            const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl2;
            // lazy max: raise m only when the tile max exceeds it by > 2^8
            const bool grow = mx > m + kRescaleLog2;
            const bool any_grow = __any_sync(0xffffffffu, grow);
            const float mn = grow ? mx : m;
            const float alpha = grow ? ptx::exp2_approx(m - mn) : 1.f;  // 0 when m = -inf
            l *= alpha;
            m = mn;
            const float mb = (m == -INFINITY) ? 0.f : m;
            // P = 2^(s*scale*log2e - m) as bf16 over the S columns; paired fp32
            // arithmetic, partial sums of the columns j mod 4 (l2[j>>1], half j&1)
            const uint64_t sl2x2 = f2(sl2, sl2), nmb = f2(-mb, -mb);
            uint64_t l2[2] = {0, 0};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float2 a = f2_split(f2_fma(f2(x[32 * c + 2 * i], x[32 * c + 2 * i + 1]), sl2x2, nmb));
                    const float p0 = ptx::exp2_approx(a.x), p1 = ptx::exp2_approx(a.y);
                    l2[i & 1] = f2_add(l2[i & 1], f2(p0, p1));
                    pk[i] = ptx::pack_bf16x2(p0, p1);
                }
                ptx::tmem_st16(tS + 16 * c, pk);
            }
            const float2 la = f2_split(l2[0]), lb = f2_split(l2[1]);
            l += (la.x + la.y) + (lb.x + lb.y);
            if (any_grow && nt > 0) {  // rescale the O accumulator after the previous PV
                if (!ptx::mbar_wait_warp(&sm.o_full[t], (nt - 1) & 1)) { ok = false; break; }
                ptx::tc_fence_after();
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
                    ptx::tmem_ld32(tO + c * 32, r);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                    reg_dep(r);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                    ptx::tmem_st32(tO + c * 32, r);
                }
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&sm.p_full[t]);
        }
        const int nlast = last[t] - first[t];
        ok = ok && ptx::mbar_wait_warp(&sm.o_full[t], nlast & 1);
        if (ok) {
            ptx::tc_fence_after();
            const float inv = (l > 0.f) ? vscale / l : 0.f;  // the value scale rides on 1/l
            store_o_row_smem(tO, inv, sm.q[t][0], sm.q[t][1], row);
            ptx::fence_proxy_async_smem();
        } else if (lane == 0) {
            atomicOr(err, kErrWait);
        }
        const bool wg_fail = ptx::named_bar_or(1 + t, 128, !ok);
        if (qs + 128 <= len) {  // a whole tile: one TMA store per D half
            if (row == 0 && !wg_fail) {
                for (int hf = 0; hf < 2; ++hf)
                    ptx::tma_store_3d(&tmo, sm.q[t][hf], hf * 64, h, start + qs);
                ptx::bulk_commit();
                ptx::bulk_wait_read0();
            }
        } else if (ok && qpos < len) {  // the sequence ends inside the tile: own row only
            uint4 *dst = reinterpret_cast<uint4 *>(out + (static_cast<long>(start + qpos) * Hq + h) * 128);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                for (int lc = 0; lc < 8; ++lc)
                    dst[hf * 8 + lc] = *reinterpret_cast<const uint4 *>(
                        sm.q[t][hf] + row * kHalfRowBytes + ((lc ^ (row & 7)) << 4));
        }
        if (ok && lse && qpos < len)
            lse[lse_index(cu, b, h, qpos, start, T, total, Hq)] =
                (m == INFINITY) ? INFINITY : (m + log2f(l)) * kLn2;
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

}  // namespace ga

}  // namespace

cudaError_t launch_prefill_ga_tc(const PrefillMaps &maps, const float *sink, float *lse,
                                 const PrefillBatch &pb, int Hq, int Hkv, int window, float scale,
                                 float vscale, unsigned int *err, cudaStream_t s) {
    if (pb.B == 0 || pb.T == 0 || pb.total == 0) return cudaSuccess;
    const size_t smem = sizeof(ga::Smem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(ga::prefill_ga_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const long blocks = static_cast<long>((pb.T + 255) / 256) * Hq * pb.B;
    ga::prefill_ga_kernel<<<static_cast<unsigned>(blocks), ga::kThreads, smem, s>>>(
        maps.q, maps.k, maps.v, maps.o, static_cast<__nv_bfloat16 *>(maps.out), sink, lse, pb.cu,
        pb.B, pb.T, pb.total, Hq, Hkv, window, scale, vscale, err);
    return cudaGetLastError();
}

}  // namespace attn

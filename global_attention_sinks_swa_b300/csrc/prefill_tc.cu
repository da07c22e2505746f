// bf16 sink-attention prefill on the 5th-generation tensor cores (sm_103a).
//
// Both kernels compute, for every query row, softmax over the visible scores
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
// Kernel 1, "GA-tiled": a CTA owns two consecutive 128-row query tiles of one
// head and streams 128-key tiles of K and V through a two-stage ring; the two
// softmax warpgroups ping-pong so that one tile's exponentials overlap the
// other tile's MMAs.  Causal (and window) tile skipping comes from
// ga_key_tiles(); only tiles crossing the diagonal or window edge are masked.
// The running max is raised lazily (only when it grows by more than 2^8), so
// the O accumulator in tensor memory is rarely rescaled.
//
// Kernel 2, "packed SWA": a tile is 128/G consecutive tokens x the G query
// heads sharing one kv head (GQA packing), against one key tile of
// round_up(128/G + W - 1, 16) keys (144 for G = 8, W = 128) that covers every
// key its rows can see, so each query tile touches exactly one K/V tile.
// Persistent CTAs (one per SM) alternate two tile slots; the O tile is staged
// in the slot's V buffer and written with a TMA store.
#include "index_math.cuh"
#include "internal.h"
#include "ptx_sm103.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned kErrWait = 0x8u;
constexpr float kRescaleLog2 = 8.0f;   // lazy-rescale threshold (log2 units)
constexpr int kHalfRowBytes = 128;     // one D half (64 bf16) per smem row

ATTN_DEV void reg_dep(uint32_t (&r)[32]) {
    asm volatile("" : ATTN_P8(0), ATTN_P8(8), ATTN_P8(16), ATTN_P8(24) : : "memory");
}
ATTN_DEV void reg_dep(uint32_t (&r)[16]) {
    asm volatile("" : ATTN_P8(0), ATTN_P8(8) : : "memory");
}

// Loads N (multiple of 16) fp32 columns of this thread's TMEM lane.
template <int N>
ATTN_DEV void tmem_load_row(uint32_t taddr, float (&x)[N]) {
    uint32_t r[N / 32 > 0 ? N / 32 : 1][32];
    uint32_t t[16];
#pragma unroll
    for (int c = 0; c < N / 32; ++c) ptx::tmem_ld32(taddr + c * 32, r[c]);
    if constexpr (N % 32) ptx::tmem_ld16(taddr + (N / 32) * 32, t);
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int c = 0; c < N / 32; ++c) {
        reg_dep(r[c]);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(r[c][i]);
    }
    if constexpr (N % 32) {
        reg_dep(t);
#pragma unroll
        for (int i = 0; i < 16; ++i) x[(N / 32) * 32 + i] = __uint_as_float(t[i]);
    }
}

// Writes P (N fp32 values) as N/2 packed bf16x2 columns at taddr.
template <int N>
ATTN_DEV void tmem_store_p(uint32_t taddr, const float (&p)[N]) {
#pragma unroll
    for (int c = 0; c < N / 32; ++c) {
        uint32_t r[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = ptx::pack_bf16x2(p[c * 32 + 2 * i], p[c * 32 + 2 * i + 1]);
        ptx::tmem_st16(taddr + c * 16, r);
    }
    if constexpr (N % 32) {
        static_assert(N % 32 == 16, "N must be a multiple of 16");
        constexpr int base = (N / 32) * 32;
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                taddr + base / 2),
            "r"(ptx::pack_bf16x2(p[base + 0], p[base + 1])),
            "r"(ptx::pack_bf16x2(p[base + 2], p[base + 3])),
            "r"(ptx::pack_bf16x2(p[base + 4], p[base + 5])),
            "r"(ptx::pack_bf16x2(p[base + 6], p[base + 7])),
            "r"(ptx::pack_bf16x2(p[base + 8], p[base + 9])),
            "r"(ptx::pack_bf16x2(p[base + 10], p[base + 11])),
            "r"(ptx::pack_bf16x2(p[base + 12], p[base + 13])),
            "r"(ptx::pack_bf16x2(p[base + 14], p[base + 15]))
            : "memory");
    }
}

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

// K-major operand tile (rows of 128 B, 8-row groups 1024 B apart), advanced by
// kk 16-element steps inside the 128-byte swizzle span.
ATTN_DEV uint64_t kmajor_desc(const uint8_t *tile, int kk) {
    return ptx::sdesc_sw128(ptx::smem_u32(tile) + kk * 32, 16, 1024);
}
// MN-major V tile: 16 keys per step (2048 B), D halves `half_stride` apart.
ATTN_DEV uint64_t vmajor_desc(const uint8_t *tile, int kk, uint32_t half_stride) {
    return ptx::sdesc_sw128(ptx::smem_u32(tile) + kk * 2048, half_stride, 1024);
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
                      const __grid_constant__ CUtensorMap tmo, const float *__restrict__ sink,
                      float *__restrict__ lse, int B, int T, int Hq, int Hkv, int window,
                      float scale, unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                         ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // block -> (pair, head, batch); heaviest (latest) pairs first for causal balance
    const int npairs = (T + 255) / 256;
    const int per = Hq * B;
    const int pair = npairs - 1 - static_cast<int>(blockIdx.x) / per;
    const int h = static_cast<int>(blockIdx.x) % Hq;
    const int b = (static_cast<int>(blockIdx.x) / Hq) % B;
    const int g = h / (Hq / Hkv);
    const int q0 = pair * 256;
    int first[2], last[2];
    bool live[2];
    for (int t = 0; t < 2; ++t) {
        live[t] = q0 + 128 * t < T;
        ga_key_tiles(q0 + 128 * t, T, window, &first[t], &last[t]);
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
                    ptx::tma_load_4d(sm.q[t][hf], &tmq, hf * 64, h, q0 + 128 * t, b, &sm.q_full);
            for (int j = jf; ok && j <= jl; ++j) {
                const int n = j - jf, st = n & 1;
                if (n >= 2 && !ptx::mbar_wait(&sm.k_empty[st], ((n >> 1) - 1) & 1)) { ok = false; break; }
                ptx::mbar_arrive_expect_tx(&sm.k_full[st], 2 * kTile);
                for (int hf = 0; hf < 2; ++hf)
                    ptx::tma_load_4d(sm.k[st][hf], &tmk, hf * 64, g, j * 128, b, &sm.k_full[st]);
                if (n >= 2 && !ptx::mbar_wait(&sm.v_empty[st], ((n >> 1) - 1) & 1)) { ok = false; break; }
                ptx::mbar_arrive_expect_tx(&sm.v_full[st], 2 * kTile);
                for (int hf = 0; hf < 2; ++hf)
                    ptx::tma_load_4d(sm.v[st][hf], &tmv, hf * 64, g, j * 128, b, &sm.v_full[st]);
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
                    if (!key_visible(qpos, j * 128 + c, window)) x[c] = -INFINITY;
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
            float r4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 4; ++c) {  // P = 2^(s*scale*log2e - m) as bf16 over the S columns
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float p0 = ptx::exp2_approx(fmaf(x[32 * c + 2 * i], sl2, -mb));
                    const float p1 = ptx::exp2_approx(fmaf(x[32 * c + 2 * i + 1], sl2, -mb));
                    r4[(2 * i) & 3] += p0;
                    r4[(2 * i + 1) & 3] += p1;
                    pk[i] = ptx::pack_bf16x2(p0, p1);
                }
                ptx::tmem_st16(tS + 16 * c, pk);
            }
            l += (r4[0] + r4[1]) + (r4[2] + r4[3]);
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
            const float inv = (l > 0.f) ? 1.f / l : 0.f;
            store_o_row_smem(tO, inv, sm.q[t][0], sm.q[t][1], row);
            ptx::fence_proxy_async_smem();
        } else if (lane == 0) {
            atomicOr(err, kErrWait);
        }
        const bool wg_fail = ptx::named_bar_or(1 + t, 128, !ok);
        if (row == 0 && !wg_fail) {
            for (int hf = 0; hf < 2; ++hf) ptx::tma_store_4d(&tmo, sm.q[t][hf], hf * 64, h, qs, b);
            ptx::bulk_commit();
            ptx::bulk_wait_read0();
        }
        if (ok && lse && qpos < T)
            lse[(static_cast<long>(b) * Hq + h) * T + qpos] =
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

// =========================================================== packed SWA kernel
namespace swa {

constexpr int kThreads = 352;  // WG0 (slot 0), WG1 (slot 1), warp 8 Q/K TMA, warp 9 MMA, warp 10 V TMA
constexpr int kN = 144;        // keys per tile (G = 8, W <= 129)
constexpr int kQBytes = 128 * kHalfRowBytes;   // 16 KB per D half
constexpr int kKBytes = kN * kHalfRowBytes;    // 18 KB per D half
constexpr int kPCols = kN / 2;                  // bf16 P columns
constexpr int kOCol = ((kPCols + 31) / 32) * 32;  // O accumulator column (96)
constexpr uint32_t kIdescS = ptx::idesc_bf16(128, kN, false, false);
constexpr uint32_t kIdescPV = ptx::idesc_bf16(128, 128, false, true);
static_assert(kOCol + 128 <= 256, "slot TMEM budget");

struct __align__(1024) Smem {
    uint8_t q[2][2][kQBytes];  // [slot][D half]
    uint8_t k[2][2][kKBytes];
    uint8_t v[2][2][kKBytes];
    uint64_t qk_full[2], v_full[2], s_full[2], p_full[2], o_full[2], tmem_free[2];
    uint32_t tmem_base;
    int abort;
};

struct TileCoord {
    int b, g, i0;
};
ATTN_DEV TileCoord tile_coord(int u, int nblk, int Hkv, int TT) {
    TileCoord c;
    c.i0 = (u % nblk) * TT;
    c.g = (u / nblk) % Hkv;
    c.b = u / (nblk * Hkv);
    return c;
}

// Scaled max over NC columns starting at column c0 of this row, restricted to
// the visible range [c_lo, c_hi], with four independent partial maxima.
template <int NC>
ATTN_DEV float chunk_max(const float (&x)[NC], int c0, int c_lo, int c_hi, float sl2) {
    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        const int c = c0 + i;
        const bool vis = static_cast<unsigned>(c - c_lo) <= static_cast<unsigned>(c_hi - c_lo);
        m4[i & 3] = fmaxf(m4[i & 3], vis ? x[i] : -INFINITY);
    }
    return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl2;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_swa_kernel(const __grid_constant__ CUtensorMap tmq,
                       const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, __nv_bfloat16 *__restrict__ out,
                       const float *__restrict__ sink, float *__restrict__ lse, int B, int T,
                       int Hq, int Hkv, int window, float scale, unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                         ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = Hq / Hkv, TT = swa_pack_tokens(G);
    const int nblk = (T + TT - 1) / TT;
    const int ntiles = nblk * Hkv * B;
    const int ncta = (ntiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                     static_cast<int>(gridDim.x);  // tiles of this CTA
    auto tile_of = [&](int k) { return static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&sm.qk_full[s], 1);
            ptx::mbar_init(&sm.v_full[s], 1);
            ptx::mbar_init(&sm.s_full[s], 1);
            ptx::mbar_init(&sm.p_full[s], 128);
            ptx::mbar_init(&sm.o_full[s], 1);
            ptx::mbar_init(&sm.tmem_free[s], 128);
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

    if (warp == 8 || warp == 10) {
        // ------------------------------------------ TMA producers (Q/K and V)
        // Q and K of a slot are free once its S MMA completed; V once its PV
        // MMA completed.  Two producer warps keep the two streams independent.
        if (lane == 0 && !skip) {
            bool ok = true;
            const bool qk = (warp == 8);
            if (qk) {
                ptx::prefetch_tmap(&tmq);
                ptx::prefetch_tmap(&tmk);
            } else {
                ptx::prefetch_tmap(&tmv);
            }
            for (int k = 0; ok && k < ncta; ++k) {
                const int s = k & 1, u = k >> 1;
                const TileCoord c = tile_coord(tile_of(k), nblk, Hkv, TT);
                const int key0 = swa_pack_key0(c.i0, G, window);
                if (qk) {
                    if (u > 0 && !ptx::mbar_wait(&sm.s_full[s], (u - 1) & 1)) { ok = false; break; }
                    ptx::mbar_arrive_expect_tx(&sm.qk_full[s], 2 * kQBytes + 2 * kKBytes);
                    for (int hf = 0; hf < 2; ++hf) {
                        ptx::tma_load_4d(sm.q[s][hf], &tmq, hf * 64, c.g * G, c.i0, c.b, &sm.qk_full[s]);
                        ptx::tma_load_4d(sm.k[s][hf], &tmk, hf * 64, c.g, key0, c.b, &sm.qk_full[s]);
                    }
                } else {
                    if (u > 0 && !ptx::mbar_wait(&sm.o_full[s], (u - 1) & 1)) { ok = false; break; }
                    ptx::mbar_arrive_expect_tx(&sm.v_full[s], 2 * kKBytes);
                    for (int hf = 0; hf < 2; ++hf)
                        ptx::tma_load_4d(sm.v[s][hf], &tmv, hf * 64, c.g, key0, c.b, &sm.v_full[s]);
                }
            }
            if (!ok) atomicOr(err, kErrWait);
        }
        __syncwarp();
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA
        if (lane == 0 && !skip) {
            auto issue_s = [&](int k) -> bool {
                const int s = k & 1, u = k >> 1;
                if (!ptx::mbar_wait(&sm.qk_full[s], u & 1)) return false;
                if (u > 0 && !ptx::mbar_wait(&sm.tmem_free[s], (u - 1) & 1)) return false;
                ptx::tc_fence_after();
                for (int kk = 0; kk < 8; ++kk)
                    ptx::mma_ss(tmem + 256 * s, kmajor_desc(sm.q[s][kk >> 2], kk & 3),
                                kmajor_desc(sm.k[s][kk >> 2], kk & 3), kIdescS, kk > 0);
                ptx::tc_commit(&sm.s_full[s]);
                return true;
            };
            bool ok = true;
            if (ncta > 0) ok = issue_s(0);
            if (ok && ncta > 1) ok = issue_s(1);
            for (int k = 0; ok && k < ncta; ++k) {
                const int s = k & 1, u = k >> 1;
                if (!ptx::mbar_wait(&sm.v_full[s], u & 1) || !ptx::mbar_wait(&sm.p_full[s], u & 1)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                for (int kk = 0; kk < kN / 16; ++kk)
                    ptx::mma_ts(tmem + 256 * s + kOCol, tmem + 256 * s + kk * 8,
                                vmajor_desc(sm.v[s][0], kk, kKBytes), kIdescPV, kk > 0);
                ptx::tc_commit(&sm.o_full[s]);
                if (k + 2 < ncta) ok = issue_s(k + 2);
            }
            if (!ok) atomicOr(err, kErrWait);
        }
        __syncwarp();
    } else if (!skip) {
        // ------------------------------------------------ softmax warpgroups
        // One thread per row (TMEM lane).  Failure decisions are warp-uniform
        // and there is no barrier inside the loop, so an error never splits a
        // warpgroup at a barrier.
        const int s = warp >> 2;
        const int row = threadIdx.x & 127;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + 256 * s + lane_off, tO = tS + kOCol;
        const int t_in = row / G, hh = row % G;
        const float sl2 = scale * kLog2e;
        for (int k = s; k < ncta; k += 2) {
            const int u = k >> 1;
            const TileCoord c = tile_coord(tile_of(k), nblk, Hkv, TT);
            const int key0 = swa_pack_key0(c.i0, G, window);
            const int qpos = c.i0 + t_in, h = c.g * G + hh;
            // visible key columns of this row: [c_lo, c_hi]
            const int c_hi = qpos - key0;
            const int c_lo = max(qpos - window + 1, 0) - key0;
            const float sig = sink[h];
            if (!ptx::mbar_wait_warp(&sm.s_full[s], u & 1)) {
                if (lane == 0) atomicOr(err, kErrWait);
                break;
            }
            ptx::tc_fence_after();
            // pass 1: row max over the visible scores, seeded with the sink logit
            float m = sig * kLog2e;
#pragma unroll
            for (int cc = 0; cc < kN / 48; ++cc) {
                float x[48];
                tmem_load_row<48>(tS + 48 * cc, x);
                m = fmaxf(m, chunk_max<48>(x, 48 * cc, c_lo, c_hi, sl2));
            }
            const bool sink_all = isinf(sig) && sig > 0.f;
            const float mb = (m == -INFINITY || sink_all) ? 0.f : m;
            // pass 2: P = 2^(s*scale*log2e - m) as bf16 over the S columns
            // (P column c/2 <= S column c, already read); four partial sums
            float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int cc = 0; cc < kN / 48; ++cc) {
                float x[48];
                tmem_load_row<48>(tS + 48 * cc, x);
#pragma unroll
                for (int i = 0; i < 48; ++i) {
                    const int col = 48 * cc + i;
                    const bool vis = static_cast<unsigned>(col - c_lo) <=
                                     static_cast<unsigned>(c_hi - c_lo);
                    x[i] = (vis && !sink_all) ? ptx::exp2_approx(fmaf(x[i], sl2, -mb)) : 0.f;
                    l4[i & 3] += x[i];
                }
                tmem_store_p<48>(tS + 24 * cc, x);
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&sm.p_full[s]);
            // the sink's own term joins the sum
            float l = (l4[0] + l4[1]) + (l4[2] + l4[3]);
            if (!(isinf(sig) && sig < 0.f) && !sink_all) l += ptx::exp2_approx(sig * kLog2e - mb);

            if (!ptx::mbar_wait_warp(&sm.o_full[s], u & 1)) {
                if (lane == 0) atomicOr(err, kErrWait);
                break;
            }
            ptx::tc_fence_after();
            // epilogue: O row from TMEM, normalised, straight to global memory
            const float inv = sink_all ? 0.f : 1.f / l;
            uint4 *dst = reinterpret_cast<uint4 *>(
                out + ((static_cast<long>(c.b) * T + min(qpos, T - 1)) * Hq + h) * 128);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {  // 32 columns at a time: load, pack, store
                uint32_t r[32];
                ptx::tmem_ld32(tO + cc * 32, r);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                reg_dep(r);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = ptx::pack_bf16x2(__uint_as_float(r[2 * i]) * inv,
                                             __uint_as_float(r[2 * i + 1]) * inv);
                if (qpos < T) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[cc * 4 + i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&sm.tmem_free[s]);  // S/O columns of this slot may be reused
            if (qpos < T && lse)
                lse[(static_cast<long>(c.b) * Hq + h) * T + qpos] =
                    sink_all ? INFINITY : (mb + log2f(l)) * kLn2;
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

}  // namespace swa

int num_sms() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

}  // namespace

int prefill_swa_tc_supported(int G, int window) {
    return G >= 1 && G <= 128 && (128 % G) == 0 && window >= 1 &&
           swa_pack_keys(G, window) == swa::kN;
}

cudaError_t launch_prefill_ga_tc(const PrefillMaps &maps, const float *sink, float *lse, int B,
                                 int T, int Hq, int Hkv, int window, float scale,
                                 unsigned int *err, cudaStream_t s) {
    if (B == 0 || T == 0) return cudaSuccess;
    const size_t smem = sizeof(ga::Smem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(ga::prefill_ga_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const long blocks = static_cast<long>((T + 255) / 256) * Hq * B;
    ga::prefill_ga_kernel<<<static_cast<unsigned>(blocks), ga::kThreads, smem, s>>>(
        maps.q, maps.k, maps.v, maps.o, sink, lse, B, T, Hq, Hkv, window, scale, err);
    return cudaGetLastError();
}

cudaError_t launch_prefill_swa_tc(const PrefillMaps &maps, const float *sink, float *lse, int B,
                                  int T, int Hq, int Hkv, int window, float scale,
                                  unsigned int *err, cudaStream_t s) {
    if (B == 0 || T == 0) return cudaSuccess;
    const size_t smem = sizeof(swa::Smem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(swa::prefill_swa_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int G = Hq / Hkv, TT = swa_pack_tokens(G);
    const long ntiles = static_cast<long>((T + TT - 1) / TT) * Hkv * B;
    const int grid = static_cast<int>(ntiles < num_sms() ? ntiles : num_sms());
    swa::prefill_swa_kernel<<<grid, swa::kThreads, smem, s>>>(
        maps.q, maps.k, maps.v, static_cast<__nv_bfloat16 *>(maps.out), sink, lse, B, T, Hq, Hkv,
        window, scale, err);
    return cudaGetLastError();
}

}  // namespace attn

// Backward pass of sink attention on the 5th-generation tensor cores
// (sm_103a), bf16 in/out, fp32 accumulation, D = 128: dQ, dK, dV and the sink
// logits' gradient dsigma.
//
// The sinks are learnable (technical-report summary "MiMo-V2", section
// "Hybrid Sliding Window Attention Architecture"), so training needs their
// gradient next to the usual ones.  With P the attention weights of the
// forward pass, p_sink the sink's weight and D_i = <dO_i, O_i>:
//   dS_ij = P_ij (<dO_i, v_j> - D_i),  dq_i = scale sum_j dS_ij k_j,
//   dk_j = scale sum_i dS_ij q_i,  dv_j = sum_i P_ij dO_i,
//   dsigma_h = -sum_i p_sink,i D_i      (the sink column carries value 0).
// P is recomputed from Q, K and the forward's log-sum-exp (which includes the
// sink): P_ij = exp(S_ij - lse_i), p_sink,i = exp(sigma_h - lse_i).
//
// Three kernels, none with atomics on the gradients:
//   bwd_pre_kernel   D_i per (b, h, i) and a block-reduced dsigma;
//   bwd_dkdv_kernel  persistent CTAs (one per SM) over items (128-key tile,
//                    kv head, b).  The key tile is the MMA's M side: per
//                    step of 64 query rows of one head of the group,
//                    S^T = K Q^T and dP^T = V dO^T go to TMEM (tcgen05.mma,
//                    K and Q / V and dO from shared memory); two compute
//                    warpgroups (alternate steps, one key row per thread)
//                    form P^T and dS^T = P^T (dP^T - D) in bf16 over the same
//                    TMEM columns; then dV += P^T dO and dK += dS^T Q run
//                    with A from TMEM.  dK and dV stay in TMEM for the whole
//                    item, and an epilogue warpgroup drains them;
//   bwd_dq_kernel    persistent CTAs over items (128-row query tile, head,
//                    b), the query rows on the M side.  The epilogue warps copy the tile's Q and
//                    dO rows into TMEM, so per step of 64 keys S = Q K^T and
//                    dP = dO V^T take A from TMEM and read only K and V from
//                    shared memory; dS = P (dP - D) in bf16 in TMEM, then
//                    dQ += dS K with A from TMEM.
// Q, dO, K and V tiles arrive by TMA (128-byte swizzle) through 4-stage
// (dK/dV) and 3-stage (dQ) rings fed by one producer warp; one thread issues
// every MMA; S/dP sit in two TMEM buffers so one step's exponentials overlap
// the next step's products.  The compute warps keep their instruction count
// low (paired fp32 arithmetic, the column mask only where a row does not see
// the whole step, no register spills): work in warps beside the tensor-core
// stream slows that stream.
// P and dS are rounded to bf16 before the products that use them, as the
// forward rounds P.  Computing dQ in its own kernel repeats S and dP (seven
// products per visible pair instead of five) but keeps the gradients free of
// fp32 atomics, which for global attention would add every (key tile, query
// tile) partial into a full-size dQ buffer.
#include <cuda_bf16.h>

#include "index_math.cuh"
#include "internal.h"
#include "ptx_sm103.cuh"
#include "tc_tile.cuh"

namespace attn {
namespace {

using namespace tc;

constexpr int kD = 128;

__global__ void __launch_bounds__(256)
    bwd_pre_kernel(const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dout,
                   const float *__restrict__ lse, const float *__restrict__ sink,
                   float *__restrict__ delta, float *__restrict__ dsink, int T, int Hq) {
    // block = (128 rows of one (b, h)); warp per row, 4 elements per lane
    const int h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float sig = sink[h];
    float part = 0.f;
    for (int r = warp; r < 128; r += 8) {
        const int i = blockIdx.x * 128 + r;
        if (i >= T) break;
        const long off = ((static_cast<long>(b) * T + i) * Hq + h) * kD + 4 * lane;
        const uint2 uo = *reinterpret_cast<const uint2 *>(o + off);
        const uint2 ud = *reinterpret_cast<const uint2 *>(dout + off);
        const float2 o0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&uo.x));
        const float2 o1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&uo.y));
        const float2 d0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ud.x));
        const float2 d1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ud.y));
        float s = o0.x * d0.x + o0.y * d0.y + o1.x * d1.x + o1.y * d1.y;
#pragma unroll
        for (int k = 16; k > 0; k >>= 1) s += __shfl_xor_sync(0xffffffffu, s, k);
        const long li = (static_cast<long>(b) * Hq + h) * T + i;
        if (lane == 0) {
            delta[li] = s;
            // p_sink = e^(sigma - lse); sigma = +inf: lse = +inf and O = 0, no gradient
            const float l = lse[li];
            if (!(isinf(sig) && sig > 0.f)) part -= expf(sig - l) * s;
        }
    }
    __shared__ float red[8];
    if (lane == 0) red[warp] = part;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < 8; ++w) t += red[w];
        atomicAdd(&dsink[h], t);
    }
}

// Writes N fp32 columns of this thread's TMEM lane (starting at taddr), times
// mul, as bf16 to dst (N/8 16-byte stores) when `store` holds.  Every lane of
// the warp must call it: the TMEM loads are warp-collective, so only the
// stores are predicated.
template <int N>
ATTN_DEV void store_row_bf16(uint32_t taddr, float mul, __nv_bfloat16 *dst, bool store) {
#pragma unroll
    for (int c = 0; c < N / 32; ++c) {
        uint32_t r[32];
        ptx::tmem_ld32(taddr + c * 32, r);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        reg_dep(r);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
            uint4 w;
            w.x = ptx::pack_bf16x2(__uint_as_float(r[8 * ch + 0]) * mul, __uint_as_float(r[8 * ch + 1]) * mul);
            w.y = ptx::pack_bf16x2(__uint_as_float(r[8 * ch + 2]) * mul, __uint_as_float(r[8 * ch + 3]) * mul);
            w.z = ptx::pack_bf16x2(__uint_as_float(r[8 * ch + 4]) * mul, __uint_as_float(r[8 * ch + 5]) * mul);
            w.w = ptx::pack_bf16x2(__uint_as_float(r[8 * ch + 6]) * mul, __uint_as_float(r[8 * ch + 7]) * mul);
            if (store) *reinterpret_cast<uint4 *>(dst + 32 * c + 8 * ch) = w;
        }
    }
}

// Eight consecutive 32-bit TMEM columns of this thread's lane (warp-collective).
ATTN_DEV void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 ATTN_I8(0)
                 : "memory");
}

// Four consecutive fp32 values from shared memory (16-byte aligned).
ATTN_DEV float4 lds4(const float *p) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(ptx::smem_u32(p)));
    return v;
}

// One compute step of 64 columns (queries for dK/dV, keys for dQ) of this
// thread's TMEM lane: P = 2^(S*scale*log2e - lse2) on the visible columns
// [lo, hi) and 0 elsewhere, dS = P (dP - delta); P (if wanted) replaces S and
// dS replaces dP as packed bf16 (32 columns each).  The negated lse2 and
// delta come per column (arrays in shared memory, kColumns) or as one value
// for the row.  The mask (kMask; without it every column is visible) is a
// select after the exponential, never a branch; the fp32 arithmetic runs on
// pairs (f32x2), half the FMA-pipe instructions.
template <bool kWantP, bool kColumns, bool kMask>
ATTN_DEV void p_ds_step(uint32_t tS, uint32_t tdP, float sl2, const float *nlse2_col,
                        const float *ndelta_col, float nlse2_row, float ndelta_row, int lo, int hi) {
    const uint64_t sl2x2 = f2(sl2, sl2);
    const uint64_t nl_row = f2(nlse2_row, nlse2_row), nd_row = f2(ndelta_row, ndelta_row);
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) {
#pragma unroll
        for (int c4 = 0; c4 < 2; ++c4) {  // 16 columns at a time
            const int cb = 32 * c2 + 16 * c4;
            uint32_t pk[8], dk[8];
            uint32_t s[16], dp[16];
            ptx::tmem_ld16(tS + cb, s);
            ptx::tmem_ld16(tdP + cb, dp);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            reg_dep(s);
            reg_dep(dp);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint64_t nl01 = nl_row, nl23 = nl_row, nd01 = nd_row, nd23 = nd_row;
                if constexpr (kColumns) {
                    const float4 lv = lds4(nlse2_col + cb + 4 * q);
                    const float4 dv = lds4(ndelta_col + cb + 4 * q);
                    nl01 = f2(lv.x, lv.y);
                    nl23 = f2(lv.z, lv.w);
                    nd01 = f2(dv.x, dv.y);
                    nd23 = f2(dv.z, dv.w);
                }
                const float2 a01 = f2_split(f2_fma(
                    f2(__uint_as_float(s[4 * q]), __uint_as_float(s[4 * q + 1])), sl2x2, nl01));
                const float2 a23 = f2_split(f2_fma(
                    f2(__uint_as_float(s[4 * q + 2]), __uint_as_float(s[4 * q + 3])), sl2x2, nl23));
                float p[4] = {ptx::exp2_approx(a01.x), ptx::exp2_approx(a01.y),
                              ptx::exp2_approx(a23.x), ptx::exp2_approx(a23.y)};
                if constexpr (kMask) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = cb + 4 * q + e;
                        p[e] = (c >= lo && c < hi) ? p[e] : 0.f;
                    }
                }
                const float2 d01 = f2_split(f2_mul(
                    f2(p[0], p[1]),
                    f2_add(f2(__uint_as_float(dp[4 * q]), __uint_as_float(dp[4 * q + 1])), nd01)));
                const float2 d23 = f2_split(f2_mul(
                    f2(p[2], p[3]),
                    f2_add(f2(__uint_as_float(dp[4 * q + 2]), __uint_as_float(dp[4 * q + 3])), nd23)));
                pk[2 * q] = ptx::pack_bf16x2(p[0], p[1]);
                pk[2 * q + 1] = ptx::pack_bf16x2(p[2], p[3]);
                dk[2 * q] = ptx::pack_bf16x2(d01.x, d01.y);
                dk[2 * q + 1] = ptx::pack_bf16x2(d23.x, d23.y);
            }
            if constexpr (kWantP) tmem_st8(tS + cb / 2, pk);
            tmem_st8(tdP + cb / 2, dk);
        }
    }
    ptx::tmem_st_wait();
}

// Visible columns [lo, hi) of a step: for key row j against query rows
// i0..i0+63 (dK/dV: visible iff j <= i and, with a window, j > i - W), and for
// query row i against keys j0..j0+63 (dQ).
ATTN_DEV void cols_for_key(int j, int i0, int window, int &lo, int &hi) {
    lo = j - i0;
    hi = window > 0 ? j - i0 + window : 1 << 30;
}
ATTN_DEV void cols_for_query(int i, int j0, int window, int &lo, int &hi) {
    lo = window > 0 ? i - window + 1 - j0 : -(1 << 30);
    hi = i - j0 + 1;
}

// Walks a persistent CTA's work items (item = cta, cta + grid, ..) and the
// steps of each, in the order every role of the CTA uses.
struct ItemCursor {
    int item, k, t, n;  // work item, its index in this CTA, step within it, global step
};

// ================================================================= dK, dV
namespace bkv {

constexpr int kBK = 128;                      // keys per item (TMEM lanes)
constexpr int kBQ = 64;                       // query rows per step
constexpr int kStages = 4;
constexpr int kThreads = 512;  // warp 0 TMA, 1 MMA, 4-7 / 8-11 compute, 12-15 epilogue
constexpr int kKTile = kBK * kHalfRowBytes;   // 16 KB per D half
constexpr int kQTile = kBQ * kHalfRowBytes;   // 8 KB per D half
constexpr uint32_t kColDV = 0, kColDK = 128, kColBuf = 256;  // buffer b: S^T 256+128b, dP^T +64
constexpr uint32_t kIdescS = ptx::idesc_bf16(128, kBQ, false, false);
constexpr uint32_t kIdescAcc = ptx::idesc_bf16(128, 128, false, true);

struct __align__(1024) Stage {
    uint8_t q[2][kQTile];     // [D half][row][64]
    uint8_t dout[2][kQTile];
    float nlse2[kBQ];         // -lse * log2(e); -inf for rows past T (so P = 0 there)
    float ndelta[kBQ];        // -D
};
struct __align__(1024) Smem {
    uint8_t k[2][kKTile];
    uint8_t v[2][kKTile];
    Stage st[kStages];
    uint64_t kv_full, kv_empty, full[kStages], empty[kStages], sdp_full[2], p_full[2];
    uint64_t acc_full, acc_empty, mma_done;
    uint32_t tmem_base;
    int abort;
};

struct Problem {
    int B, T, Hq, Hkv, G, window, nitems;
    // item -> (key tile, kv head, sequence); key tile 0 (the most query rows
    // under causal attention) first
    ATTN_DEV void item(int it, int &j0, int &g, int &b, int &qt0, int &nqt) const {
        const int per = Hkv * B;
        j0 = (it / per) * kBK;
        g = it % Hkv;
        b = (it / Hkv) % B;
        int qt1;
        bwd_kv_query_tiles(j0, T, window, kBK, kBQ, &qt0, &qt1);
        nqt = qt1 - qt0 + 1;
    }
};

__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmdo,
                    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                    const float *__restrict__ lse, const float *__restrict__ delta,
                    __nv_bfloat16 *__restrict__ dk, __nv_bfloat16 *__restrict__ dv, Problem pr,
                    float scale, unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                         ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x, grid = gridDim.x;
    const int T = pr.T, Hq = pr.Hq, Hkv = pr.Hkv, G = pr.G, window = pr.window;

    if (threadIdx.x == 0) {
        ptx::mbar_init(&sm.kv_full, 1);
        ptx::mbar_init(&sm.kv_empty, 1);
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(&sm.full[i], 1);
            ptx::mbar_init(&sm.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&sm.sdp_full[i], 1);
            ptx::mbar_init(&sm.p_full[i], 4);  // one arrival per warp of the group
        }
        ptx::mbar_init(&sm.acc_full, 1);
        ptx::mbar_init(&sm.acc_empty, 4);      // one arrival per epilogue warp
        ptx::mbar_init(&sm.mma_done, 1);
        sm.abort = ptx::prior_timeout(err) ? 1 : 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(&sm.tmem_base, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const bool skip = sm.abort != 0;  // an earlier launch timed out: do nothing
    auto aborted = [&]() { return *reinterpret_cast<volatile int *>(&sm.abort) != 0; };
    auto fail = [&]() {
        *reinterpret_cast<volatile int *>(&sm.abort) = 1;
        atomicOr(err, kErrWait);
    };

    if (warp == 0 && !skip) {
        // --------------- TMA (lane 0); the lse/D rows of each step (whole warp)
        int n = 0, k = 0;
        bool ok = true;
        if (lane == 0) {
            ptx::prefetch_tmap(&tmq);
            ptx::prefetch_tmap(&tmdo);
            ptx::prefetch_tmap(&tmk);
            ptx::prefetch_tmap(&tmv);
        }
        for (int it = cta; ok && it < pr.nitems; it += grid, ++k) {
            int j0, g, b, qt0, nqt;
            pr.item(it, j0, g, b, qt0, nqt);
            if (k >= 1 && !(ok = ptx::mbar_wait_warp(&sm.kv_empty, (k - 1) & 1))) break;
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(&sm.kv_full, 4 * kKTile);
                for (int hf = 0; hf < 2; ++hf) {
                    ptx::tma_load_3d(sm.k[hf], &tmk, hf * 64, g, b * T + j0, &sm.kv_full);
                    ptx::tma_load_3d(sm.v[hf], &tmv, hf * 64, g, b * T + j0, &sm.kv_full);
                }
            }
            for (int t = 0; t < G * nqt; ++t, ++n) {
                const int h = g * G + t / nqt, i0 = (qt0 + t % nqt) * kBQ;
                const long base = (static_cast<long>(b) * Hq + h) * T;
                float l2[2], dl[2];  // loads in flight while the stage drains
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int i = i0 + lane + 32 * e;
                    l2[e] = i < T ? -lse[base + i] * kLog2e : -INFINITY;
                    dl[e] = i < T ? -delta[base + i] : 0.f;
                }
                const int s = n % kStages;
                if (n >= kStages && (aborted() || !(ok = ptx::mbar_wait_warp(&sm.empty[s], ((n / kStages) - 1) & 1)))) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    sm.st[s].nlse2[lane + 32 * e] = l2[e];
                    sm.st[s].ndelta[lane + 32 * e] = dl[e];
                }
                __syncwarp();
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(&sm.full[s], 4 * kQTile);
                    for (int hf = 0; hf < 2; ++hf) {
                        ptx::tma_load_3d(sm.st[s].q[hf], &tmq, hf * 64, h, b * T + i0, &sm.full[s]);
                        ptx::tma_load_3d(sm.st[s].dout[hf], &tmdo, hf * 64, h, b * T + i0, &sm.full[s]);
                    }
                }
            }
        }
        if (!ok && lane == 0) fail();
        // copies in flight land before the CTA may exit (bounded waits)
        if (lane == 0) {
            if (k > 0) ptx::mbar_wait(&sm.kv_full, (k - 1) & 1);
            for (int s = 0; s < kStages; ++s) {
                const int uses = (n - s + kStages - 1) / kStages;
                if (uses > 0) ptx::mbar_wait(&sm.full[s], (uses - 1) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 1 && !skip) {
        // ---------------------------------------------------------- MMAs
        if (lane == 0) {
            bool ok = true, issued = false;
            int pn = -1, pk = 0, pt = 0, pN = 0;  // the step whose dV/dK is still due
            // dV += P^T dO and dK += dS^T Q of step n (item k, step t of N)
            auto acc_step = [&](int n, int k, int t, int N) {
                const int s = n % kStages, bb = n & 1;
                if (!ptx::mbar_wait(&sm.p_full[bb], (n >> 1) & 1)) return false;
                if (t == 0 && k >= 1 && !ptx::mbar_wait(&sm.acc_empty, (k - 1) & 1)) return false;
                ptx::tc_fence_after();
                const uint32_t tP = tmem + kColBuf + 128 * bb, tdS = tP + 64;
                for (int kk = 0; kk < kBQ / 16; ++kk)
                    ptx::mma_ts(tmem + kColDV, tP + kk * 8, vmajor_desc(sm.st[s].dout[0], kk, kQTile),
                                kIdescAcc, (t > 0 || kk > 0) ? 1u : 0u);
                for (int kk = 0; kk < kBQ / 16; ++kk)
                    ptx::mma_ts(tmem + kColDK, tdS + kk * 8, vmajor_desc(sm.st[s].q[0], kk, kQTile),
                                kIdescAcc, (t > 0 || kk > 0) ? 1u : 0u);
                ptx::tc_commit(&sm.empty[s]);
                if (t == N - 1) ptx::tc_commit(&sm.acc_full);
                return true;
            };
            int n = 0, k = 0;
            for (int it = cta; ok && it < pr.nitems; it += grid, ++k) {
                int j0, g, b, qt0, nqt;
                pr.item(it, j0, g, b, qt0, nqt);
                const int N = G * nqt;
                if (!(ok = !aborted() && ptx::mbar_wait(&sm.kv_full, k & 1))) break;
                for (int t = 0; t < N; ++t, ++n) {
                    // S^T = K Q^T and dP^T = V dO^T into buffer n mod 2
                    const int s = n % kStages, bb = n & 1;
                    if (!(ok = ptx::mbar_wait(&sm.full[s], (n / kStages) & 1))) break;
                    ptx::tc_fence_after();
                    const uint32_t tS = tmem + kColBuf + 128 * bb, tdP = tS + 64;
                    for (int kk = 0; kk < 8; ++kk)
                        ptx::mma_ss(tS, kmajor_desc(sm.k[kk >> 2], kk & 3),
                                    kmajor_desc(sm.st[s].q[kk >> 2], kk & 3), kIdescS, kk > 0);
                    for (int kk = 0; kk < 8; ++kk)
                        ptx::mma_ss(tdP, kmajor_desc(sm.v[kk >> 2], kk & 3),
                                    kmajor_desc(sm.st[s].dout[kk >> 2], kk & 3), kIdescS, kk > 0);
                    ptx::tc_commit(&sm.sdp_full[bb]);
                    if (t == N - 1) ptx::tc_commit(&sm.kv_empty);
                    issued = true;
                    if (pn >= 0 && !(ok = acc_step(pn, pk, pt, pN))) break;
                    pn = n;
                    pk = k;
                    pt = t;
                    pN = N;
                }
            }
            if (ok && pn >= 0) ok = acc_step(pn, pk, pt, pN);
            if (!ok) fail();
            if (issued) {  // every MMA completes before TMEM is released (bounded)
                ptx::tc_commit(&sm.mma_done);
                ptx::mbar_wait(&sm.mma_done, 0);
            }
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 12 && !skip) {
        // ------------------------- compute: group j takes the steps n = j mod 2
        const int j = (warp - 4) >> 2, row = threadIdx.x & 127;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + kColBuf + 128 * j, tdP = tS + 64;
        const float sl2 = scale * kLog2e;
        bool ok = true;
        int n = 0;
        for (int it = cta; ok && it < pr.nitems; it += grid) {
            int j0, g, b, qt0, nqt;
            pr.item(it, j0, g, b, qt0, nqt);
            const int key = j0 + row;
            for (int t = 0; t < G * nqt; ++t, ++n) {
                if ((n & 1) != j) continue;
                if (!(ok = !__any_sync(0xffffffffu, aborted()) &&
                           ptx::mbar_wait_warp(&sm.sdp_full[j], (n >> 1) & 1)))
                    break;
                ptx::tc_fence_after();
                const int i0 = (qt0 + t % nqt) * kBQ;
                const Stage &st = sm.st[n % kStages];
                int lo, hi;
                cols_for_key(key, i0, window, lo, hi);
                // a step whose 64 columns this warp's rows all see skips the mask
                if (__all_sync(0xffffffffu, lo <= 0 && hi >= kBQ))
                    p_ds_step<true, true, false>(tS, tdP, sl2, st.nlse2, st.ndelta, 0.f, 0.f, lo, hi);
                else
                    p_ds_step<true, true, true>(tS, tdP, sl2, st.nlse2, st.ndelta, 0.f, 0.f, lo, hi);
                ptx::tc_fence_before();
                if (lane == 0) ptx::mbar_arrive(&sm.p_full[j]);
            }
        }
        if (!ok && lane == 0) fail();
    } else if (warp >= 12 && !skip) {
        // ------------------- epilogue: dV and dK (x scale) of each item -> bf16
        const int row = threadIdx.x & 127;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        int k = 0;
        for (int it = cta; it < pr.nitems; it += grid, ++k) {
            int j0, g, b, qt0, nqt;
            pr.item(it, j0, g, b, qt0, nqt);
            if (__any_sync(0xffffffffu, aborted()) || !ptx::mbar_wait_warp(&sm.acc_full, k & 1)) {
                if (lane == 0) fail();
                break;
            }
            ptx::tc_fence_after();
            const int key = j0 + row;
            const long off = ((static_cast<long>(b) * T + (key < T ? key : 0)) * Hkv + g) * kD;
            store_row_bf16<128>(tmem + lane_off + kColDV, 1.f, dv + off, key < T);
            store_row_bf16<128>(tmem + lane_off + kColDK, scale, dk + off, key < T);
            ptx::tc_fence_before();
            if (lane == 0) ptx::mbar_arrive(&sm.acc_empty);
        }
    }
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

}  // namespace bkv

// ===================================================================== dQ
namespace bq {

constexpr int kBQ = 128;                      // query rows per item (TMEM lanes)
constexpr int kBK = 64;                       // keys per step
constexpr int kStages = 3;
constexpr int kThreads = 512;  // warp 0 TMA, 1 MMA, 4-7 / 8-11 compute, 12-15 epilogue
constexpr int kQTile = kBQ * kHalfRowBytes;   // 16 KB per D half
constexpr int kKTile = kBK * kHalfRowBytes;   // 8 KB per D half
constexpr uint32_t kColDQ = 0, kColQ = 128, kColDO = 192, kColBuf = 256;  // buffer b: S 256+128b, dP +64
constexpr uint32_t kIdescS = ptx::idesc_bf16(128, kBK, false, false);
constexpr uint32_t kIdescAcc = ptx::idesc_bf16(128, 128, false, true);

struct __align__(1024) QBuf {
    uint8_t q[2][kQTile];
    uint8_t dout[2][kQTile];
};
struct __align__(1024) Stage {
    uint8_t k[2][kKTile];
    uint8_t v[2][kKTile];
};
struct __align__(1024) Smem {
    QBuf qb[2];               // items alternate between two Q/dO buffers
    Stage st[kStages];
    uint64_t q_full[2], q_empty[2], full[kStages], empty[kStages], sdp_full[2], p_full[2];
    uint64_t qdo_ready, qdo_used, dq_full, dq_empty, mma_done;
    uint32_t tmem_base;
    int abort;
};

struct Problem {
    int B, T, Hq, Hkv, window, nitems;
    // item -> (query tile, head, sequence); the last query tiles (the most
    // keys under causal attention) first
    ATTN_DEV void item(int it, int &i0, int &h, int &b, int &kt0, int &nkt) const {
        const int nqt = (T + kBQ - 1) / kBQ, per = Hq * B;
        i0 = (nqt - 1 - it / per) * kBQ;
        h = it % Hq;
        b = (it / Hq) % B;
        int kt1;
        bwd_q_key_tiles(i0, T, window, kBQ, kBK, &kt0, &kt1);
        nkt = kt1 - kt0 + 1;
    }
};

__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmdo,
                  const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const float *__restrict__ lse, const float *__restrict__ delta,
                  __nv_bfloat16 *__restrict__ dq, Problem pr, float scale, unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                         ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x, grid = gridDim.x;
    const int T = pr.T, Hq = pr.Hq, G = pr.Hq / pr.Hkv, window = pr.window;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&sm.q_full[i], 1);
            ptx::mbar_init(&sm.q_empty[i], 4);  // the epilogue warps, once Q and dO are in TMEM
            ptx::mbar_init(&sm.sdp_full[i], 1);
            ptx::mbar_init(&sm.p_full[i], 4);
        }
        ptx::mbar_init(&sm.qdo_ready, 4);
        ptx::mbar_init(&sm.qdo_used, 1);
        ptx::mbar_init(&sm.dq_full, 1);
        ptx::mbar_init(&sm.dq_empty, 4);
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(&sm.full[i], 1);
            ptx::mbar_init(&sm.empty[i], 1);
        }
        ptx::mbar_init(&sm.mma_done, 1);
        sm.abort = ptx::prior_timeout(err) ? 1 : 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(&sm.tmem_base, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const bool skip = sm.abort != 0;
    auto aborted = [&]() { return *reinterpret_cast<volatile int *>(&sm.abort) != 0; };
    auto fail = [&]() {
        *reinterpret_cast<volatile int *>(&sm.abort) = 1;
        atomicOr(err, kErrWait);
    };

    if (warp == 0 && !skip) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            ptx::prefetch_tmap(&tmq);
            ptx::prefetch_tmap(&tmdo);
            ptx::prefetch_tmap(&tmk);
            ptx::prefetch_tmap(&tmv);
            bool ok = true;
            int n = 0, k = 0;
            for (int it = cta; ok && it < pr.nitems; it += grid, ++k) {
                int i0, h, b, kt0, nkt;
                pr.item(it, i0, h, b, kt0, nkt);
                const int g = h / G, qs = k & 1;
                if (k >= 2 && !(ok = !aborted() && ptx::mbar_wait(&sm.q_empty[qs], ((k >> 1) - 1) & 1))) break;
                ptx::mbar_arrive_expect_tx(&sm.q_full[qs], 4 * kQTile);
                for (int hf = 0; hf < 2; ++hf) {
                    ptx::tma_load_3d(sm.qb[qs].q[hf], &tmq, hf * 64, h, b * T + i0, &sm.q_full[qs]);
                    ptx::tma_load_3d(sm.qb[qs].dout[hf], &tmdo, hf * 64, h, b * T + i0, &sm.q_full[qs]);
                }
                for (int t = 0; t < nkt; ++t, ++n) {
                    const int s = n % kStages, j0 = (kt0 + t) * kBK;
                    if (n >= kStages && !(ok = ptx::mbar_wait(&sm.empty[s], ((n / kStages) - 1) & 1))) break;
                    ptx::mbar_arrive_expect_tx(&sm.full[s], 4 * kKTile);
                    for (int hf = 0; hf < 2; ++hf) {
                        ptx::tma_load_3d(sm.st[s].k[hf], &tmk, hf * 64, g, b * T + j0, &sm.full[s]);
                        ptx::tma_load_3d(sm.st[s].v[hf], &tmv, hf * 64, g, b * T + j0, &sm.full[s]);
                    }
                }
            }
            if (!ok) fail();
            // copies in flight land before exit (bounded)
            for (int qs = 0; qs < 2; ++qs) {
                const int uses = (k - qs + 1) / 2;
                if (uses > 0) ptx::mbar_wait(&sm.q_full[qs], (uses - 1) & 1);
            }
            for (int s = 0; s < kStages; ++s) {
                const int uses = (n - s + kStages - 1) / kStages;
                if (uses > 0) ptx::mbar_wait(&sm.full[s], (uses - 1) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 1 && !skip) {
        // ---------------------------------------------------------- MMAs
        if (lane == 0) {
            bool ok = true, issued = false;
            int pn = -1, pk = 0, pt = 0, pN = 0;  // the step whose dQ product is still due
            // dQ += dS K of step n (item k, step t of N), dS in TMEM, K in shared memory
            auto acc_step = [&](int n, int k, int t, int N) {
                const int s = n % kStages, bb = n & 1;
                if (!ptx::mbar_wait(&sm.p_full[bb], (n >> 1) & 1)) return false;
                if (t == 0 && k >= 1 && !ptx::mbar_wait(&sm.dq_empty, (k - 1) & 1)) return false;
                ptx::tc_fence_after();
                const uint32_t tdS = tmem + kColBuf + 128 * bb + 64;
                for (int kk = 0; kk < kBK / 16; ++kk)
                    ptx::mma_ts(tmem + kColDQ, tdS + kk * 8, vmajor_desc(sm.st[s].k[0], kk, kKTile),
                                kIdescAcc, (t > 0 || kk > 0) ? 1u : 0u);
                ptx::tc_commit(&sm.empty[s]);
                if (t == N - 1) ptx::tc_commit(&sm.dq_full);
                return true;
            };
            int n = 0, k = 0;
            for (int it = cta; ok && it < pr.nitems; it += grid, ++k) {
                int i0, h, b, kt0, nkt;
                pr.item(it, i0, h, b, kt0, nkt);
                // this item's Q and dO rows are in TMEM (copied by the epilogue warps)
                if (!(ok = !aborted() && ptx::mbar_wait(&sm.qdo_ready, k & 1))) break;
                for (int t = 0; t < nkt; ++t, ++n) {
                    // S = Q K^T and dP = dO V^T into buffer n mod 2, A from TMEM
                    const int s = n % kStages, bb = n & 1;
                    if (!(ok = ptx::mbar_wait(&sm.full[s], (n / kStages) & 1))) break;
                    ptx::tc_fence_after();
                    const uint32_t tS = tmem + kColBuf + 128 * bb, tdP = tS + 64;
                    for (int kk = 0; kk < 8; ++kk)
                        ptx::mma_ts(tS, tmem + kColQ + kk * 8, kmajor_desc(sm.st[s].k[kk >> 2], kk & 3),
                                    kIdescS, kk > 0);
                    for (int kk = 0; kk < 8; ++kk)
                        ptx::mma_ts(tdP, tmem + kColDO + kk * 8, kmajor_desc(sm.st[s].v[kk >> 2], kk & 3),
                                    kIdescS, kk > 0);
                    ptx::tc_commit(&sm.sdp_full[bb]);
                    if (t == nkt - 1) ptx::tc_commit(&sm.qdo_used);  // TMEM Q/dO free once these complete
                    issued = true;
                    if (pn >= 0 && !(ok = acc_step(pn, pk, pt, pN))) break;
                    pn = n;
                    pk = k;
                    pt = t;
                    pN = nkt;
                }
            }
            if (ok && pn >= 0) ok = acc_step(pn, pk, pt, pN);
            if (!ok) fail();
            if (issued) {
                ptx::tc_commit(&sm.mma_done);
                ptx::mbar_wait(&sm.mma_done, 0);
            }
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 12 && !skip) {
        // ------------------------- compute: group j takes the steps n = j mod 2
        const int j = (warp - 4) >> 2, row = threadIdx.x & 127;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + kColBuf + 128 * j, tdP = tS + 64;
        const float sl2 = scale * kLog2e;
        bool ok = true;
        int n = 0;
        for (int it = cta; ok && it < pr.nitems; it += grid) {
            int i0, h, b, kt0, nkt;
            pr.item(it, i0, h, b, kt0, nkt);
            const int i = i0 + row;
            // this row's lse and D, read while the first step's products run
            const long li = (static_cast<long>(b) * Hq + h) * T + (i < T ? i : 0);
            const float nlse2 = i < T ? -lse[li] * kLog2e : -INFINITY;  // rows past T: P = 0
            const float ndlt = i < T ? -delta[li] : 0.f;
            for (int t = 0; t < nkt; ++t, ++n) {
                if ((n & 1) != j) continue;
                if (!(ok = !__any_sync(0xffffffffu, aborted()) &&
                           ptx::mbar_wait_warp(&sm.sdp_full[j], (n >> 1) & 1)))
                    break;
                ptx::tc_fence_after();
                const int j0 = (kt0 + t) * kBK;
                int lo, hi;
                cols_for_query(i, j0, window, lo, hi);
                if (__all_sync(0xffffffffu, lo <= 0 && hi >= kBK))
                    p_ds_step<false, false, false>(tS, tdP, sl2, nullptr, nullptr, nlse2, ndlt, lo, hi);
                else
                    p_ds_step<false, false, true>(tS, tdP, sl2, nullptr, nullptr, nlse2, ndlt, lo, hi);
                ptx::tc_fence_before();
                if (lane == 0) ptx::mbar_arrive(&sm.p_full[j]);
            }
        }
        if (!ok && lane == 0) fail();
    } else if (warp >= 12 && !skip) {
        // ---- epilogue: each item's Q and dO rows into TMEM, then the previous
        // item's dQ (x scale) -> bf16
        const int row = threadIdx.x & 127;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        auto drain = [&](int k, int i0, int h, int b) {  // dQ of item k
            if (__any_sync(0xffffffffu, aborted()) || !ptx::mbar_wait_warp(&sm.dq_full, k & 1))
                return false;
            ptx::tc_fence_after();
            const int i = i0 + row;
            store_row_bf16<128>(tmem + lane_off + kColDQ, scale,
                                dq + ((static_cast<long>(b) * T + (i < T ? i : 0)) * Hq + h) * kD, i < T);
            ptx::tc_fence_before();
            if (lane == 0) ptx::mbar_arrive(&sm.dq_empty);
            return true;
        };
        bool ok = true;
        int k = 0, pi0 = 0, ph = 0, pb = 0;  // the previous item
        for (int it = cta; it < pr.nitems; it += grid, ++k) {
            int i0, h, b, kt0, nkt;
            pr.item(it, i0, h, b, kt0, nkt);
            const int qs = k & 1;
            // the tile's Q and dO have landed, and the previous item's
            // products no longer read the TMEM copies
            if (__any_sync(0xffffffffu, aborted()) || !ptx::mbar_wait_warp(&sm.q_full[qs], (k >> 1) & 1) ||
                (k >= 1 && !ptx::mbar_wait_warp(&sm.qdo_used, (k - 1) & 1))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            row_to_tmem(sm.qb[qs].q[0], sm.qb[qs].q[1], tmem + lane_off + kColQ, row);
            row_to_tmem(sm.qb[qs].dout[0], sm.qb[qs].dout[1], tmem + lane_off + kColDO, row);
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(&sm.qdo_ready);
                ptx::mbar_arrive(&sm.q_empty[qs]);  // the shared-memory tile may take item k + 2
            }
            if (k >= 1 && !(ok = drain(k - 1, pi0, ph, pb))) break;
            pi0 = i0;
            ph = h;
            pb = b;
        }
        if (ok && k >= 1) ok = drain(k - 1, pi0, ph, pb);
        if (!ok && lane == 0) fail();
    }
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

}  // namespace bq

// Streaming multiprocessors of the current device (cached per device).
int sm_count() {
    static int count[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!count[dev] &&
        cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        count[dev] = 148;
    return count[dev];
}

}  // namespace

size_t prefill_backward_workspace(int B, int T, int Hq) {
    const size_t del = static_cast<size_t>(B) * Hq * T * sizeof(float);
    return (del + 255) & ~static_cast<size_t>(255);
}

cudaError_t launch_prefill_backward(const BwdMaps &maps, const void *o, const float *lse,
                                    const void *dout, const float *sink, void *dq, void *dk,
                                    void *dv, float *dsink, void *workspace, int B, int T, int Hq,
                                    int Hkv, int window, float scale, unsigned int *err,
                                    cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(dsink, 0, sizeof(float) * Hq, s);
    if (e != cudaSuccess || B == 0 || T == 0) return e;
    float *delta = static_cast<float *>(workspace);
    bwd_pre_kernel<<<dim3((T + 127) / 128, Hq, B), 256, 0, s>>>(
        static_cast<const __nv_bfloat16 *>(o), static_cast<const __nv_bfloat16 *>(dout), lse, sink,
        delta, dsink, T, Hq);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem_kv = sizeof(bkv::Smem) + 1024;
    e = cudaFuncSetAttribute(bkv::bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_kv));
    if (e != cudaSuccess) return e;
    const int nsm = sm_count();
    bkv::Problem pk{B, T, Hq, Hkv, Hq / Hkv, window, ((T + bkv::kBK - 1) / bkv::kBK) * Hkv * B};
    bkv::bwd_dkdv_kernel<<<pk.nitems < nsm ? pk.nitems : nsm, bkv::kThreads, smem_kv, s>>>(
        maps.q_rows64, maps.dout_rows64, maps.k_rows128, maps.v_rows128, lse, delta,
        static_cast<__nv_bfloat16 *>(dk), static_cast<__nv_bfloat16 *>(dv), pk, scale, err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem_q = sizeof(bq::Smem) + 1024;
    e = cudaFuncSetAttribute(bq::bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_q));
    if (e != cudaSuccess) return e;
    bq::Problem pq{B, T, Hq, Hkv, window, ((T + bq::kBQ - 1) / bq::kBQ) * Hq * B};
    bq::bwd_dq_kernel<<<pq.nitems < nsm ? pq.nitems : nsm, bq::kThreads, smem_q, s>>>(
        maps.q_rows128, maps.dout_rows128, maps.k_rows64, maps.v_rows64, lse, delta,
        static_cast<__nv_bfloat16 *>(dq), pq, scale, err);
    return cudaGetLastError();
}

}  // namespace attn

// Backward pass of sink attention (bf16 in/out, fp32 accumulation, D = 128):
// dQ, dK, dV and the sink logits' gradient dsigma.
//
// The sinks are learnable (technical-report summary "MiMo-V2", section
// "Hybrid Sliding Window Attention Architecture"), so training needs their
// gradient next to the usual ones.  With P the attention weights of the
// forward pass, p_sink the sink's weight and D_i = <dO_i, O_i>:
//   dS_ij = P_ij (<dO_i, v_j> - D_i),  dq_i = scale sum_j dS_ij k_j,
//   dk_j = scale sum_i dS_ij q_i,  dv_j = sum_i P_ij dO_i,
//   dsigma_h = -sum_i p_sink,i D_i      (the sink column carries value 0).
// P is recomputed from Q, K and the forward's log-sum-exp (which includes the
// sink), so P_ij = exp(S_ij - lse_i) and p_sink,i = exp(sigma_h - lse_i).
//
// Kernels:
//   bwd_pre_kernel   D_i per (b, h, i) and a block-reduced dsigma;
//   bwd_main_kernel  one CTA per (64-key tile, kv head, b); warp w owns keys
//                    16w..16w+15 and keeps their dK, dV in registers while it
//                    walks every query head of the group and every 32-row
//                    query tile that sees the key tile (S^T = K Q^T, dP^T =
//                    V dO^T, dV += P^T dO, dK += dS^T Q on mma.sync
//                    m16n8k16); dQ += dS K goes through shared memory and
//                    fp32 atomics into a workspace (about 3 tiles add into a
//                    row for W = 128; every key tile for GA);
//   bwd_dq_kernel    workspace -> bf16 dq.
#include <cuda_bf16.h>

#include "index_math.cuh"
#include "internal.h"
#include "ptx_sm103.cuh"

namespace attn {
namespace {

constexpr int kD = 128;
constexpr int kBK = 64;                 // keys per tile (4 warps x 16)
constexpr int kBQ = 32;                 // query rows per step
constexpr int kThreads = 128;
constexpr int kDsStride = kBQ * 2 + 16;  // bytes per key row of the dS^T tile (padded)
constexpr float kLog2e = 1.4426950408889634f;

struct __align__(128) BwdSmem {
    uint8_t k[2][kBK * 128];      // [D half][key][64] bf16, 128-byte rows, swizzled
    uint8_t v[2][kBK * 128];
    uint8_t q[2][2][kBQ * 128];   // [buffer][D half][row][64]: the next step loads
    uint8_t dout[2][2][kBQ * 128];  // while this one computes
    uint8_t ds[kBK * kDsStride];  // dS^T [key][row] bf16
    float lse[2][kBQ];            // the step's rows' lse and D (zero past T)
    float delta[2][kBQ];
};

// Byte offset of element (row, d) in a swizzled [rows][64] half tile; d % 8 == 0.
__device__ __forceinline__ uint32_t sw(int row, int d) {
    return static_cast<uint32_t>(row * 128 + ((((d >> 3) ^ row) & 7) << 4));
}

// Rows row0 .. row0+N-1 of head h of a [rows, H, 128] bf16 tensor -> a
// swizzled [N][128] tile in two D halves; rows at or past nvalid read as zero.
template <int N>
__device__ __forceinline__ void load_tile(uint8_t *half0, uint8_t *half1,
                                          const __nv_bfloat16 *__restrict__ src, long row0,
                                          int nvalid, int H, int h) {
    for (int x = threadIdx.x; x < N * 16; x += kThreads) {
        const int r = x >> 4, c = x & 15;  // row, 16-byte chunk (8 elements)
        uint4 val = make_uint4(0, 0, 0, 0);
        if (r < nvalid)
            val = *reinterpret_cast<const uint4 *>(src + ((row0 + r) * H + h) * kD + c * 8);
        *reinterpret_cast<uint4 *>((c < 8 ? half0 : half1) + sw(r, (c & 7) * 8)) = val;
    }
}

// Asynchronous form of load_tile for the query-side tiles, with the rows'
// lse and D; rows at or past T are filled with zeros.
__device__ __forceinline__ void prefetch_step(BwdSmem &sm, int buf, const __nv_bfloat16 *q,
                                              const __nv_bfloat16 *dout, const float *lse,
                                              const float *delta, int b, int h, int i0, int T,
                                              int Hq) {
    for (int x = threadIdx.x; x < kBQ * 16; x += kThreads) {
        const int r = x >> 4, c = x & 15;
        const bool ok = i0 + r < T;
        const long off = ((static_cast<long>(b) * T + (ok ? i0 + r : 0)) * Hq + h) * kD + c * 8;
        const uint32_t o = sw(r, (c & 7) * 8);
        ptx::cp_async16(sm.q[buf][c >> 3] + o, q + off, ok ? 16u : 0u);
        ptx::cp_async16(sm.dout[buf][c >> 3] + o, dout + off, ok ? 16u : 0u);
    }
    if (threadIdx.x < kBQ) {
        const int i = i0 + threadIdx.x;
        const bool ok = i < T;
        const long li = (static_cast<long>(b) * Hq + h) * T + (ok ? i : 0);
        ptx::cp_async4(&sm.lse[buf][threadIdx.x], lse + li, ok ? 4u : 0u);
        ptx::cp_async4(&sm.delta[buf][threadIdx.x], delta + li, ok ? 4u : 0u);
    }
}

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

__global__ void __launch_bounds__(kThreads)
    bwd_main_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                    const __nv_bfloat16 *__restrict__ v, const __nv_bfloat16 *__restrict__ dout,
                    const float *__restrict__ lse, const float *__restrict__ delta,
                    float *__restrict__ dq_acc, __nv_bfloat16 *__restrict__ dk,
                    __nv_bfloat16 *__restrict__ dv, int T, int Hq, int Hkv, int window,
                    float scale) {
    extern __shared__ uint8_t smem_raw[];
    BwdSmem &sm = *reinterpret_cast<BwdSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                              ~static_cast<uintptr_t>(127));
    const int j0 = blockIdx.x * kBK, g = blockIdx.y, b = blockIdx.z;
    const int G = Hq / Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, cq = lane & 3;  // fragment row group, column pair
    const int mi = lane >> 3;                 // ldmatrix: matrix fed by this lane
    const float sl2 = scale * kLog2e;

    const int nk = min(kBK, T - j0);
    load_tile<kBK>(sm.k[0], sm.k[1], k, static_cast<long>(b) * T + j0, nk, Hkv, g);
    load_tile<kBK>(sm.v[0], sm.v[1], v, static_cast<long>(b) * T + j0, nk, Hkv, g);

    // rows that see a key of this tile: [j0, last]
    int last = T - 1;
    if (window > 0) last = min(last, j0 + kBK - 1 + window - 1);

    float dka[16][4], dva[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) dka[n][e] = dva[n][e] = 0.f;

    const int kw = warp * 16;  // this warp's first key within the tile
    // steps: every query head of the group x every 32-row tile in [j0, last]
    const int nt = (last - j0) / kBQ + 1;
    const int nsteps = G * nt;
    prefetch_step(sm, 0, q, dout, lse, delta, b, g * G, j0, T, Hq);
    ptx::cp_async_commit();
    for (int step = 0; step < nsteps; ++step) {
        const int h = g * G + step / nt;
        const int i0 = j0 + (step % nt) * kBQ;
        const int buf = step & 1;
        if (step + 1 < nsteps) {  // the other buffer was released at the end of the last step
            prefetch_step(sm, buf ^ 1, q, dout, lse, delta, b, g * G + (step + 1) / nt,
                          j0 + ((step + 1) % nt) * kBQ, T, Hq);
            ptx::cp_async_commit();
            ptx::cp_async_wait<1>();
        } else {
            ptx::cp_async_wait<0>();
        }
        __syncthreads();  // this step's tiles (every thread's copies) have landed
        {

            // ---- S^T = K_w Q^T and dP^T = V_w dO^T: [16 keys x 32 rows]
            float st[4][4], dpt[4][4];
#pragma unroll
            for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) st[n][e] = dpt[n][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int dA = kk * 16 + 8 * (lane >> 4);   // A: rows kw.. (+8), cols dA
                const int rA = kw + (lane & 7) + 8 * (mi & 1);
                uint32_t ka[4], va[4];
                ptx::ldsm_x4(ptx::smem_u32(sm.k[dA >> 6]) + sw(rA, dA & 63), ka[0], ka[1], ka[2], ka[3]);
                ptx::ldsm_x4(ptx::smem_u32(sm.v[dA >> 6]) + sw(rA, dA & 63), va[0], va[1], va[2], va[3]);
#pragma unroll
                for (int np = 0; np < 2; ++np) {       // B: rows 16np.. (n), cols kk*16 (+8)
                    const int rB = np * 16 + (lane & 7) + 8 * (lane >> 4);
                    const int dB = kk * 16 + 8 * (mi & 1);
                    uint32_t qb[4], ob[4];
                    ptx::ldsm_x4(ptx::smem_u32(sm.q[buf][dB >> 6]) + sw(rB, dB & 63), qb[0], qb[1], qb[2], qb[3]);
                    ptx::ldsm_x4(ptx::smem_u32(sm.dout[buf][dB >> 6]) + sw(rB, dB & 63), ob[0], ob[1], ob[2], ob[3]);
                    ptx::mma_bf16_16816(st[2 * np], ka, qb[0], qb[1]);
                    ptx::mma_bf16_16816(st[2 * np + 1], ka, qb[2], qb[3]);
                    ptx::mma_bf16_16816(dpt[2 * np], va, ob[0], ob[1]);
                    ptx::mma_bf16_16816(dpt[2 * np + 1], va, ob[2], ob[3]);
                }
            }
            // ---- P^T and dS^T (element e: key kw + gq + 8(e>>1), row 8n + 2cq + (e&1))
#pragma unroll
            for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = 8 * n + 2 * cq + (e & 1);
                    const int key = j0 + kw + gq + 8 * (e >> 1);
                    const bool vis = key_visible(i0 + r, key, window) & (key < T) & (i0 + r < T);
                    const float p =
                        vis ? ptx::exp2_approx(st[n][e] * sl2 - sm.lse[buf][r] * kLog2e) : 0.f;
                    st[n][e] = p;
                    dpt[n][e] = p * (dpt[n][e] - sm.delta[buf][r]);
                }
            // ---- dV += P^T dO, dK += dS^T Q  ([16 keys x 128 d], k = 32 rows)
#pragma unroll
            for (int kc = 0; kc < 2; ++kc) {
                uint32_t pa[4], sa[4];
                pa[0] = ptx::pack_bf16x2(st[2 * kc][0], st[2 * kc][1]);
                pa[1] = ptx::pack_bf16x2(st[2 * kc][2], st[2 * kc][3]);
                pa[2] = ptx::pack_bf16x2(st[2 * kc + 1][0], st[2 * kc + 1][1]);
                pa[3] = ptx::pack_bf16x2(st[2 * kc + 1][2], st[2 * kc + 1][3]);
                sa[0] = ptx::pack_bf16x2(dpt[2 * kc][0], dpt[2 * kc][1]);
                sa[1] = ptx::pack_bf16x2(dpt[2 * kc][2], dpt[2 * kc][3]);
                sa[2] = ptx::pack_bf16x2(dpt[2 * kc + 1][0], dpt[2 * kc + 1][1]);
                sa[3] = ptx::pack_bf16x2(dpt[2 * kc + 1][2], dpt[2 * kc + 1][3]);
                const int rB = kc * 16 + (lane & 7) + 8 * (mi & 1);  // k = row
#pragma unroll
                for (int nd = 0; nd < 8; ++nd) {
                    const int dB = nd * 16 + 8 * (lane >> 4);         // n = d
                    uint32_t ob[4], qb[4];
                    ptx::ldsm_x4_t(ptx::smem_u32(sm.dout[buf][dB >> 6]) + sw(rB, dB & 63), ob[0], ob[1], ob[2], ob[3]);
                    ptx::ldsm_x4_t(ptx::smem_u32(sm.q[buf][dB >> 6]) + sw(rB, dB & 63), qb[0], qb[1], qb[2], qb[3]);
                    ptx::mma_bf16_16816(dva[2 * nd], pa, ob[0], ob[1]);
                    ptx::mma_bf16_16816(dva[2 * nd + 1], pa, ob[2], ob[3]);
                    ptx::mma_bf16_16816(dka[2 * nd], sa, qb[0], qb[1]);
                    ptx::mma_bf16_16816(dka[2 * nd + 1], sa, qb[2], qb[3]);
                }
            }
            // ---- dS^T -> shared memory for dQ = dS K
#pragma unroll
            for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int key = kw + gq + 8 * h2, r = 8 * n + 2 * cq;
                    *reinterpret_cast<uint32_t *>(sm.ds + key * kDsStride + r * 2) =
                        ptx::pack_bf16x2(dpt[n][2 * h2], dpt[n][2 * h2 + 1]);
                }
            __syncthreads();
            // ---- dQ [32 rows x 128 d] = dS [32 x 64 keys] K [64 x 128]; warp w: d 32w..32w+31
            float dqa[2][4][4];
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int n = 0; n < 4; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) dqa[m][n][e] = 0.f;
#pragma unroll
            for (int kc = 0; kc < 4; ++kc) {
                uint32_t a[2][4];
#pragma unroll
                for (int m = 0; m < 2; ++m) {  // A = dS rows 16m.., keys 16kc..: from dS^T, transposed
                    const int keyrow = kc * 16 + (lane & 7) + 8 * (lane >> 4);
                    const int rowcol = m * 16 + 8 * (mi & 1);
                    ptx::ldsm_x4_t(ptx::smem_u32(sm.ds + keyrow * kDsStride + rowcol * 2), a[m][0],
                                   a[m][1], a[m][2], a[m][3]);
                }
#pragma unroll
                for (int np = 0; np < 2; ++np) {  // B = K keys 16kc.. (k), d 32w + 16np.. (n)
                    const int rB = kc * 16 + (lane & 7) + 8 * (mi & 1);
                    const int dB = warp * 32 + np * 16 + 8 * (lane >> 4);
                    uint32_t kb[4];
                    ptx::ldsm_x4_t(ptx::smem_u32(sm.k[dB >> 6]) + sw(rB, dB & 63), kb[0], kb[1], kb[2], kb[3]);
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        ptx::mma_bf16_16816(dqa[m][2 * np], a[m], kb[0], kb[1]);
                        ptx::mma_bf16_16816(dqa[m][2 * np + 1], a[m], kb[2], kb[3]);
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int n = 0; n < 4; ++n)
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int i = i0 + m * 16 + gq + 8 * h2;
                        if (i < T) {
                            const int d = warp * 32 + n * 8 + 2 * cq;
                            float *dst = dq_acc + ((static_cast<long>(b) * T + i) * Hq + h) * kD + d;
                            atomicAdd(reinterpret_cast<float2 *>(dst),
                                      make_float2(dqa[m][n][2 * h2], dqa[m][n][2 * h2 + 1]));
                        }
                    }
        }
        __syncthreads();  // done with this step's buffer and ds before they are refilled
    }
    // ---- dK (x scale) and dV of this warp's 16 keys
#pragma unroll
    for (int n = 0; n < 16; ++n)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int key = j0 + kw + gq + 8 * h2;
            if (key < T) {
                const long off = ((static_cast<long>(b) * T + key) * Hkv + g) * kD + n * 8 + 2 * cq;
                *reinterpret_cast<uint32_t *>(dk + off) =
                    ptx::pack_bf16x2(dka[n][2 * h2] * scale, dka[n][2 * h2 + 1] * scale);
                *reinterpret_cast<uint32_t *>(dv + off) =
                    ptx::pack_bf16x2(dva[n][2 * h2], dva[n][2 * h2 + 1]);
            }
        }
}

__global__ void bwd_dq_kernel(const float4 *__restrict__ acc, uint2 *__restrict__ dq, long n4,
                              float scale) {
    for (long x = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; x < n4;
         x += static_cast<long>(gridDim.x) * blockDim.x) {
        const float4 a = acc[x];
        dq[x] = make_uint2(ptx::pack_bf16x2(a.x * scale, a.y * scale),
                           ptx::pack_bf16x2(a.z * scale, a.w * scale));
    }
}

}  // namespace

size_t prefill_backward_workspace(int B, int T, int Hq) {
    const size_t acc = static_cast<size_t>(B) * T * Hq * kD * sizeof(float);
    const size_t del = static_cast<size_t>(B) * Hq * T * sizeof(float);
    return ((acc + 255) & ~static_cast<size_t>(255)) + ((del + 255) & ~static_cast<size_t>(255));
}

cudaError_t launch_prefill_backward(const void *q, const void *k, const void *v, const void *o,
                                    const float *lse, const void *dout, const float *sink,
                                    void *dq, void *dk, void *dv, float *dsink, void *workspace,
                                    int B, int T, int Hq, int Hkv, int window, float scale,
                                    cudaStream_t s) {
    if (B == 0 || T == 0) return cudaMemsetAsync(dsink, 0, sizeof(float) * Hq, s);
    const size_t acc_bytes = static_cast<size_t>(B) * T * Hq * kD * sizeof(float);
    float *acc = static_cast<float *>(workspace);
    float *delta = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                             ((acc_bytes + 255) & ~static_cast<size_t>(255)));
    cudaError_t e = cudaMemsetAsync(acc, 0, acc_bytes, s);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(dsink, 0, sizeof(float) * Hq, s);
    if (e != cudaSuccess) return e;
    bwd_pre_kernel<<<dim3((T + 127) / 128, Hq, B), 256, 0, s>>>(
        static_cast<const __nv_bfloat16 *>(o), static_cast<const __nv_bfloat16 *>(dout), lse, sink,
        delta, dsink, T, Hq);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem = sizeof(BwdSmem) + 128;
    e = cudaFuncSetAttribute(bwd_main_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    bwd_main_kernel<<<dim3((T + kBK - 1) / kBK, Hkv, B), kThreads, smem, s>>>(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<const __nv_bfloat16 *>(v), static_cast<const __nv_bfloat16 *>(dout), lse, delta,
        acc, static_cast<__nv_bfloat16 *>(dk), static_cast<__nv_bfloat16 *>(dv), T, Hq, Hkv, window,
        scale);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long n4 = static_cast<long>(B) * T * Hq * kD / 4;
    bwd_dq_kernel<<<1184, 256, 0, s>>>(reinterpret_cast<const float4 *>(acc),
                                       static_cast<uint2 *>(dq), n4, scale);
    return cudaGetLastError();
}

}  // namespace attn

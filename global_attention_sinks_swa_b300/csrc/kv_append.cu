// KV-cache appends for MTP verify: write the q_len new keys/values of each
// request into the SWA ring (slot p mod R) or the GA paged cache (page
// page_table[b][p / P], offset p % P).  The ring is the fixed-size SWA cache
// of the release announcement ("小米开源 MiMo-V2-Flash", section "将效率推向极限");
// R = W + q_max - 1 holds the union of the windows of the q_max queries of one
// verify pass (figure "Multi-Token Prediction": 1 real + 3 draft tokens).
//
// One block per (request, new-token index); each thread copies 16-byte
// vectors.  Bad indices set a device error bit and skip the copy.  Launched as
// programmatic dependents: a block waits for the preceding kernel's memory
// before its first global access, then lets the next kernel (a verify that
// prefetches its cache while this copy runs) launch.
#include <cuda_bf16.h>

#include "index_math.cuh"
#include "internal.h"
#include "ptx_sm103.cuh"

namespace attn {
namespace {

constexpr unsigned kErrPage = 0x1u, kErrCtx = 0x2u, kErrQlen = 0x4u;

__device__ __forceinline__ bool request_token(const int32_t *cu_q, const int32_t *seq_lens, int b,
                                              int t, int q_max, unsigned *err, int *row, int *pos) {
    const int r0 = cu_q[b], q_len = cu_q[b + 1] - r0, L = seq_lens[b];
    if (q_len > q_max || q_len < 0) {
        if (t == 0 && threadIdx.x == 0) atomicOr(err, kErrQlen);
        return false;
    }
    if (L < q_len) {
        if (t == 0 && threadIdx.x == 0) atomicOr(err, kErrCtx);
        return false;
    }
    if (t >= q_len) return false;
    *row = r0 + t;
    *pos = L - q_len + t;
    return true;
}

__global__ void ring_append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                   const int32_t *__restrict__ cu_q,
                                   const int32_t *__restrict__ seq_lens, uint4 *__restrict__ ring_k,
                                   uint4 *__restrict__ ring_v, int Hkv, int vecs_per_row, int R,
                                   int q_max, unsigned *err) {
    ptx::grid_dep_wait();  // the preceding kernel's writes are visible from here on
    ptx::grid_dep_launch_dependents();
    const int b = blockIdx.x, t = blockIdx.y;
    int row, pos;
    if (!request_token(cu_q, seq_lens, b, t, q_max, err, &row, &pos)) return;
    const int slot = pos % R;
    const int n = Hkv * vecs_per_row;
    for (int x = threadIdx.x; x < n; x += blockDim.x) {
        const int g = x / vecs_per_row, c = x % vecs_per_row;
        const long src = (static_cast<long>(row) * Hkv + g) * vecs_per_row + c;
        const long dst = ((static_cast<long>(b) * Hkv + g) * R + slot) * vecs_per_row + c;
        ring_k[dst] = k_new[src];
        ring_v[dst] = v_new[src];
    }
}

__global__ void paged_append_kernel(const uint4 *__restrict__ k_new,
                                    const uint4 *__restrict__ v_new,
                                    const int32_t *__restrict__ cu_q,
                                    const int32_t *__restrict__ seq_lens,
                                    uint4 *__restrict__ k_pages, uint4 *__restrict__ v_pages,
                                    const int32_t *__restrict__ page_table, int max_pages,
                                    int num_pages, int page_size, int Hkv, int vecs_per_row,
                                    int q_max, unsigned *err) {
    ptx::grid_dep_wait();  // the preceding kernel's writes are visible from here on
    ptx::grid_dep_launch_dependents();
    const int b = blockIdx.x, t = blockIdx.y;
    int row, pos;
    if (!request_token(cu_q, seq_lens, b, t, q_max, err, &row, &pos)) return;
    const int pidx = pos / page_size, off = pos % page_size;
    if (pidx >= max_pages) {
        if (threadIdx.x == 0) atomicOr(err, kErrCtx);
        return;
    }
    const int page = page_table[static_cast<long>(b) * max_pages + pidx];
    if (page < 0 || page >= num_pages) {
        if (threadIdx.x == 0) atomicOr(err, kErrPage);
        return;
    }
    const int n = Hkv * vecs_per_row;
    for (int x = threadIdx.x; x < n; x += blockDim.x) {
        const int g = x / vecs_per_row, c = x % vecs_per_row;
        const long src = (static_cast<long>(row) * Hkv + g) * vecs_per_row + c;
        const long dst =
            ((static_cast<long>(page) * Hkv + g) * page_size + off) * vecs_per_row + c;
        k_pages[dst] = k_new[src];
        v_pages[dst] = v_new[src];
    }
}

// 8-bit pages: the D = 128 bf16 values of a new row of kv head g become 128
// E4M3 codes of value / scale[g]; one thread per 16 values.
__global__ void paged_append_fp8_kernel(const uint4 *__restrict__ k_new,
                                        const uint4 *__restrict__ v_new,
                                        const int32_t *__restrict__ cu_q,
                                        const int32_t *__restrict__ seq_lens,
                                        uint4 *__restrict__ k_pages, uint4 *__restrict__ v_pages,
                                        const int32_t *__restrict__ page_table, int max_pages,
                                        int num_pages, int page_size,
                                        const float *__restrict__ k_scale,
                                        const float *__restrict__ v_scale, int Hkv, int q_max,
                                        unsigned *err) {
    ptx::grid_dep_wait();  // the preceding kernel's writes are visible from here on
    ptx::grid_dep_launch_dependents();
    const int b = blockIdx.x, t = blockIdx.y;
    int row, pos;
    if (!request_token(cu_q, seq_lens, b, t, q_max, err, &row, &pos)) return;
    const int pidx = pos / page_size, off = pos % page_size;
    if (pidx >= max_pages) {
        if (threadIdx.x == 0) atomicOr(err, kErrCtx);
        return;
    }
    const int page = page_table[static_cast<long>(b) * max_pages + pidx];
    if (page < 0 || page >= num_pages) {
        if (threadIdx.x == 0) atomicOr(err, kErrPage);
        return;
    }
    constexpr int kChunks = 128 / 16;  // 16 values per thread
    for (int x = threadIdx.x; x < Hkv * kChunks * 2; x += blockDim.x) {
        const int which = x / (Hkv * kChunks);  // 0: K, 1: V
        const int y = x - which * Hkv * kChunks;
        const int g = y / kChunks, c = y % kChunks;
        const uint4 *src = (which ? v_new : k_new) + ((static_cast<long>(row) * Hkv + g) * 16 + 2 * c);
        const float sc = (which ? v_scale : k_scale)[g];
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 u = src[h];
            const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
            uint16_t code[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(p2[i]);
                code[i] = ptx::f32x2_to_e4m3x2(__fdiv_rn(f.x, sc), __fdiv_rn(f.y, sc));
            }
            w[2 * h] = code[0] | (static_cast<uint32_t>(code[1]) << 16);
            w[2 * h + 1] = code[2] | (static_cast<uint32_t>(code[3]) << 16);
        }
        const long dst = ((static_cast<long>(page) * Hkv + g) * page_size + off) * kChunks + c;
        (which ? v_pages : k_pages)[dst] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

}  // namespace

cudaError_t launch_ring_append(const void *k_new, const void *v_new, const int32_t *cu_q,
                               const int32_t *seq_lens, void *ring_k, void *ring_v, int B, int Hkv,
                               int D, int R, int q_max, int elem_bytes, unsigned int *err,
                               cudaStream_t s) {
    if (B == 0 || q_max == 0) return cudaSuccess;
    const int vpr = D * elem_bytes / 16;
    return launch_pdl(ring_append_kernel, dim3(B, q_max), dim3(128), 0, s,
                      static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), cu_q,
                      seq_lens, static_cast<uint4 *>(ring_k), static_cast<uint4 *>(ring_v), Hkv,
                      vpr, R, q_max, err);
}

cudaError_t launch_paged_append(const void *k_new, const void *v_new, const int32_t *cu_q,
                                const int32_t *seq_lens, void *k_pages, void *v_pages,
                                const int32_t *page_table, int max_pages, int num_pages,
                                int page_size, int B, int Hkv, int D, int q_max, int elem_bytes,
                                unsigned int *err, cudaStream_t s) {
    if (B == 0 || q_max == 0) return cudaSuccess;
    const int vpr = D * elem_bytes / 16;
    return launch_pdl(paged_append_kernel, dim3(B, q_max), dim3(128), 0, s,
                      static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), cu_q,
                      seq_lens, static_cast<uint4 *>(k_pages), static_cast<uint4 *>(v_pages),
                      page_table, max_pages, num_pages, page_size, Hkv, vpr, q_max, err);
}

}  // namespace attn

namespace attn {

cudaError_t launch_paged_append_fp8(const void *k_new, const void *v_new, const int32_t *cu_q,
                                    const int32_t *seq_lens, void *k_pages, void *v_pages,
                                    const int32_t *page_table, int max_pages, int num_pages,
                                    int page_size, const float *k_scale, const float *v_scale,
                                    int B, int Hkv, int q_max, unsigned int *err, cudaStream_t s) {
    if (B == 0 || q_max == 0) return cudaSuccess;
    return launch_pdl(paged_append_fp8_kernel, dim3(B, q_max), dim3(128), 0, s,
                      static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), cu_q,
                      seq_lens, static_cast<uint4 *>(k_pages), static_cast<uint4 *>(v_pages),
                      page_table, max_pages, num_pages, page_size, k_scale, v_scale, Hkv, q_max,
                      err);
}

}  // namespace attn

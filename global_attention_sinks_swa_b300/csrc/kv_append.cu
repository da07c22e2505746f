// KV-cache appends for MTP verify: write the q_len new keys/values of each
// request into the SWA ring (slot p mod R) or the GA paged cache (page
// page_table[b][p / P], offset p % P).  The ring is the fixed-size SWA cache
// of the release announcement ("小米开源 MiMo-V2-Flash", section "将效率推向极限");
// R = W + q_max - 1 holds the union of the windows of the q_max queries of one
// verify pass (figure "Multi-Token Prediction": 1 real + 3 draft tokens).
//
// One block per (request, new-token index); each thread copies 16-byte
// vectors.  Bad indices set a device error bit and skip the copy.
#include "index_math.cuh"
#include "internal.h"

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

}  // namespace

cudaError_t launch_ring_append(const void *k_new, const void *v_new, const int32_t *cu_q,
                               const int32_t *seq_lens, void *ring_k, void *ring_v, int B, int Hkv,
                               int D, int R, int q_max, int elem_bytes, unsigned int *err,
                               cudaStream_t s) {
    if (B == 0 || q_max == 0) return cudaSuccess;
    const int vpr = D * elem_bytes / 16;
    ring_append_kernel<<<dim3(B, q_max), 128, 0, s>>>(
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), cu_q, seq_lens,
        static_cast<uint4 *>(ring_k), static_cast<uint4 *>(ring_v), Hkv, vpr, R, q_max, err);
    return cudaGetLastError();
}

cudaError_t launch_paged_append(const void *k_new, const void *v_new, const int32_t *cu_q,
                                const int32_t *seq_lens, void *k_pages, void *v_pages,
                                const int32_t *page_table, int max_pages, int num_pages,
                                int page_size, int B, int Hkv, int D, int q_max, int elem_bytes,
                                unsigned int *err, cudaStream_t s) {
    if (B == 0 || q_max == 0) return cudaSuccess;
    const int vpr = D * elem_bytes / 16;
    paged_append_kernel<<<dim3(B, q_max), 128, 0, s>>>(
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), cu_q, seq_lens,
        static_cast<uint4 *>(k_pages), static_cast<uint4 *>(v_pages), page_table, max_pages,
        num_pages, page_size, Hkv, vpr, q_max, err);
    return cudaGetLastError();
}

}  // namespace attn

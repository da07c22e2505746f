// Index dumps: replay the kernels' tile schedules and masks (the same
// functions from index_math.cuh) and write integer results the tests compare
// bit for bit with the definitions (visible iff 0 <= j <= i and, for SWA,
// j >= i - W + 1; ring slot p mod R; page page_table[b][p / P]).
#include "index_math.cuh"
#include "internal.h"
#include "tc_tile.cuh"

namespace attn {
namespace {

// mode 0: GA tiling (two 128-row query tiles per CTA, key tiles of 128;
// interior tiles admit every pair without a mask).  One thread per query row.
__global__ void visits_ga_kernel(int32_t *visits, int T, int window) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= T) return;
    const int qs = (i / kTileM) * kTileM;  // start of this row's query tile
    int first, last;
    ga_key_tiles(qs, T, window, &first, &last);
    for (int j = first; j <= last; ++j) {
        const bool masked = ga_tile_needs_mask(qs, j, window);
        for (int c = 0; c < kTileN; ++c) {
            const int kp = j * kTileN + c;
            if (kp >= T) break;
            if (!masked || key_visible(i, kp, window)) visits[static_cast<long>(i) * T + kp] += 1;
        }
    }
}

// mode 1: packed SWA tiling, G heads x 128/G tokens per tile; head 0 only.
__global__ void visits_swa_kernel(int32_t *visits, int T, int window, int G) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= T) return;
    const int TT = swa_pack_tokens(G);
    const int i0 = (i / TT) * TT;
    const int key0 = swa_pack_key0(i0, G, window), N = swa_pack_keys(G, window);
    for (int c = 0; c < N; ++c) {
        const int kp = key0 + c;
        if (kp >= 0 && kp < T && key_visible(i, kp, window))
            visits[static_cast<long>(i) * T + kp] += 1;
    }
}

// Streaming SWA schedule: one thread per CTA of the kernel's grid replays
// that CTA's run of tiles, the ring bookkeeping (which key block each ring
// slot holds when a tile reads it) and the admitted columns, for query head 0
// of each kv group.  visits [B*Hkv, T, T+1]; column T counts admitted keys
// outside [0, T).
__global__ void swa_stream_visits_kernel(int32_t *visits, int B, int T, int Hkv, int window,
                                         int grid) {
    const int cta = blockIdx.x * blockDim.x + threadIdx.x;
    if (cta >= grid) return;
    const int32_t *cu = nullptr;  // equal lengths (the packed order is replayed on the host)
    const int total = B * T;
    const int ntiles = swa_total_tiles(cu, B, T, total, Hkv);
    int u0, u1;
    swa_stream_range(cta, grid, ntiles, &u0, &u1);
    if (u0 >= u1) return;
    SwaRingCursor cur;
    SwaTileCursor t = swa_cursor_at(cu, B, T, total, Hkv, u0);
    int slot_key[kSwaRingBlocks];
    for (int s = 0; s < kSwaRingBlocks; ++s) slot_key[s] = -(1 << 30);
    for (int u = u0; u < u1; ++u) {
        if (u > u0) swa_cursor_next(t, cu, B, T, total, Hkv);
        const int bg = t.b * Hkv + t.g, i0 = t.blk * kSwaTokens;
        const int key0 = i0 + kSwaTokens - kSwaKeys;
        swa_ring_step(cur, bg, kSwaTileBlocks);
        for (int s = cur.first_new; s < cur.first_new + cur.n_new; ++s)
            slot_key[s % kSwaRingBlocks] = key0 + kSwaBlockKeys * (s - cur.base);
        const bool interior = key0 >= 0;
        for (int tt = 0; tt < kSwaTokens; ++tt) {
            const int qpos = i0 + tt;
            if (qpos >= t.len) break;
            int c_lo, c_hi;
            swa_row_cols(qpos, key0, window, &c_lo, &c_hi);
            int32_t *row = visits + (static_cast<long>(bg) * T + qpos) * (T + 1);
            for (int j = 0; j < kSwaTileBlocks; ++j) {
                const int kb = slot_key[(cur.base + j) % kSwaRingBlocks];
                for (int cc = 0; cc < kSwaBlockKeys; ++cc) {
                    if (!swa_col_admitted(j * kSwaBlockKeys + cc, c_lo, c_hi, interior)) continue;
                    const int key = kb + cc;
                    atomicAdd(&row[(key >= 0 && key < t.len) ? key : T], 1);
                }
            }
        }
    }
}

__global__ void verify_positions_kernel(int32_t *out, int kind, const int32_t *cu_q,
                                        const int32_t *seq_lens, int q_max, int window, int R,
                                        int max_pages, int page_size) {
    const int b = blockIdx.x, t = blockIdx.y;
    const int L = seq_lens[b], q_len = cu_q[b + 1] - cu_q[b];
    const int i = L - q_len + t;  // query position
    if (kind == 0) {
        // visibility as the tensor-core ring kernel decides it (two slot
        // intervals), positions as both ring kernels compute them
        const RingVisible vis = ring_visible_slots(L, R, window, i);
        for (int s = threadIdx.x; s < R; s += blockDim.x) {
            const int p = ring_slot_position(s, L, R);
            out[(static_cast<long>(b) * q_max + t) * R + s] = (t < q_len && vis.contains(s)) ? p : -1;
        }
    } else {
        const long n = static_cast<long>(max_pages) * page_size;
        int32_t *o = out + (static_cast<long>(b) * q_max + t) * n;
        for (long x = threadIdx.x; x < n; x += blockDim.x) o[x] = -1;
        __syncthreads();
        if (t >= q_len) return;
        const int nsplit = verify_num_splits(max_pages * page_size, kVerifyChunkPages * page_size);
        for (int s = 0; s < nsplit; ++s) {
            int pb, pe;
            verify_split_pages(s, L, page_size, kVerifyChunkPages, &pb, &pe);
            for (int pi = pb; pi < pe; ++pi)
                for (int off = threadIdx.x; off < page_size; off += blockDim.x) {
                    const int p = pi * page_size + off;
                    if (key_visible(i, p, 0)) o[p] = p;
                }
        }
    }
}

// A pipeline wait that nothing completes: thread 0 waits on a fresh mbarrier
// with the kernels' bounded wait, which gives up after its time limit and
// records the wait-timeout bit exactly as a stalled pipeline would.
__global__ void wait_timeout_kernel(unsigned *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !ptx::mbar_wait(&bar, 0)) atomicOr(err, tc::kErrWait);
}

}  // namespace

cudaError_t launch_debug_prefill_visits(int32_t *visits, int mode, int T, int window, int G,
                                        cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    cudaError_t e = cudaMemsetAsync(visits, 0, sizeof(int32_t) * static_cast<size_t>(T) * T, s);
    if (e != cudaSuccess) return e;
    const int blocks = (T + 127) / 128;
    if (mode == 0)
        visits_ga_kernel<<<blocks, 128, 0, s>>>(visits, T, window);
    else
        visits_swa_kernel<<<blocks, 128, 0, s>>>(visits, T, window, G);
    return cudaGetLastError();
}

cudaError_t launch_debug_swa_stream_visits(int32_t *visits, int B, int T, int Hkv, int window,
                                           int grid, cudaStream_t s) {
    if (B == 0 || T == 0 || grid == 0) return cudaSuccess;
    cudaError_t e = cudaMemsetAsync(
        visits, 0, sizeof(int32_t) * static_cast<size_t>(B) * Hkv * T * (T + 1), s);
    if (e != cudaSuccess) return e;
    swa_stream_visits_kernel<<<(grid + 127) / 128, 128, 0, s>>>(visits, B, T, Hkv, window, grid);
    return cudaGetLastError();
}

cudaError_t launch_debug_verify_positions(int32_t *out, int kind, const int32_t *cu_q,
                                          const int32_t *seq_lens, int B, int q_max, int window,
                                          int R, int max_pages, int page_size, cudaStream_t s) {
    if (B == 0 || q_max == 0) return cudaSuccess;
    verify_positions_kernel<<<dim3(B, q_max), 128, 0, s>>>(out, kind, cu_q, seq_lens, q_max,
                                                          window, R, max_pages, page_size);
    return cudaGetLastError();
}

cudaError_t launch_debug_wait_timeout(unsigned *err, cudaStream_t s) {
    wait_timeout_kernel<<<1, 32, 0, s>>>(err);
    return cudaGetLastError();
}

}  // namespace attn

// Host-side interface between the C ABI (attn_api.cu) and the kernel files.
// Each launcher only enqueues; argument validation happens in attn_api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

// Launches `kernel` with programmatic stream serialization: it may begin while
// the preceding kernel of the stream is still running (once that kernel lets
// dependents launch), so every kernel launched this way calls
// ptx::grid_dep_wait() before it reads or writes global memory.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Sequences of a prefill batch: B sequences of T tokens each (cu == nullptr,
// total = B*T), or B packed sequences given by the device array cu[B+1] with
// cu[B] = total tokens and T >= the longest one (T sizes grids only).
struct PrefillBatch {
    const int32_t *cu;
    int B, T, total;
};

// fp32 CUDA-core prefill (window <= 0: global attention).  The output is
// multiplied by vscale.
cudaError_t launch_prefill_f32(const float *q, const float *k, const float *v, const float *sink,
                               float *o, float *lse, const PrefillBatch &pb, int Hq, int Hkv,
                               int D, int window, float scale, float vscale, unsigned int *err,
                               cudaStream_t s);

// Tensor maps of a bf16 prefill problem (built by attn_api.cu).
struct PrefillMaps {
    CUtensorMap q;  // box rows of Q  (layout depends on the kernel)
    CUtensorMap k;  // key tile
    CUtensorMap v;  // value tile
    CUtensorMap o;  // output store
    void *out;      // output base pointer (kernels that store O without TMA)
};

// The prefill maps view Q, K, V and O as [total tokens, heads, D] (3-D).
// tcgen05 GA-tiled prefill (full causal, or window-limited when window > 0).
cudaError_t launch_prefill_ga_tc(const PrefillMaps &maps, const float *sink, float *lse,
                                 const PrefillBatch &pb, int Hq, int Hkv, int window, float scale,
                                 float vscale, unsigned int *err, cudaStream_t s);
// tcgen05 streaming SWA prefill (G = 8: 16 tokens x 8 heads per tile, window
// in [114, 129]); one persistent CTA per SM over prefill_swa_grid() CTAs.
cudaError_t launch_prefill_swa_tc(const PrefillMaps &maps, const float *sink, float *lse,
                                  const PrefillBatch &pb, int Hq, int Hkv, int window, float scale,
                                  float vscale, unsigned int *err, cudaStream_t s);
int prefill_swa_tc_supported(int G, int window);
// CTAs of the streaming kernel for a batch of at most max_tiles tiles.
int prefill_swa_grid(long max_tiles);

// Backward of the bf16 prefill (D = 128, batches of equal length): dq, dk, dv
// (bf16) and dsink (fp32), from q, k, v, the forward's o and lse, and dout.
// The maps view q/dout [B*T, Hq, 128] and k/v [B*T, Hkv, 128] with boxes of
// (64, 1, rows) for the row counts in their names.
struct BwdMaps {
    CUtensorMap q_rows64, dout_rows64, k_rows128, v_rows128;   // dK/dV kernel
    CUtensorMap q_rows128, dout_rows128, k_rows64, v_rows64;   // dQ kernel
};
size_t prefill_backward_workspace(int B, int T, int Hq);
cudaError_t launch_prefill_backward(const BwdMaps &maps, const void *o, const float *lse,
                                    const void *dout, const float *sink, void *dq, void *dk,
                                    void *dv, float *dsink, void *workspace, int B, int T, int Hq,
                                    int Hkv, int window, float scale, unsigned int *err,
                                    cudaStream_t s);

// KV-cache appends (plain 16-byte copies).
cudaError_t launch_ring_append(const void *k_new, const void *v_new, const int32_t *cu_q,
                               const int32_t *seq_lens, void *ring_k, void *ring_v, int B, int Hkv,
                               int D, int R, int q_max, int elem_bytes, unsigned int *err,
                               cudaStream_t s);
cudaError_t launch_paged_append(const void *k_new, const void *v_new, const int32_t *cu_q,
                                const int32_t *seq_lens, void *k_pages, void *v_pages,
                                const int32_t *page_table, int max_pages, int num_pages,
                                int page_size, int B, int Hkv, int D, int q_max, int elem_bytes,
                                unsigned int *err, cudaStream_t s);
// 8-bit paged append: bf16 new rows -> E4M3 codes of row / scale[kv head]
// (fp32 division, round to nearest even, saturated at 448), D = 128.
cudaError_t launch_paged_append_fp8(const void *k_new, const void *v_new, const int32_t *cu_q,
                                    const int32_t *seq_lens, void *k_pages, void *v_pages,
                                    const int32_t *page_table, int max_pages, int num_pages,
                                    int page_size, const float *k_scale, const float *v_scale,
                                    int B, int Hkv, int q_max, unsigned int *err, cudaStream_t s);

// Verify (bf16, D = 128, mma.sync tensor cores, TMA-staged K/V).
struct VerifyMaps {
    CUtensorMap k;  // [.., Hkv, 64-row block, D] view of the ring or page pool
    CUtensorMap v;
    CUtensorMap q;  // tensor-core ring kernel: [B*q_max, Hq, D] view of q (boxes of 8 heads)
};
constexpr int kVerifyRows = 32;       // q_max * G rows per (request, kv head), padded
constexpr int kVerifyBlock = 64;      // keys per pipeline stage (one GA page)
constexpr int kVerifyChunkPages = 64; // pages per split of the GA context (4096 tokens)

// tcgen05 ring verify: persistent CTAs over (request, kv head) units, the
// whole ring of a unit in one pass; K/V maps with a box of kVerifyRingKeys
// slot rows.
constexpr int kVerifyRingKeys = 144;  // ring slots covered (R <= 144), multiple of 16
constexpr int kVerifyRingUnitsPerCta = 64;  // (request, kv head) units per persistent CTA, at most
int verify_ring_tc_supported(int G, int R, int q_max);
cudaError_t launch_verify_ring_tc(const VerifyMaps &maps, const int32_t *cu_q,
                                  const int32_t *seq_lens, const float *sink, void *o, int B,
                                  int Hq, int Hkv, int window, int R, int q_max, float scale,
                                  unsigned int *err, cudaStream_t s);
cudaError_t launch_verify_ring(const VerifyMaps &maps, const void *q, const int32_t *cu_q,
                               const int32_t *seq_lens, const float *sink, void *o, int B, int Hq,
                               int Hkv, int window, int R, int q_max, float scale,
                               unsigned int *err, cudaStream_t s);
cudaError_t launch_verify_paged(const VerifyMaps &maps, const void *q, const int32_t *cu_q,
                                const int32_t *seq_lens, const int32_t *page_table, int max_pages,
                                int num_pages, const float *sink, void *o, float *ws_o,
                                float *ws_ml, int nsplit, int B, int Hq, int Hkv, int q_max,
                                int max_ctx, float scale, const float *k_scale,
                                const float *v_scale, unsigned int *err, cudaStream_t s);

// Index dumps.
cudaError_t launch_debug_prefill_visits(int32_t *visits, int mode, int T, int window, int G,
                                        cudaStream_t s);
cudaError_t launch_debug_swa_stream_visits(int32_t *visits, int B, int T, int Hkv, int window,
                                           int grid, cudaStream_t s);
cudaError_t launch_debug_verify_positions(int32_t *out, int kind, const int32_t *cu_q,
                                          const int32_t *seq_lens, int B, int q_max, int window,
                                          int R, int max_pages, int page_size, cudaStream_t s);

}  // namespace attn

/*
 * attn_sink.h -- C ABI of the B300 (sm_103a) sink-attention library.
 *
 * The operation: causal attention with a per-query-head learnable "sink"
 * logit that joins the softmax denominator and carries no value, over either a
 * sliding window of W keys (SWA layers, W = 128) or the full causal prefix
 * (global-attention, GA, layers), in two modes: prefill over whole sequences,
 * and the MTP self-speculative verify step that scores 1 real + up to 3 draft
 * tokens per request against that request's KV cache.
 *
 * Sources (MiMo-V2-Flash):
 *   [ARCH]   technical-report summary (fanfer.top, "MiMo-V2"), section
 *            "MiMo-V2-Flash Model Architecture": 5 SWA layers then 1 GA layer
 *            per hybrid block, sliding window W = 128.
 *   [SINK]   same summary, section "Hybrid Sliding Window Attention
 *            Architecture": learnable attention-sink bias in the gpt-oss style.
 *            The formula that followed was lost from the page; this library
 *            implements the reading "one extra softmax column per query head,
 *            logit sigma_h compared unscaled with the scaled scores, zero value".
 *   [KV]     release announcement (aihot.news, "小米开源 MiMo-V2-Flash"), section
 *            "将效率推向极限": SWA keeps a fixed-size KV cache.
 *   [MTP]    same announcement, figure "Multi-Token Prediction": the main model
 *            verifies token i and drafts i+1..i+3 in one pass and keeps the
 *            accepted prefix; summary section "MTP加速" (16K in / 1K out).
 *   [SERVE]  summary section "MTP加速": serving measured with 16K-token prompts
 *            at several in-node batch sizes (batches of prompts of unequal
 *            length, packed here by cu_seqlens).
 *   [FP8]    technical-report summary, section "MiMo-V2-Flash Model Architecture":
 *            an FP8 mixed-precision framework; dpshk.com article, section
 *            "关键配置参数": FP8 quantization enabled at inference to cut memory.
 *            Verify is bound by reading the cache, so 8-bit GA pages halve the
 *            bytes of a verify step.
 *   [CFG]    dpshk.com article on MiMo-V2-Flash-Base ("小米AI团队揭秘"), section
 *            "轻量级多token预测技术": config.json lists attention_value_scale =
 *            0.707 without saying what it scales; read here as a factor on the
 *            attention output (equivalently on V).
 *
 * Definition (all entry points):  for query position i of head h (kv head
 * g = h / (Hq/Hkv)), visible keys j satisfy 0 <= j <= i and, for SWA,
 * j >= i - W + 1.  With S_j = scale * <q_i, k_j>,
 *     m = max(sigma_h, max_j S_j),  Z = e^(sigma_h - m) + sum_j e^(S_j - m),
 *     o_i = sum_j e^(S_j - m) / Z * v_j,     lse_i = m + ln Z.
 * sigma_h = +inf gives o_i = 0; sigma_h = -inf is plain softmax attention.
 *
 * Conventions:
 *   - every pointer argument is a DEVICE pointer owned by the caller, except
 *     where marked (host); the library never allocates and keeps no state
 *     between calls other than a device error word;
 *   - every call only enqueues work on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and returns without synchronising;
 *   - tensors are dense row-major; q/k/v/o/cache pointers must be 16-byte
 *     aligned (ATTN_ERR_INVALID_ARG otherwise);
 *   - argument errors detectable on the host return ATTN_ERR_INVALID_ARG or
 *     ATTN_ERR_UNSUPPORTED before anything is enqueued; attn_last_error()
 *     then describes the problem;
 *   - errors only the device can see (a page id outside the pool, a sequence
 *     longer than the cache, q_len > q_max, a pipeline wait that timed out)
 *     set bits in a device error word, the offending work is skipped (never a
 *     trap), and attn_check_device_error() reports them;
 *   - while ATTN_DEVERR_WAIT_TIMEOUT is set, the pipelined kernels (the
 *     tensor-core prefill, verify and backward kernels, the ones with bounded
 *     barrier waits) return without doing any work, so a stalled pipeline is
 *     not run into again: their outputs keep their previous contents (the
 *     backward still writes dsink).  The fp32 prefill and the appends run as
 *     usual.  attn_check_device_error() clears the word.
 */
#ifndef ATTN_SINK_H
#define ATTN_SINK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum attn_status {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,   /* bad size, null or misaligned pointer        */
    ATTN_ERR_UNSUPPORTED = 2,   /* well-formed but not implemented (e.g. D)    */
    ATTN_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed           */
    ATTN_ERR_DEVICE_FAULT = 4   /* the device error word is non-zero           */
} attn_status_t;

typedef enum attn_dtype {
    ATTN_BF16 = 0,              /* bf16 I/O, fp32 accumulation, P rounded to bf16 before PV */
    ATTN_F32 = 1                /* fp32 I/O and fp32 arithmetic on CUDA cores (no TF32)     */
} attn_dtype_t;

/* Bits of the device error word. */
#define ATTN_DEVERR_PAGE_OOB     0x1u  /* page_table entry outside [0, num_pages)           */
#define ATTN_DEVERR_CTX_OOB      0x2u  /* seq_len > max_ctx, > max_pages*page_size, or < q_len */
#define ATTN_DEVERR_QLEN         0x4u  /* cu_q gives q_len > q_max                          */
#define ATTN_DEVERR_WAIT_TIMEOUT 0x8u  /* an in-kernel pipeline wait exceeded its time limit  */
#define ATTN_DEVERR_SEQLENS      0x10u /* a packed prefill batch gave an invalid sequence span */

/* Library version (major*10000 + minor*100 + patch). */
int attn_version(void);

/* Thread-local description of the last host-side error ("" if none).  The
 * string stays valid until the next call from the same thread. */
const char *attn_last_error(void);

/* Synchronises `stream`, reads and clears the device error word of the current
 * device.  *bits_out (host, may be NULL) receives the ATTN_DEVERR_* bits.
 * Returns ATTN_OK when the word was zero, ATTN_ERR_DEVICE_FAULT when not, and
 * ATTN_ERR_CUDA when the synchronisation itself failed. */
attn_status_t attn_check_device_error(void *stream, unsigned int *bits_out);

/* ---------------------------------------------------------------- prefill ---
 * Sliding-window prefill [ARCH][SINK].
 *   q [B,T,Hq,D], k [B,T,Hkv,D], v [B,T,Hkv,D], o [B,T,Hq,D]   (dtype)
 *   sink [Hq] fp32 logits;  lse [B,Hq,T] fp32 natural-log LSE, or NULL
 *   window >= 1 (keys i-window+1..i);  scale > 0 (usually 1/sqrt(D))
 * Supported: ATTN_BF16 with D = 128 and 128 % (Hq/Hkv) == 0 on the tensor cores
 * (Hq/Hkv = 8 with window in [114, 129] on the streaming kernel, any other
 * ratio or window on the GA-tiled kernel with window-limited tile skipping);
 * ATTN_F32 with D in {64,128} on the fp32 CUDA-core path.
 * While ATTN_DEVERR_WAIT_TIMEOUT is set (conventions above) the bf16
 * tensor-core kernels of this call return at once and o / lse keep their
 * previous contents: a caller that never polls attn_check_device_error()
 * cannot tell, so poll after each step or batch of steps. */
attn_status_t attn_swa_sink_prefill(const void *q, const void *k, const void *v, const float *sink,
                                    void *o, float *lse, int B, int T, int Hq, int Hkv, int D,
                                    int window, float scale, attn_dtype_t dtype, void *stream);

/* Global (full causal) prefill [ARCH][SINK]; arguments, kernel support and the
 * behaviour under ATTN_DEVERR_WAIT_TIMEOUT as above, without window. */
attn_status_t attn_ga_sink_prefill(const void *q, const void *k, const void *v, const float *sink,
                                   void *o, float *lse, int B, int T, int Hq, int Hkv, int D,
                                   float scale, attn_dtype_t dtype, void *stream);

/* Packed (variable-length) prefill [ARCH][SINK][SERVE], with the output scale
 * of the model configuration [CFG] (attention_value_scale).
 *   q [total,Hq,D], k [total,Hkv,D], v [total,Hkv,D], o [total,Hq,D]   (dtype)
 *   cu_seqlens [B+1] int32 on the device: sequence b is tokens cu_seqlens[b] ..
 *     cu_seqlens[b+1]-1 with positions 0 .. len-1; cu_seqlens[0] = 0 and
 *     cu_seqlens[B] = total_tokens.  Sequences never see each other's keys.
 *   max_seqlen >= every length (sizes the grid);  lse [Hq,total] fp32 or NULL
 *   value_scale multiplies the output (o = value_scale * sum_j p_ij v_j; the
 *     LSE is unscaled); 1 gives the plain definition.
 * A span that is decreasing, outside [0, total_tokens) or longer than
 * max_seqlen is skipped (its rows are not written) and sets
 * ATTN_DEVERR_SEQLENS.  Everything else as in the calls above (same dtype,
 * D and kernel support; the sliding-window form keeps window >= 1; while
 * ATTN_DEVERR_WAIT_TIMEOUT is set the bf16 kernels write nothing). */
attn_status_t attn_swa_sink_prefill_varlen(const void *q, const void *k, const void *v,
                                           const int32_t *cu_seqlens, const float *sink, void *o,
                                           float *lse, int B, int total_tokens, int max_seqlen,
                                           int Hq, int Hkv, int D, int window, float scale,
                                           float value_scale, attn_dtype_t dtype, void *stream);
attn_status_t attn_ga_sink_prefill_varlen(const void *q, const void *k, const void *v,
                                          const int32_t *cu_seqlens, const float *sink, void *o,
                                          float *lse, int B, int total_tokens, int max_seqlen,
                                          int Hq, int Hkv, int D, float scale, float value_scale,
                                          attn_dtype_t dtype, void *stream);

/* ---------------------------------------------------------------- backward ---
 * Gradients of the bf16 prefill [SINK][ARCH] (the sinks are learnable, so
 * dsink is part of it), batches of equal length, D = 128:
 *   inputs  q [B,T,Hq,D], k, v [B,T,Hkv,D], o [B,T,Hq,D] and lse [B,Hq,T] of
 *           the forward call with the same arguments (lse from its `lse`
 *           output), dout [B,T,Hq,D] = dL/do, sink [Hq];
 *   outputs dq [B,T,Hq,D], dk, dv [B,T,Hkv,D] (bf16), dsink [Hq] fp32
 *           (overwritten, not accumulated);
 *   window 0 = global attention, else the sliding window; scale as forward.
 * dS_ij = P_ij (<dout_i, v_j> - D_i) with D_i = <dout_i, o_i> and P from the
 * lse; dsink_h = -sum_i p_sink,i D_i.  `workspace` (device, 256-byte
 * aligned, attn_sink_prefill_backward_workspace bytes = 4*B*Hq*T rounded up
 * to 256) holds D; its contents need no initialisation.  dq, dk and dv are
 * computed on the tensor cores without atomics, so repeated calls give
 * identical results.  While ATTN_DEVERR_WAIT_TIMEOUT is set only dsink is
 * written (dq, dk, dv keep their previous contents): poll
 * attn_check_device_error(). */
size_t attn_sink_prefill_backward_workspace(int B, int T, int Hq, int D);
attn_status_t attn_sink_prefill_backward(const void *q, const void *k, const void *v,
                                         const void *o, const float *lse, const void *dout,
                                         const float *sink, void *dq, void *dk, void *dv,
                                         float *dsink, void *workspace, size_t workspace_bytes,
                                         int B, int T, int Hq, int Hkv, int D, int window,
                                         float scale, attn_dtype_t dtype, void *stream);

/* ------------------------------------------------------------ KV caches ---
 * SWA ring [KV][MTP]: ring_k, ring_v [B,Hkv,R,D] with R = ring_slots >=
 * window + q_max - 1 (131 for W = 128, q_max = 4); position p of request b
 * lives in slot p mod R.
 * GA paged cache: k_pages, v_pages [num_pages,Hkv,page_size,D] (page_size =
 * 64), page_table [B,max_pages] int32; position p of request b lives in page
 * page_table[b, p / page_size] at offset p % page_size.
 *
 * Append: request b's q_len = cu_q[b+1]-cu_q[b] new tokens (k_new, v_new
 * [cu_q[B],Hkv,D], rows cu_q[b]..) take positions seq_lens[b]-q_len ..
 * seq_lens[b]-1 (seq_lens counts them).  cu_q [B+1], seq_lens [B] int32. */
attn_status_t attn_swa_ring_append(const void *k_new, const void *v_new, const int32_t *cu_q,
                                   const int32_t *seq_lens, void *ring_k, void *ring_v,
                                   int B, int Hkv, int D, int ring_slots, int q_max,
                                   attn_dtype_t dtype, void *stream);

attn_status_t attn_ga_paged_append(const void *k_new, const void *v_new, const int32_t *cu_q,
                                   const int32_t *seq_lens, void *k_pages, void *v_pages,
                                   const int32_t *page_table, int max_pages, int num_pages,
                                   int page_size, int B, int Hkv, int D, int q_max,
                                   attn_dtype_t dtype, void *stream);

/* 8-bit GA paged cache [FP8]: k_pages, v_pages [num_pages,Hkv,page_size,D]
 * uint8 E4M3 codes (sign, 4 exponent bits with bias 7, 3 mantissa bits; no
 * infinities; largest finite 448); entry = code * k_scale[g] (v_scale[g] for
 * V), k_scale/v_scale [Hkv] fp32 on the device, chosen by the caller.  The
 * append takes bf16 k_new/v_new [cu_q[B],Hkv,D] and stores the code of
 * value / scale (fp32 division, round to nearest even, finite values beyond
 * 448 saturated).  D = 128; errors as for attn_ga_paged_append. */
attn_status_t attn_ga_paged_append_fp8(const void *k_new, const void *v_new,
                                       const int32_t *cu_q, const int32_t *seq_lens,
                                       void *k_pages, void *v_pages, const int32_t *page_table,
                                       int max_pages, int num_pages, int page_size,
                                       const float *k_scale, const float *v_scale, int B, int Hkv,
                                       int D, int q_max, void *stream);

/* ----------------------------------------------------------------- verify ---
 * MTP verify [MTP]: request b scores its q_len = cu_q[b+1]-cu_q[b] <= q_max
 * new tokens (positions seq_lens[b]-q_len .. seq_lens[b]-1, already appended)
 * against its cache; draft t sees the history and drafts 0..t.
 *   q, o [cu_q[B],Hq,D] (dtype);  sink [Hq] fp32;  q_max <= 4.
 * Rejected drafts are rolled back by the caller lowering seq_lens; the next
 * append overwrites their slots.  Supported: ATTN_BF16, D = 128,
 * q_max * (Hq/Hkv) <= 32.  While ATTN_DEVERR_WAIT_TIMEOUT is set the verify
 * kernels (and the split-KV merge) write nothing and o keeps its previous
 * contents: poll attn_check_device_error() after each step. */
attn_status_t attn_swa_sink_verify(const void *q, const int32_t *cu_q, const void *ring_k,
                                   const void *ring_v, const int32_t *seq_lens, const float *sink,
                                   void *o, int B, int Hq, int Hkv, int D, int window,
                                   int ring_slots, int q_max, float scale, attn_dtype_t dtype,
                                   void *stream);

/* Bytes of scratch that attn_ga_sink_verify needs for these sizes (split-KV
 * partial results).  max_ctx bounds every seq_lens[b]. */
size_t attn_ga_sink_verify_workspace(int B, int Hq, int Hkv, int D, int q_max, int max_ctx);

/* GA verify over the paged cache, split over chunks of the context and merged
 * by log-sum-exp; the sink enters once, in the merge.  `workspace` is a device
 * buffer of at least attn_ga_sink_verify_workspace(...) bytes, 256-byte
 * aligned, owned by the caller; its contents need no initialisation and are
 * garbage afterwards.  Calls that share a workspace must not overlap. */
attn_status_t attn_ga_sink_verify(const void *q, const int32_t *cu_q, const void *k_pages,
                                  const void *v_pages, const int32_t *page_table, int max_pages,
                                  int num_pages, int page_size, const int32_t *seq_lens,
                                  const float *sink, void *o, void *workspace,
                                  size_t workspace_bytes, int B, int Hq, int Hkv, int D,
                                  int q_max, int max_ctx, float scale, attn_dtype_t dtype,
                                  void *stream);

/* GA verify over the 8-bit paged cache [FP8] (layout and scales as for
 * attn_ga_paged_append_fp8): half the cache bytes of attn_ga_sink_verify per
 * token.  q and o bf16; the codes become f16 exactly, and both products run
 * with f16 operands (q rounded to f16, so |q| must stay below 65504) and
 * fp32 accumulation.  Workspace, sizes and errors as attn_ga_sink_verify. */
attn_status_t attn_ga_sink_verify_fp8(const void *q, const int32_t *cu_q, const void *k_pages,
                                      const void *v_pages, const int32_t *page_table,
                                      int max_pages, int num_pages, int page_size,
                                      const int32_t *seq_lens, const float *sink,
                                      const float *k_scale, const float *v_scale, void *o,
                                      void *workspace, size_t workspace_bytes, int B, int Hq,
                                      int Hkv, int D, int q_max, int max_ctx, float scale,
                                      void *stream);

/* The same GA verify for callers that cannot allocate device memory (for
 * example code inside a host program that reserved all device memory up front
 * in its own pool and allows no later cudaMalloc, or a decode loop that must
 * not pay an allocation's latency and possible device synchronisation).  It
 * allocates nothing: the split-KV partials go to a 64 MiB file-scope device
 * array inside the library, which every GPU that loads the library holds until
 * the process exits.  The pages have no counterpart to this entry point.
 *   - Arguments and results as attn_ga_sink_verify, without the workspace.
 *   - Sizes whose scratch (attn_ga_sink_verify_workspace) exceeds 64 MiB are
 *     rejected with ATTN_ERR_UNSUPPORTED before anything is enqueued.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents;
 *     every value a call reads is written earlier in the same call, so nothing
 *     needs clearing.  Calls that overlap on the GPU (other streams, other
 *     host threads on the same device) race on the array. */
attn_status_t attn_ga_sink_verify_noalloc(const void *q, const int32_t *cu_q, const void *k_pages,
                                          const void *v_pages, const int32_t *page_table,
                                          int max_pages, int num_pages, int page_size,
                                          const int32_t *seq_lens, const float *sink, void *o,
                                          int B, int Hq, int Hkv, int D, int q_max, int max_ctx,
                                          float scale, attn_dtype_t dtype, void *stream);

/* ------------------------------------------------------------ index dumps ---
 * Integer-exact views of the kernels' own index arithmetic (same device
 * functions), for bit-exact tests against the definitions above.
 *
 * attn_debug_prefill_visits: counts, for every (query i, key j) of one head of
 * a length-T sequence, how many times the prefill kernel's tile schedule and
 * mask admit key j for query i.  visits [T,T] int32 (device).  mode 0 = the
 * GA tiling (window <= 0 for full causal, else window-limited), mode 1 = the
 * packed SWA tiling with G = Hq/Hkv heads per tile.  Correct kernels give 1
 * exactly on visible pairs and 0 elsewhere. */
attn_status_t attn_debug_prefill_visits(int32_t *visits, int mode, int T, int window, int G,
                                        void *stream);

/* attn_debug_swa_stream_visits: the schedule of the streaming SWA prefill
 * kernel (8 query heads per kv head, window in [114, 129]) replayed with
 * `grid` persistent CTAs (0 = the grid the kernel launches): for every
 * (b, kv head g) and query position i, visits[(b*Hkv+g), i, j] counts how many
 * times a CTA's tile admits key j for query i, with the key position taken
 * from the CTA's shared-memory ring of 16-key blocks (which block each ring
 * slot holds).  visits [B*Hkv, T, T+1] int32 (device); column T counts
 * admitted keys outside [0, T).  Correct schedules give 1 exactly on the
 * visible pairs and 0 elsewhere. */
attn_status_t attn_debug_swa_stream_visits(int32_t *visits, int B, int T, int Hkv, int window,
                                           int grid, void *stream);

/* attn_debug_verify_positions: for each request b, query t < q_max and cache
 * slot s, the absolute position the verify kernel assigns to the key it reads
 * there if that key is visible to query t, else -1.
 *   kind 0 (ring):  out [B,q_max,ring_slots], slot = ring slot;
 *   kind 1 (paged): out [B,q_max,max_pages*page_size], slot = page-table
 *                   index * page_size + offset (the physical page read is
 *                   page_table[b, slot / page_size]).
 * cu_q, seq_lens as for verify; page_size is ignored for kind 0. */
attn_status_t attn_debug_verify_positions(int32_t *out, int kind, const int32_t *cu_q,
                                          const int32_t *seq_lens, int B, int q_max, int window,
                                          int ring_slots, int max_pages, int page_size,
                                          void *stream);

/* attn_debug_wait_timeout: enqueues one kernel whose only pipeline wait (an
 * mbarrier phase that nothing completes) runs out after the kernels' wait
 * limit of 2 s and sets ATTN_DEVERR_WAIT_TIMEOUT in the device error word, as
 * a stalled pipeline would.  Pipelined kernels launched while that bit is set
 * (tensor-core prefill, verify) return without doing any work;
 * attn_check_device_error() reports and clears it.
 * For tests of the failure path: no trap, no fault, and the context stays
 * usable.  Errors: ATTN_ERR_CUDA if no device is current or the launch fails. */
attn_status_t attn_debug_wait_timeout(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_SINK_H */

// C ABI of the sink-attention library: argument validation, TMA tensor-map
// encoding and dispatch.  Every call only enqueues work on the caller's
// stream; nothing here allocates device memory.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "attn_sink.h"
#include "index_math.cuh"
#include "internal.h"

#include <cmath>

#define ATTN_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

// Device error word (one per device; kernels get its address as an argument).
__device__ unsigned int g_attn_device_error;

thread_local char g_last_error[512] = "";

attn_status_t fail(attn_status_t st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

attn_status_t ok() {
    g_last_error[0] = '\0';
    return ATTN_OK;
}

attn_status_t cuda_fail(cudaError_t e, const char *what) {
    return fail(ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

// Address of the error word on the current device (looked up once per device).
unsigned int *device_error_word() {
    static unsigned int *addr[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_device_error) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<unsigned int *>(p);
    }
    return addr[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 4-D tiled map, 128-byte swizzle, zero fill out of bounds.  dims innermost
// first; strides (bytes) for dims 1..3; box sizes per dim.
bool make_map_4d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, const uint64_t dims[4],
                 const uint64_t strides[3], const uint32_t box[4]) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gd[4] = {dims[0], dims[1], dims[2], dims[3]};
    cuuint64_t gs[3] = {strides[0], strides[1], strides[2]};
    cuuint32_t bx[4] = {box[0], box[1], box[2], box[3]};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = fn(m, dt, 4, const_cast<void *>(base), gd, gs, bx, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [rows, H, 128] bf16 tensor viewed as (128, H, rows) with a box of (64, bh, bt).
bool map_3d(CUtensorMap *m, const void *base, uint64_t rows, int H, uint32_t bh,
            uint32_t bt = 1) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gd[3] = {128, static_cast<cuuint64_t>(H), rows};
    cuuint64_t gs[2] = {256, static_cast<cuuint64_t>(H) * 256};
    cuuint32_t bx[3] = {64, bh, bt};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), gd, gs, bx, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

// Both prefill entry points, batches of equal length (cu == nullptr, total =
// B*T) and packed batches (cu[B+1] on the device, T = the longest sequence).
attn_status_t prefill_common(const void *q, const void *k, const void *v, const int32_t *cu,
                             const float *sink, void *o, float *lse, int B, int T, long total,
                             int Hq, int Hkv, int D, int window, float scale, float vscale,
                             attn_dtype_t dtype, void *stream, bool swa) {
    if (!q || !k || !v || !sink || !o) return fail(ATTN_ERR_INVALID_ARG, "null pointer argument");
    if (B < 0 || T < 0 || total < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0)
        return fail(ATTN_ERR_INVALID_ARG, "bad sizes B=%d T=%d total=%ld Hq=%d Hkv=%d D=%d", B, T,
                    total, Hq, Hkv, D);
    if (swa && window < 1) return fail(ATTN_ERR_INVALID_ARG, "window must be >= 1 (got %d)", window);
    if (!(scale > 0.f)) return fail(ATTN_ERR_INVALID_ARG, "scale must be > 0");
    if (!std::isfinite(vscale)) return fail(ATTN_ERR_INVALID_ARG, "value_scale must be finite");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return fail(ATTN_ERR_INVALID_ARG, "q/k/v/o must be 16-byte aligned");
    if (total * Hq >= (1ll << 31)) return fail(ATTN_ERR_UNSUPPORTED, "tokens*Hq must be < 2^31");
    unsigned *err = device_error_word();
    if (!err) return fail(ATTN_ERR_CUDA, "no CUDA device / error word unavailable");
    cudaStream_t s = as_stream(stream);
    const int win = swa ? window : 0;
    const attn::PrefillBatch pb{cu, B, T, static_cast<int>(total)};
    if (dtype == ATTN_F32) {
        if (D != 64 && D != 128) return fail(ATTN_ERR_UNSUPPORTED, "fp32 prefill needs D in {64,128}");
        if (B == 0 || total == 0) return ok();
        cudaError_t e = attn::launch_prefill_f32(
            static_cast<const float *>(q), static_cast<const float *>(k),
            static_cast<const float *>(v), sink, static_cast<float *>(o), lse, pb, Hq, Hkv, D, win,
            scale, vscale, err, s);
        return e == cudaSuccess ? ok() : cuda_fail(e, "prefill_f32 launch");
    }
    if (dtype != ATTN_BF16) return fail(ATTN_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (D != 128) return fail(ATTN_ERR_UNSUPPORTED, "bf16 prefill needs D = 128 (got %d)", D);
    if (B == 0 || total == 0 || T == 0) return ok();
    const int G = Hq / Hkv;
    attn::PrefillMaps maps;
    maps.out = o;
    const uint64_t rows = static_cast<uint64_t>(total);
    const bool packed = swa && attn::prefill_swa_tc_supported(G, window);
    bool good;
    if (packed) {  // Q tiles of 16 tokens x 8 heads; K/V in 16-key ring blocks
        const uint32_t TT = static_cast<uint32_t>(attn::kSwaTokens);
        const uint32_t NB = static_cast<uint32_t>(attn::kSwaBlockKeys);
        good = map_3d(&maps.q, q, rows, Hq, G, TT) && map_3d(&maps.k, k, rows, Hkv, 1, NB) &&
               map_3d(&maps.v, v, rows, Hkv, 1, NB);
    } else {
        good = map_3d(&maps.q, q, rows, Hq, 1, 128) && map_3d(&maps.k, k, rows, Hkv, 1, 128) &&
               map_3d(&maps.v, v, rows, Hkv, 1, 128) && map_3d(&maps.o, o, rows, Hq, 1, 128);
    }
    if (!good) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the prefill maps");
    cudaError_t e = packed ? attn::launch_prefill_swa_tc(maps, sink, lse, pb, Hq, Hkv, window,
                                                         scale, vscale, err, s)
                           : attn::launch_prefill_ga_tc(maps, sink, lse, pb, Hq, Hkv, win, scale,
                                                        vscale, err, s);
    return e == cudaSuccess ? ok() : cuda_fail(e, "prefill launch");
}

attn_status_t check_append(const void *k_new, const void *v_new, const int32_t *cu_q,
                           const int32_t *seq_lens, const void *kc, const void *vc, int B, int Hkv,
                           int D, int q_max, attn_dtype_t dtype) {
    if (!k_new || !v_new || !cu_q || !seq_lens || !kc || !vc)
        return fail(ATTN_ERR_INVALID_ARG, "null pointer argument");
    if (B < 0 || Hkv <= 0 || D <= 0 || q_max < 0)
        return fail(ATTN_ERR_INVALID_ARG, "bad sizes B=%d Hkv=%d D=%d q_max=%d", B, Hkv, D, q_max);
    if (dtype != ATTN_BF16 && dtype != ATTN_F32) return fail(ATTN_ERR_INVALID_ARG, "unknown dtype");
    const int eb = dtype == ATTN_BF16 ? 2 : 4;
    if ((D * eb) % 16) return fail(ATTN_ERR_UNSUPPORTED, "D * element size must be a multiple of 16");
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(kc) || !aligned16(vc))
        return fail(ATTN_ERR_INVALID_ARG, "k/v pointers must be 16-byte aligned");
    return ATTN_OK;
}

attn_status_t check_verify(const void *q, const int32_t *cu_q, const int32_t *seq_lens,
                           const float *sink, const void *o, const void *kc, const void *vc, int B,
                           int Hq, int Hkv, int D, int q_max, float scale, attn_dtype_t dtype) {
    if (!q || !cu_q || !seq_lens || !sink || !o || !kc || !vc)
        return fail(ATTN_ERR_INVALID_ARG, "null pointer argument");
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0 || q_max < 1)
        return fail(ATTN_ERR_INVALID_ARG, "bad sizes B=%d Hq=%d Hkv=%d D=%d q_max=%d", B, Hq, Hkv,
                    D, q_max);
    if (!(scale > 0.f)) return fail(ATTN_ERR_INVALID_ARG, "scale must be > 0");
    if (dtype != ATTN_BF16) return fail(ATTN_ERR_UNSUPPORTED, "verify supports bf16 only");
    if (D != 128) return fail(ATTN_ERR_UNSUPPORTED, "verify needs D = 128 (got %d)", D);
    if (q_max * (Hq / Hkv) > attn::kVerifyRows)
        return fail(ATTN_ERR_UNSUPPORTED, "q_max * Hq/Hkv must be <= %d", attn::kVerifyRows);
    if (!aligned16(q) || !aligned16(o) || !aligned16(kc) || !aligned16(vc))
        return fail(ATTN_ERR_INVALID_ARG, "q/o/cache pointers must be 16-byte aligned");
    return ATTN_OK;
}

size_t ws_segment(size_t bytes) { return (bytes + 255) & ~static_cast<size_t>(255); }

}  // namespace

ATTN_EXPORT int attn_version(void) { return 100; }

ATTN_EXPORT const char *attn_last_error(void) { return g_last_error; }

ATTN_EXPORT attn_status_t attn_check_device_error(void *stream, unsigned int *bits_out) {
    cudaError_t e = cudaStreamSynchronize(as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    unsigned int bits = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&bits, g_attn_device_error, sizeof(bits));
    if (e != cudaSuccess) return cuda_fail(e, "read device error word");
    if (bits) {
        e = cudaMemcpyToSymbol(g_attn_device_error, &zero, sizeof(zero));
        if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
    }
    if (bits_out) *bits_out = bits;
    if (bits) return fail(ATTN_ERR_DEVICE_FAULT, "device error bits 0x%x", bits);
    return ok();
}

ATTN_EXPORT attn_status_t attn_swa_sink_prefill(const void *q, const void *k, const void *v,
                                                const float *sink, void *o, float *lse, int B,
                                                int T, int Hq, int Hkv, int D, int window,
                                                float scale, attn_dtype_t dtype, void *stream) {
    return prefill_common(q, k, v, nullptr, sink, o, lse, B, T, static_cast<long>(B) * T, Hq, Hkv,
                          D, window, scale, 1.f, dtype, stream, true);
}

ATTN_EXPORT attn_status_t attn_ga_sink_prefill(const void *q, const void *k, const void *v,
                                               const float *sink, void *o, float *lse, int B, int T,
                                               int Hq, int Hkv, int D, float scale,
                                               attn_dtype_t dtype, void *stream) {
    return prefill_common(q, k, v, nullptr, sink, o, lse, B, T, static_cast<long>(B) * T, Hq, Hkv,
                          D, 0, scale, 1.f, dtype, stream, false);
}

ATTN_EXPORT size_t attn_sink_prefill_backward_workspace(int B, int T, int Hq, int D) {
    if (B <= 0 || T <= 0 || Hq <= 0 || D != 128) return 0;
    return attn::prefill_backward_workspace(B, T, Hq);
}

ATTN_EXPORT attn_status_t attn_sink_prefill_backward(
    const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dout,
    const float *sink, void *dq, void *dk, void *dv, float *dsink, void *workspace,
    size_t workspace_bytes, int B, int T, int Hq, int Hkv, int D, int window, float scale,
    attn_dtype_t dtype, void *stream) {
    if (!q || !k || !v || !o || !lse || !dout || !sink || !dq || !dk || !dv || !dsink)
        return fail(ATTN_ERR_INVALID_ARG, "null pointer argument");
    if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0 || window < 0)
        return fail(ATTN_ERR_INVALID_ARG, "bad sizes B=%d T=%d Hq=%d Hkv=%d D=%d window=%d", B, T,
                    Hq, Hkv, D, window);
    if (!(scale > 0.f)) return fail(ATTN_ERR_INVALID_ARG, "scale must be > 0");
    if (dtype != ATTN_BF16 || D != 128)
        return fail(ATTN_ERR_UNSUPPORTED, "the backward pass supports bf16 with D = 128");
    if (static_cast<long long>(B) * T * Hq >= (1ll << 31))
        return fail(ATTN_ERR_UNSUPPORTED, "B*T*Hq must be < 2^31");
    const void *ptrs[8] = {q, k, v, o, dout, dq, dk, dv};
    for (const void *p : ptrs)
        if (!aligned16(p)) return fail(ATTN_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
    const size_t need = attn_sink_prefill_backward_workspace(B, T, Hq, D);
    if (need > 0 && (!workspace || workspace_bytes < need))
        return fail(ATTN_ERR_INVALID_ARG, "workspace too small: need %zu bytes", need);
    if (need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(ATTN_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    unsigned *err = device_error_word();
    if (!err) return fail(ATTN_ERR_CUDA, "no CUDA device / error word unavailable");
    attn::BwdMaps maps;
    const uint64_t rows = static_cast<uint64_t>(B) * T;
    if (B > 0 && T > 0 &&
        !(map_3d(&maps.q_rows64, q, rows, Hq, 1, 64) && map_3d(&maps.dout_rows64, dout, rows, Hq, 1, 64) &&
          map_3d(&maps.k_rows128, k, rows, Hkv, 1, 128) && map_3d(&maps.v_rows128, v, rows, Hkv, 1, 128) &&
          map_3d(&maps.q_rows128, q, rows, Hq, 1, 128) && map_3d(&maps.dout_rows128, dout, rows, Hq, 1, 128) &&
          map_3d(&maps.k_rows64, k, rows, Hkv, 1, 64) && map_3d(&maps.v_rows64, v, rows, Hkv, 1, 64)))
        return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the backward maps");
    cudaError_t e = attn::launch_prefill_backward(maps, o, lse, dout, sink, dq, dk, dv, dsink,
                                                  workspace, B, T, Hq, Hkv, window, scale, err,
                                                  as_stream(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "backward launch");
}

ATTN_EXPORT attn_status_t attn_swa_sink_prefill_varlen(
    const void *q, const void *k, const void *v, const int32_t *cu_seqlens, const float *sink,
    void *o, float *lse, int B, int total_tokens, int max_seqlen, int Hq, int Hkv, int D,
    int window, float scale, float value_scale, attn_dtype_t dtype, void *stream) {
    if (!cu_seqlens) return fail(ATTN_ERR_INVALID_ARG, "null pointer argument");
    return prefill_common(q, k, v, cu_seqlens, sink, o, lse, B, max_seqlen, total_tokens, Hq, Hkv,
                          D, window, scale, value_scale, dtype, stream, true);
}

ATTN_EXPORT attn_status_t attn_ga_sink_prefill_varlen(
    const void *q, const void *k, const void *v, const int32_t *cu_seqlens, const float *sink,
    void *o, float *lse, int B, int total_tokens, int max_seqlen, int Hq, int Hkv, int D,
    float scale, float value_scale, attn_dtype_t dtype, void *stream) {
    if (!cu_seqlens) return fail(ATTN_ERR_INVALID_ARG, "null pointer argument");
    return prefill_common(q, k, v, cu_seqlens, sink, o, lse, B, max_seqlen, total_tokens, Hq, Hkv,
                          D, 0, scale, value_scale, dtype, stream, false);
}

ATTN_EXPORT attn_status_t attn_swa_ring_append(const void *k_new, const void *v_new,
                                               const int32_t *cu_q, const int32_t *seq_lens,
                                               void *ring_k, void *ring_v, int B, int Hkv, int D,
                                               int ring_slots, int q_max, attn_dtype_t dtype,
                                               void *stream) {
    attn_status_t st = check_append(k_new, v_new, cu_q, seq_lens, ring_k, ring_v, B, Hkv, D, q_max,
                                    dtype);
    if (st != ATTN_OK) return st;
    if (ring_slots < 1) return fail(ATTN_ERR_INVALID_ARG, "ring_slots must be >= 1");
    unsigned *err = device_error_word();
    if (!err) return fail(ATTN_ERR_CUDA, "no CUDA device / error word unavailable");
    cudaError_t e = attn::launch_ring_append(k_new, v_new, cu_q, seq_lens, ring_k, ring_v, B, Hkv,
                                             D, ring_slots, q_max, dtype == ATTN_BF16 ? 2 : 4, err,
                                             as_stream(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "ring append launch");
}

ATTN_EXPORT attn_status_t attn_ga_paged_append(const void *k_new, const void *v_new,
                                               const int32_t *cu_q, const int32_t *seq_lens,
                                               void *k_pages, void *v_pages,
                                               const int32_t *page_table, int max_pages,
                                               int num_pages, int page_size, int B, int Hkv, int D,
                                               int q_max, attn_dtype_t dtype, void *stream) {
    attn_status_t st = check_append(k_new, v_new, cu_q, seq_lens, k_pages, v_pages, B, Hkv, D,
                                    q_max, dtype);
    if (st != ATTN_OK) return st;
    if (!page_table || max_pages < 1 || num_pages < 1 || page_size < 1)
        return fail(ATTN_ERR_INVALID_ARG, "bad page table arguments");
    unsigned *err = device_error_word();
    if (!err) return fail(ATTN_ERR_CUDA, "no CUDA device / error word unavailable");
    cudaError_t e = attn::launch_paged_append(k_new, v_new, cu_q, seq_lens, k_pages, v_pages,
                                              page_table, max_pages, num_pages, page_size, B, Hkv,
                                              D, q_max, dtype == ATTN_BF16 ? 2 : 4, err,
                                              as_stream(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "paged append launch");
}

ATTN_EXPORT attn_status_t attn_ga_paged_append_fp8(
    const void *k_new, const void *v_new, const int32_t *cu_q, const int32_t *seq_lens,
    void *k_pages, void *v_pages, const int32_t *page_table, int max_pages, int num_pages,
    int page_size, const float *k_scale, const float *v_scale, int B, int Hkv, int D, int q_max,
    void *stream) {
    attn_status_t st = check_append(k_new, v_new, cu_q, seq_lens, k_pages, v_pages, B, Hkv, D,
                                    q_max, ATTN_BF16);
    if (st != ATTN_OK) return st;
    if (!k_scale || !v_scale) return fail(ATTN_ERR_INVALID_ARG, "null pointer argument");
    if (D != 128) return fail(ATTN_ERR_UNSUPPORTED, "the 8-bit cache needs D = 128 (got %d)", D);
    if (!page_table || max_pages < 1 || num_pages < 1 || page_size < 1)
        return fail(ATTN_ERR_INVALID_ARG, "bad page table arguments");
    unsigned *err = device_error_word();
    if (!err) return fail(ATTN_ERR_CUDA, "no CUDA device / error word unavailable");
    cudaError_t e = attn::launch_paged_append_fp8(k_new, v_new, cu_q, seq_lens, k_pages, v_pages,
                                                  page_table, max_pages, num_pages, page_size,
                                                  k_scale, v_scale, B, Hkv, q_max, err,
                                                  as_stream(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "fp8 paged append launch");
}

ATTN_EXPORT attn_status_t attn_swa_sink_verify(const void *q, const int32_t *cu_q,
                                               const void *ring_k, const void *ring_v,
                                               const int32_t *seq_lens, const float *sink, void *o,
                                               int B, int Hq, int Hkv, int D, int window,
                                               int ring_slots, int q_max, float scale,
                                               attn_dtype_t dtype, void *stream) {
    attn_status_t st = check_verify(q, cu_q, seq_lens, sink, o, ring_k, ring_v, B, Hq, Hkv, D,
                                    q_max, scale, dtype);
    if (st != ATTN_OK) return st;
    if (window < 1) return fail(ATTN_ERR_INVALID_ARG, "window must be >= 1");
    if (ring_slots < window + q_max - 1)
        return fail(ATTN_ERR_INVALID_ARG, "ring_slots (%d) < window + q_max - 1 (%d)", ring_slots,
                    window + q_max - 1);
    if (B == 0) return ok();
    unsigned *err = device_error_word();
    if (!err) return fail(ATTN_ERR_CUDA, "no CUDA device / error word unavailable");
    attn::VerifyMaps maps;
    const bool tc = attn::verify_ring_tc_supported(Hq / Hkv, ring_slots, q_max) != 0;
    uint64_t dims[4] = {128, static_cast<uint64_t>(ring_slots), static_cast<uint64_t>(Hkv),
                        static_cast<uint64_t>(B)};
    uint64_t strides[3] = {256, static_cast<uint64_t>(ring_slots) * 256,
                           static_cast<uint64_t>(Hkv) * ring_slots * 256};
    // tensor-core kernel: the whole ring in one box; otherwise 64-slot blocks
    uint32_t box[4] = {64, static_cast<uint32_t>(tc ? attn::kVerifyRingKeys : attn::kVerifyBlock), 1,
                       1};
    if (!make_map_4d(&maps.k, ring_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dims, strides, box) ||
        !make_map_4d(&maps.v, ring_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dims, strides, box))
        return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the ring maps");
    // q [cu_q[B], Hq, D] seen as B*q_max rows: an upper bound of cu_q[B] that
    // only bounds the map; the kernel reads the rows of its request and
    // rejects a request whose rows would pass B*q_max
    if (tc && !map_3d(&maps.q, q, static_cast<uint64_t>(B) * q_max, Hq, Hq / Hkv))
        return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the q map");
    cudaError_t e =
        tc ? attn::launch_verify_ring_tc(maps, cu_q, seq_lens, sink, o, B, Hq, Hkv, window,
                                         ring_slots, q_max, scale, err, as_stream(stream))
           : attn::launch_verify_ring(maps, q, cu_q, seq_lens, sink, o, B, Hq, Hkv, window,
                                      ring_slots, q_max, scale, err, as_stream(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "swa verify launch");
}

ATTN_EXPORT size_t attn_ga_sink_verify_workspace(int B, int Hq, int Hkv, int D, int q_max,
                                                 int max_ctx) {
    (void)Hq;
    (void)D;
    (void)q_max;
    if (B <= 0 || Hkv <= 0 || max_ctx <= 0) return 0;
    const int nsplit = attn::verify_num_splits(max_ctx, attn::kVerifyChunkPages * attn::kVerifyBlock);
    if (nsplit <= 1) return 0;
    const size_t units = static_cast<size_t>(B) * Hkv * nsplit;
    return ws_segment(units * attn::kVerifyRows * 128 * sizeof(float)) +
           ws_segment(units * attn::kVerifyRows * 2 * sizeof(float));
}

namespace {
// GA paged verify, bf16 pages (k_scale == nullptr) or E4M3 pages with
// per-kv-head scales.
attn_status_t ga_verify_common(const void *q, const int32_t *cu_q, const void *k_pages,
                               const void *v_pages, const int32_t *page_table, int max_pages,
                               int num_pages, int page_size, const int32_t *seq_lens,
                               const float *sink, void *o, void *workspace,
                               size_t workspace_bytes, int B, int Hq, int Hkv, int D, int q_max,
                               int max_ctx, float scale, attn_dtype_t dtype, const float *k_scale,
                               const float *v_scale, void *stream) {
    attn_status_t st = check_verify(q, cu_q, seq_lens, sink, o, k_pages, v_pages, B, Hq, Hkv, D,
                                    q_max, scale, dtype);
    if (st != ATTN_OK) return st;
    if (!page_table || max_pages < 1 || num_pages < 1)
        return fail(ATTN_ERR_INVALID_ARG, "bad page table arguments");
    if (page_size != attn::kVerifyBlock)
        return fail(ATTN_ERR_UNSUPPORTED, "page_size must be %d", attn::kVerifyBlock);
    if (max_ctx < 1) return fail(ATTN_ERR_INVALID_ARG, "max_ctx must be >= 1");
    const size_t need = attn_ga_sink_verify_workspace(B, Hq, Hkv, D, q_max, max_ctx);
    if (need > 0 && (!workspace || workspace_bytes < need))
        return fail(ATTN_ERR_INVALID_ARG, "workspace too small: need %zu bytes", need);
    if (need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(ATTN_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (B == 0) return ok();
    unsigned *err = device_error_word();
    if (!err) return fail(ATTN_ERR_CUDA, "no CUDA device / error word unavailable");
    attn::VerifyMaps maps;
    const bool fp8 = k_scale != nullptr;
    const uint64_t row = fp8 ? 128 : 256;  // bytes per cached token of one kv head
    uint64_t dims[4] = {128, static_cast<uint64_t>(page_size), static_cast<uint64_t>(Hkv),
                        static_cast<uint64_t>(num_pages)};
    uint64_t strides[3] = {row, static_cast<uint64_t>(page_size) * row,
                           static_cast<uint64_t>(Hkv) * page_size * row};
    uint32_t box[4] = {fp8 ? 128u : 64u, static_cast<uint32_t>(attn::kVerifyBlock), 1, 1};
    const CUtensorMapDataType dt =
        fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!make_map_4d(&maps.k, k_pages, dt, dims, strides, box) ||
        !make_map_4d(&maps.v, v_pages, dt, dims, strides, box))
        return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the page maps");
    const int nsplit =
        attn::verify_num_splits(max_ctx, attn::kVerifyChunkPages * attn::kVerifyBlock);
    float *ws_o = nullptr, *ws_ml = nullptr;
    if (nsplit > 1) {
        const size_t units = static_cast<size_t>(B) * Hkv * nsplit;
        ws_o = static_cast<float *>(workspace);
        ws_ml = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                          ws_segment(units * attn::kVerifyRows * 128 * sizeof(float)));
    }
    cudaError_t e = attn::launch_verify_paged(maps, q, cu_q, seq_lens, page_table, max_pages,
                                              num_pages, sink, o, ws_o, ws_ml, nsplit, B, Hq, Hkv,
                                              q_max, max_ctx, scale, k_scale, v_scale, err,
                                              as_stream(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "ga verify launch");
}
}  // namespace

ATTN_EXPORT attn_status_t attn_ga_sink_verify(const void *q, const int32_t *cu_q,
                                              const void *k_pages, const void *v_pages,
                                              const int32_t *page_table, int max_pages,
                                              int num_pages, int page_size,
                                              const int32_t *seq_lens, const float *sink, void *o,
                                              void *workspace, size_t workspace_bytes, int B,
                                              int Hq, int Hkv, int D, int q_max, int max_ctx,
                                              float scale, attn_dtype_t dtype, void *stream) {
    return ga_verify_common(q, cu_q, k_pages, v_pages, page_table, max_pages, num_pages,
                            page_size, seq_lens, sink, o, workspace, workspace_bytes, B, Hq, Hkv,
                            D, q_max, max_ctx, scale, dtype, nullptr, nullptr, stream);
}

ATTN_EXPORT attn_status_t attn_ga_sink_verify_fp8(
    const void *q, const int32_t *cu_q, const void *k_pages, const void *v_pages,
    const int32_t *page_table, int max_pages, int num_pages, int page_size,
    const int32_t *seq_lens, const float *sink, const float *k_scale, const float *v_scale,
    void *o, void *workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int D, int q_max,
    int max_ctx, float scale, void *stream) {
    if (!k_scale || !v_scale) return fail(ATTN_ERR_INVALID_ARG, "null pointer argument");
    return ga_verify_common(q, cu_q, k_pages, v_pages, page_table, max_pages, num_pages,
                            page_size, seq_lens, sink, o, workspace, workspace_bytes, B, Hq, Hkv,
                            D, q_max, max_ctx, scale, ATTN_BF16, k_scale, v_scale, stream);
}

// ---------------------------------------------- GA verify without allocation
// Some callers cannot call cudaMalloc at all: code that runs inside a host
// program which reserved all device memory up front in its own pool and
// forbids later allocations, or a latency-critical decode loop that must
// never risk the implicit device synchronisation and latency of an
// allocation.  attn_ga_sink_verify_noalloc serves them: its split-KV partials
// live in this file-scope device array instead of a caller workspace.  Every
// GPU that loads the library holds the array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
static __device__ __align__(256) unsigned char g_verify_scratch[kNoAllocScratchBytes];

namespace {
// Device address of g_verify_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device with cudaGetSymbolAddress (with that device current) and cached.
void *noalloc_scratch() {
    static void *addr[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress((void **)&ptr, g_verify_scratch) != cudaSuccess) return nullptr;
        addr[dev] = ptr;
    }
    return addr[dev];
}
}  // namespace

ATTN_EXPORT attn_status_t attn_ga_sink_verify_noalloc(
    const void *q, const int32_t *cu_q, const void *k_pages, const void *v_pages,
    const int32_t *page_table, int max_pages, int num_pages, int page_size,
    const int32_t *seq_lens, const float *sink, void *o, int B, int Hq, int Hkv, int D, int q_max,
    int max_ctx, float scale, attn_dtype_t dtype, void *stream) {
    const size_t need = attn_ga_sink_verify_workspace(B, Hq, Hkv, D, q_max, max_ctx);
    if (need > kNoAllocScratchBytes)
        return fail(ATTN_ERR_UNSUPPORTED,
                    "split-KV scratch of %zu bytes exceeds the %zu-byte static scratch of "
                    "attn_ga_sink_verify_noalloc (lower B or max_ctx, or pass a workspace to "
                    "attn_ga_sink_verify)",
                    need, kNoAllocScratchBytes);
    void *scratch = nullptr;
    if (need > 0) {
        scratch = noalloc_scratch();
        if (!scratch)
            return fail(ATTN_ERR_CUDA, "cudaGetSymbolAddress of the static verify scratch failed");
    }
    return attn_ga_sink_verify(q, cu_q, k_pages, v_pages, page_table, max_pages, num_pages,
                               page_size, seq_lens, sink, o, scratch,
                               need > 0 ? kNoAllocScratchBytes : 0, B, Hq, Hkv, D, q_max, max_ctx,
                               scale, dtype, stream);
}

ATTN_EXPORT attn_status_t attn_debug_prefill_visits(int32_t *visits, int mode, int T, int window,
                                                    int G, void *stream) {
    if (!visits || T < 0 || (mode != 0 && mode != 1))
        return fail(ATTN_ERR_INVALID_ARG, "bad arguments");
    if (mode == 1 && (G < 1 || 128 % G != 0 || window < 1 ||
                      attn::swa_pack_keys(G, window) > 256))
        return fail(ATTN_ERR_UNSUPPORTED, "packed SWA tiling needs 128 % G == 0 and a window that fits");
    cudaError_t e = attn::launch_debug_prefill_visits(visits, mode, T, window, G, as_stream(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "debug prefill visits");
}

ATTN_EXPORT attn_status_t attn_debug_swa_stream_visits(int32_t *visits, int B, int T, int Hkv,
                                                       int window, int grid, void *stream) {
    if (!visits || B < 0 || T < 0 || Hkv < 1 || grid < 0)
        return fail(ATTN_ERR_INVALID_ARG, "bad arguments");
    if (!attn::prefill_swa_tc_supported(attn::kSwaHeads, window))
        return fail(ATTN_ERR_UNSUPPORTED, "the streaming SWA kernel needs a window in [114, 129]");
    if (grid == 0 && B > 0 && T > 0)
        grid = attn::prefill_swa_grid(static_cast<long>(B) * Hkv * attn::swa_seq_blocks(T));
    cudaError_t e = attn::launch_debug_swa_stream_visits(visits, B, T, Hkv, window, grid,
                                                         as_stream(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "debug swa stream visits");
}

ATTN_EXPORT attn_status_t attn_debug_verify_positions(int32_t *out, int kind, const int32_t *cu_q,
                                                      const int32_t *seq_lens, int B, int q_max,
                                                      int window, int ring_slots, int max_pages,
                                                      int page_size, void *stream) {
    if (!out || !cu_q || !seq_lens || B < 0 || q_max < 1 || (kind != 0 && kind != 1))
        return fail(ATTN_ERR_INVALID_ARG, "bad arguments");
    if (kind == 0 && ring_slots < 1) return fail(ATTN_ERR_INVALID_ARG, "ring_slots must be >= 1");
    if (kind == 1 && (max_pages < 1 || page_size < 1))
        return fail(ATTN_ERR_INVALID_ARG, "bad page arguments");
    cudaError_t e = attn::launch_debug_verify_positions(out, kind, cu_q, seq_lens, B, q_max, window,
                                                        ring_slots, max_pages, page_size,
                                                        as_stream(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "debug verify positions");
}

namespace attn {
cudaError_t launch_debug_wait_timeout(unsigned *err, cudaStream_t s);  // debug_index.cu
}

ATTN_EXPORT attn_status_t attn_debug_wait_timeout(void *stream) {
    unsigned *err = device_error_word();
    if (!err) return fail(ATTN_ERR_CUDA, "no CUDA device / error word unavailable");
    cudaError_t e = attn::launch_debug_wait_timeout(err, as_stream(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "debug wait timeout");
}

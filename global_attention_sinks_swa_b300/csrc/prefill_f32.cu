// fp32 sink-attention prefill on CUDA cores (FFMA, no TF32): the fp32-I/O path
// of attn_{swa,ga}_sink_prefill{,_varlen}.  One warp computes one output row
// with an online softmax whose running max starts at the sink logit and whose
// running sum starts at the sink's own term (technical-report summary,
// section "Hybrid Sliding Window Attention Architecture": learnable sink bias;
// the sink adds to the denominator only).  Keys are the causal window
// (section "MiMo-V2-Flash Model Architecture": W = 128) or the full prefix.
#include "attn_sink.h"
#include "index_math.cuh"
#include "internal.h"
#include "ptx_sm103.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kWarpsPerBlock = 8;

template <int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    prefill_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                       const float *__restrict__ v, const float *__restrict__ sink,
                       float *__restrict__ o, float *__restrict__ lse,
                       const int32_t *__restrict__ cu, int B, int T, int total, int Hq, int Hkv,
                       int window, float scale, float vscale, unsigned *err) {
    constexpr int E = D / 32;  // elements per lane
    const int lane = threadIdx.x & 31;
    const long row = static_cast<long>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
    const long nrows = static_cast<long>(total) * Hq;
    if (row >= nrows) return;
    // rows are ordered (h, token) so that the warps of a block share keys
    const int tok = static_cast<int>(row % total);
    const int h = static_cast<int>(row / total);
    int b;
    if (!cu) {
        b = tok / T;
    } else {  // the last sequence starting at or before tok
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (cu[mid] <= tok) lo = mid;
            else hi = mid - 1;
        }
        b = lo;
    }
    const SeqSpan span = seq_span(cu, b, T, total);
    if (!span.ok) {
        if (lane == 0 && h == 0) atomicOr(err, ATTN_DEVERR_SEQLENS);
        return;
    }
    const int i = tok - span.start;
    if (i < 0 || i >= span.len) return;  // a token outside every valid sequence
    const int g = h / (Hq / Hkv);

    const float *qrow = q + (static_cast<long>(tok) * Hq + h) * D;
    float qv[E], acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        qv[e] = qrow[lane + 32 * e] * (scale * kLog2e);  // scores in log2 units
        acc[e] = 0.f;
    }
    float *orow = o + (static_cast<long>(tok) * Hq + h) * D;
    const float sig = sink[h];
    if (isinf(sig) && sig > 0.f) {  // the sink takes all the probability mass
#pragma unroll
        for (int e = 0; e < E; ++e) orow[lane + 32 * e] = 0.f;
        if (lse && lane == 0) lse[lse_index(cu, b, h, i, span.start, T, total, Hq)] = INFINITY;
        return;
    }
    float m = sig * kLog2e;                   // running max (log2 units)
    float l = isinf(sig) ? 0.f : 1.f;         // running sum, seeded with e^(sigma - m)
    int lo = 0;
    if (window > 0) lo = max(0, i - window + 1);
    const long kstride = static_cast<long>(Hkv) * D;
    const float *kb = k + (static_cast<long>(span.start) * Hkv + g) * D;
    const float *vb = v + (static_cast<long>(span.start) * Hkv + g) * D;
    for (int j = lo; j <= i; ++j) {
        if (!key_visible(i, j, window)) continue;
        const float *kr = kb + j * kstride;
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) s = fmaf(qv[e], kr[lane + 32 * e], s);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        const float mn = fmaxf(m, s);
        const float alpha = ptx::exp2_approx(m - mn);   // 0 when m = -inf
        const float p = ptx::exp2_approx(s - mn);
        l = fmaf(l, alpha, p);
        const float *vr = vb + j * kstride;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(acc[e], alpha, p * vr[lane + 32 * e]);
        m = mn;
    }
    const float inv = vscale / l;  // the value scale rides on 1/l
#pragma unroll
    for (int e = 0; e < E; ++e) orow[lane + 32 * e] = acc[e] * inv;
    if (lse && lane == 0)
        lse[lse_index(cu, b, h, i, span.start, T, total, Hq)] = (m + log2f(l)) * 0.6931471805599453f;
}

}  // namespace

cudaError_t launch_prefill_f32(const float *q, const float *k, const float *v, const float *sink,
                               float *o, float *lse, const PrefillBatch &pb, int Hq, int Hkv,
                               int D, int window, float scale, float vscale, unsigned int *err,
                               cudaStream_t s) {
    if (pb.B == 0) return cudaSuccess;
    const long nrows = static_cast<long>(pb.total) * Hq;
    if (nrows == 0) return cudaSuccess;
    dim3 grid(static_cast<unsigned>((nrows + kWarpsPerBlock - 1) / kWarpsPerBlock));
    dim3 block(kWarpsPerBlock * 32);
    if (D == 64)
        prefill_f32_kernel<64><<<grid, block, 0, s>>>(q, k, v, sink, o, lse, pb.cu, pb.B, pb.T,
                                                     pb.total, Hq, Hkv, window, scale, vscale, err);
    else
        prefill_f32_kernel<128><<<grid, block, 0, s>>>(q, k, v, sink, o, lse, pb.cu, pb.B, pb.T,
                                                      pb.total, Hq, Hkv, window, scale, vscale, err);
    return cudaGetLastError();
}

}  // namespace attn

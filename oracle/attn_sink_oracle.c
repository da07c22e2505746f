/*
 * Sink-attention oracle: plain, slow, fp64 CPU reference.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only tests, the smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no code with the CUDA library.
 *
 * What it computes (the plain definition, no blocking, no online softmax):
 *
 *   For batch b, query head h (key/value head g = h / (Hq/Hkv)) and query
 *   position i, the visible key positions are
 *       V_i = { j : 0 <= j <= i  and (global  or  j >= i - W + 1) }
 *   (a causal sliding window of W keys including the query itself, or the
 *   full causal prefix for a global-attention layer).  With
 *       S_j = scale * <q[b,i,h,:], k[b,j,g,:]>            (fp64)
 *       m   = max(sigma_h, max_{j in V_i} S_j)
 *       Z   = exp(sigma_h - m) + sum_{j in V_i} exp(S_j - m)
 *   the output row is
 *       o[b,i,h,:] = sum_{j in V_i} exp(S_j - m) / Z * v[b,j,g,:]
 *   the sink probability is p_sink = exp(sigma_h - m) / Z and the row's
 *   log-sum-exp is lse = m + log Z.  The sink logit sigma_h joins the
 *   softmax denominator only and carries no value.
 *   Special cases: sigma_h = +inf gives o = 0, p_sink = 1, lse = +inf;
 *   sigma_h = -inf drops the sink term (plain softmax attention).
 *
 * Sources:
 *   - window W = 128 and the 5:1 interleave of sliding-window and global
 *     layers: MiMo-V2-Flash technical-report summary (fanfer.top, "MiMo-V2"),
 *     section "MiMo-V2-Flash Model Architecture"; release announcement
 *     (aihot.news, "小米开源 MiMo-V2-Flash"), section "将效率推向极限".
 *   - the learnable per-head attention-sink bias "in the gpt-oss style": same
 *     summary, section "Hybrid Sliding Window Attention Architecture".  The
 *     formula after that sentence was lost from the page; the reading used here
 *     is that the sink logit is one extra softmax column per query head with
 *     no value vector, compared unscaled with the scaled scores.
 *   - MTP verify (1 real + up to 3 draft tokens scored in one pass, each draft
 *     seeing the earlier ones): release announcement, figure
 *     "Multi-Token Prediction" (验证 / 接受 / 拒绝 / 放弃).
 *
 * Inputs are fp32 arrays (bf16 tensors widen to fp32 exactly); all arithmetic
 * is fp64.  Layouts are row-major:
 *   prefill  q, o [B,T,Hq,D];  k, v [B,T,Hkv,D];  sink [Hq];  lse, psink [B,Hq,T]
 *   verify   q, o [sum_q,Hq,D] (request b owns rows cu_q[b]..cu_q[b+1]-1);
 *            k_hist, v_hist [B,Lmax,Hkv,D] hold each request's keys/values by
 *            absolute position; seq_lens[b] counts positions incl. the new ones.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC attn_sink_oracle.c -o liboracle.so -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

/* One output row by the plain definition.  kv rows for positions lo..hi are at
 * kbase + j*kstride and vbase + j*vstride.  `scores` has room for hi-lo+1. */
static void sink_softmax_row(const float *qv, const float *kbase, const float *vbase,
                             long kstride, long vstride, int lo, int hi,
                             double sigma, double scale, int D, double *scores,
                             double *out, double *lse, double *psink)
{
    int n = hi - lo + 1;
    if (n < 0) n = 0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (isinf(sigma) && sigma > 0) {            /* the sink takes all the mass */
        if (lse) *lse = INFINITY;
        if (psink) *psink = 1.0;
        return;
    }
    double m = sigma;                            /* -inf when there is no sink */
    for (int t = 0; t < n; ++t) {
        const float *kv = kbase + (long)(lo + t) * kstride;
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += (double)qv[d] * (double)kv[d];
        s *= scale;
        scores[t] = s;
        if (s > m) m = s;
    }
    double zsink = isinf(sigma) ? 0.0 : exp(sigma - m);
    double z = zsink;
    for (int t = 0; t < n; ++t) z += exp(scores[t] - m);
    for (int t = 0; t < n; ++t) {
        double w = exp(scores[t] - m) / z;
        const float *vv = vbase + (long)(lo + t) * vstride;
        for (int d = 0; d < D; ++d) out[d] += w * (double)vv[d];
    }
    if (lse) *lse = m + log(z);
    if (psink) *psink = zsink / z;
}

/* Visible key range [lo, hi] of query position i (see header). */
static void visible_range(int i, int window, int *lo, int *hi)
{
    *hi = i;
    *lo = (window > 0 && i - window + 1 > 0) ? i - window + 1 : 0;
}

/* Prefill over whole sequences.  window <= 0 selects global (full causal)
 * attention.  lse / psink may be NULL.  Returns 0, or -1 on bad sizes. */
int oracle_prefill(const float *q, const float *k, const float *v, const float *sink,
                   double *o, double *lse, double *psink,
                   int B, int T, int Hq, int Hkv, int D, int window, double scale)
{
    if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv) return -1;
    const int G = Hq / Hkv;
    const long nrows = (long)B * T * Hq;
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
#pragma omp for schedule(dynamic, 64)
        for (long r = 0; r < nrows; ++r) {
            int h = (int)(r % Hq);
            int i = (int)((r / Hq) % T);
            int b = (int)(r / ((long)Hq * T));
            int g = h / G;
            int lo, hi;
            visible_range(i, window, &lo, &hi);
            const float *qv = q + (((long)b * T + i) * Hq + h) * D;
            const float *kb = k + ((long)b * T * Hkv + g) * D;
            const float *vb = v + ((long)b * T * Hkv + g) * D;
            long st = (long)Hkv * D;
            long lidx = ((long)b * Hq + h) * T + i;
            sink_softmax_row(qv, kb, vb, st, st, lo, hi, (double)sink[h], scale, D, scores,
                             o + r * D, lse ? lse + lidx : NULL, psink ? psink + lidx : NULL);
        }
        free(scores);
    }
    return 0;
}

/* Prefill restricted to chosen rows: rows[3*n+0..2] = (b, i, h).  Output row n
 * goes to o[n*D..], lse[n], psink[n].  Used where the full problem is too large
 * for the CPU (the rows are computed exactly as oracle_prefill would). */
int oracle_prefill_rows(const float *q, const float *k, const float *v, const float *sink,
                        const int32_t *rows, long nsel, double *o, double *lse, double *psink,
                        int B, int T, int Hq, int Hkv, int D, int window, double scale)
{
    if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv) return -1;
    for (long n = 0; n < nsel; ++n) {
        int b = rows[3 * n], i = rows[3 * n + 1], h = rows[3 * n + 2];
        if (b < 0 || b >= B || i < 0 || i >= T || h < 0 || h >= Hq) return -1;
    }
    const int G = Hq / Hkv;
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
#pragma omp for schedule(dynamic, 1)
        for (long n = 0; n < nsel; ++n) {
            int b = rows[3 * n], i = rows[3 * n + 1], h = rows[3 * n + 2];
            int g = h / G, lo, hi;
            visible_range(i, window, &lo, &hi);
            const float *qv = q + (((long)b * T + i) * Hq + h) * D;
            const float *kb = k + ((long)b * T * Hkv + g) * D;
            const float *vb = v + ((long)b * T * Hkv + g) * D;
            long st = (long)Hkv * D;
            sink_softmax_row(qv, kb, vb, st, st, lo, hi, (double)sink[h], scale, D, scores,
                             o + n * D, lse ? lse + n : NULL, psink ? psink + n : NULL);
        }
        free(scores);
    }
    return 0;
}

/* MTP verify: request b has q_len = cu_q[b+1]-cu_q[b] new query tokens at
 * positions seq_lens[b]-q_len .. seq_lens[b]-1; query t sees the history up to
 * and including its own position (earlier drafts included), restricted to the
 * window for SWA.  Keys/values are read by absolute position from the linear
 * history; the oracle never sees a ring buffer or a page table.
 * lse / psink are [sum_q, Hq] or NULL. */
int oracle_verify(const float *q, const int32_t *cu_q, const float *k_hist, const float *v_hist,
                  int Lmax, const int32_t *seq_lens, const float *sink,
                  double *o, double *lse, double *psink,
                  int B, int Hq, int Hkv, int D, int window, double scale)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv) return -1;
    for (int b = 0; b < B; ++b) {
        int ql = cu_q[b + 1] - cu_q[b];
        if (ql < 0 || seq_lens[b] < ql || seq_lens[b] > Lmax) return -1;
    }
    const int G = Hq / Hkv;
    const long nq = cu_q[B];
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)(Lmax > 0 ? Lmax : 1));
#pragma omp for schedule(dynamic, 1)
        for (long r = 0; r < nq * Hq; ++r) {
            long row = r / Hq;
            int h = (int)(r % Hq);
            int b = 0;
            while (cu_q[b + 1] <= row) ++b;
            int ql = cu_q[b + 1] - cu_q[b];
            int t = (int)(row - cu_q[b]);
            int i = seq_lens[b] - ql + t;                 /* absolute query position */
            int g = h / G, lo, hi;
            visible_range(i, window, &lo, &hi);
            const float *qv = q + (row * Hq + h) * D;
            const float *kb = k_hist + ((long)b * Lmax * Hkv + g) * D;
            const float *vb = v_hist + ((long)b * Lmax * Hkv + g) * D;
            long st = (long)Hkv * D;
            sink_softmax_row(qv, kb, vb, st, st, lo, hi, (double)sink[h], scale, D, scores,
                             o + r * D, lse ? lse + r : NULL, psink ? psink + r : NULL);
        }
        free(scores);
    }
    return 0;
}

// MTP verify attention with sinks (bf16 in/out, fp32 accumulation, D = 128).
//
// The step: the main model scores the real token and up to three MTP drafts of
// every request in one pass, each draft seeing the earlier ones (release
// announcement "小米开源 MiMo-V2-Flash", figure "Multi-Token Prediction";
// technical-report summary, section "MTP加速").  Decoding is bound by reading
// the KV cache; scoring q_len tokens per read raises attention's arithmetic
// intensity without more cache traffic.  The kernel exploits exactly that: one
// CTA reads each (request, kv head) cache block once and scores all
// q_len x G query rows of that kv head against it (GQA packing, G = Hq/Hkv).
//
// Shapes: rows r = t*G + hh (t = draft index, hh = head within the kv group),
// at most 32 rows = two m16 tiles; keys stream in blocks of 64 (one GA page,
// or a third of the 131-slot SWA ring) through a 3-stage TMA ring of
// 128-byte-swizzled shared-memory tiles.  Warp roles: warp 4 issues the TMA
// loads; warps 0-3 compute, warp w owning rows [16(w&1), +16) and keys
// [32(w>>1), +32) of every block, with mma.sync m16n8k16 for S = QK^T and
// O += PV and an online softmax in registers (its running max raised only
// when a block exceeds it by more than 2^8).  The two key halves merge in
// shared memory; the sink logit joins the denominator once, in the final
// merge (in-kernel for the ring, in the split combine for the paged cache).
//
// 8-bit paged cache (FP8 = true): pages hold E4M3 codes, entry = code * the
// kv head's scale (K and V each have one), which halves the bytes read per
// token.  TMA brings 8 KB code blocks into a deeper ring (the same bytes in
// flight as the bf16 ring), and the codes go from shared memory straight into
// f16 mma.sync fragments (cvt.f16x2.e4m3x2 is exact), with Q rounded to f16
// and P in f16:
//   K: ldmatrix of 16-byte code rows gives a thread 4 consecutive d of one
//      key; fragment k positions {2c,2c+1 | 2c+8,2c+9} are taken to mean d
//      {4c,4c+1 | 4c+2,4c+3} of the 16-d chunk, and Q is loaded with the
//      same order (the sum over d does not care);
//   V: ldmatrix.trans gives two keys x two adjacent d; byte permutes split
//      them into an "even d" and an "odd d" fragment, so O tile 2j holds
//      d = 16j + 2n and tile 2j+1 holds d = 16j + 2n + 1: a thread's four
//      accumulators of a row are four consecutive d.
// The K scale folds into the score scale, the V scale into the output.
#include "index_math.cuh"
#include "internal.h"
#include "ptx_sm103.cuh"

namespace attn {
namespace {

constexpr int kD = 128;
constexpr int kStages = 3;
constexpr int kConsumers = 4;                 // compute warps
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kHalfBytes = kVerifyBlock * 128;  // 64 rows x 128 B (64 bf16)
constexpr int kStageBytes = 4 * kHalfBytes;      // K and V, two D halves each
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale threshold (log2 units)
constexpr unsigned kErrPage = 0x1u, kErrCtx = 0x2u, kErrQlen = 0x4u, kErrWait = 0x8u;
constexpr int kMergeStride = kD + 8;     // floats per row of the key-half merge buffer
constexpr int kStageRowBytes = 2 * kD + 16;  // bytes per row of the bf16 output staging

constexpr int kBlock8Bytes = kVerifyBlock * kD;  // one 8-bit block: 64 rows x 128 codes
template <bool FP8>
constexpr int kStagesOf = FP8 ? 2 * kStages : kStages;  // the same bytes in flight

template <bool FP8>
struct __align__(1024) VerifySmem {
    uint8_t k[kStages][2][kHalfBytes];  // after the loop: the key-half merge buffer
    uint8_t v[kStages][2][kHalfBytes];  // after the loop: the bf16 output staging
    uint8_t q[2][kVerifyRows * 128];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    float merge_ml[2][16][2];
    int abort;
    __device__ uint8_t *kt(int st, int hf) { return k[st][hf]; }  // 16-bit tiles computed on
    __device__ uint8_t *vt(int st, int hf) { return v[st][hf]; }
    __device__ float *merge() { return reinterpret_cast<float *>(k[0][0]); }
    __device__ uint8_t *ostage() { return v[0][0]; }
};
template <>
struct __align__(1024) VerifySmem<true> {
    uint8_t k8[kStagesOf<true>][kBlock8Bytes];  // E4M3 code ring; after the loop: merge buffer
    uint8_t v8[kStagesOf<true>][kBlock8Bytes];  // after the loop: the bf16 output staging
    uint8_t q[2][kVerifyRows * 128];             // Q in f16
    uint64_t full[kStagesOf<true>];
    uint64_t empty[kStagesOf<true>];
    float merge_ml[2][16][2];
    int abort;
    __device__ float *merge() { return reinterpret_cast<float *>(k8[0]); }
    __device__ uint8_t *ostage() { return v8[0]; }
};

static_assert(2 * 16 * kMergeStride * sizeof(float) <= sizeof(VerifySmem<false>::k), "merge buffer");
static_assert(kVerifyRows * kStageRowBytes <= sizeof(VerifySmem<false>::v), "output staging");
static_assert(2 * 16 * kMergeStride * sizeof(float) <= sizeof(VerifySmem<true>::k8), "merge buffer");
static_assert(kVerifyRows * kStageRowBytes <= sizeof(VerifySmem<true>::v8), "output staging");

// Byte offset of element (row, d) inside a 128B-swizzled [rows][64] half tile;
// d a multiple of 8.
__device__ __forceinline__ uint32_t sw128(int row, int d) {
    return static_cast<uint32_t>(row * 128 + ((((d >> 3) ^ row) & 7) << 4));
}

struct KeySource {
    // ring: blocks cover slots [64*blk, 64*blk+64) of the R-slot ring
    // paged: block = one page of page_table[b][pb + blk]
    int kind;        // 0 ring, 1 paged
    int L, R, r0;    // sequence length, ring slots, L mod R
    int pb;          // first page-table index of this split (paged)
    __device__ __forceinline__ int position(int blk, int c) const {
        if (kind == 0) {
            const int s = blk * kVerifyBlock + c;
            return s < R ? ring_slot_position_r0(s, L, R, r0) : -1;
        }
        return (pb + blk) * kVerifyBlock + c;
    }
};

// Output accumulators as 16 pairs (x, y) = O[row][d], O[row][d+1] per row half
// h2 of a thread: bf16 path, tile i holds d = 8i + 2c, +1; 8-bit path, tiles
// 2j / 2j+1 hold the even / odd d of chunk j, pair i = (j, e) is d = 16j+4c+2e.
template <bool FP8>
__device__ __forceinline__ float &acc_x(float (&o)[16][4], int i, int h2) {
    if constexpr (FP8) return o[2 * (i >> 1)][2 * h2 + (i & 1)];
    else return o[i][2 * h2];
}
template <bool FP8>
__device__ __forceinline__ float &acc_y(float (&o)[16][4], int i, int h2) {
    if constexpr (FP8) return o[2 * (i >> 1) + 1][2 * h2 + (i & 1)];
    else return o[i][2 * h2 + 1];
}
template <bool FP8>
__device__ __forceinline__ int acc_d(int i, int c) {
    if constexpr (FP8) return 16 * (i >> 1) + 4 * c + 2 * (i & 1);
    else return 8 * i + 2 * c;
}

template <bool FP8>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    if constexpr (FP8) ptx::mma_f16_16816(c, a, b0, b1);
    else ptx::mma_bf16_16816(c, a, b0, b1);
}
template <bool FP8>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
    if constexpr (FP8) return ptx::pack_f16x2(lo, hi);
    else return ptx::pack_bf16x2(lo, hi);
}

// Row-wise merge of two online-softmax states (log2 units): (m,l,o) <- (m,l,o) + (mb,lb,ob).
__device__ __forceinline__ float merge_scale(float m, float mb, float *sa, float *sb) {
    const float mm = fmaxf(m, mb);
    const float base = (mm == -INFINITY) ? 0.f : mm;
    *sa = ptx::exp2_approx(m - base);
    *sb = ptx::exp2_approx(mb - base);
    return mm;
}

template <bool FP8>
__global__ void __launch_bounds__(kThreads, 2)
    verify_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const __nv_bfloat16 *__restrict__ q, const int32_t *__restrict__ cu_q,
                  const int32_t *__restrict__ seq_lens, const int32_t *__restrict__ page_table,
                  int max_pages, int num_pages, const float *__restrict__ sink,
                  __nv_bfloat16 *__restrict__ o, float *__restrict__ ws_o,
                  float *__restrict__ ws_ml, int nsplit, int kind, int Hq, int Hkv, int window,
                  int R, int q_max, int max_ctx, float scale, int finalize,
                  const float *__restrict__ k_scale, const float *__restrict__ v_scale,
                  unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    VerifySmem<FP8> &sm = *reinterpret_cast<VerifySmem<FP8> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int G = Hq / Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = cu_q[b], q_len = cu_q[b + 1] - r0, L = seq_lens[b];

    // ---- validate the request (uniform across the CTA)
    if (q_len <= 0) return;
    if (q_len > q_max || q_len * G > kVerifyRows) {
        if (threadIdx.x == 0 && split == 0 && g == 0) atomicOr(err, kErrQlen);
        return;
    }
    KeySource src{kind, L, R, kind == 0 && R > 0 ? L % R : 0, 0};
    int nblk;
    if (kind == 0) {
        if (L < q_len) {
            if (threadIdx.x == 0 && g == 0) atomicOr(err, kErrCtx);
            return;
        }
        nblk = (R + kVerifyBlock - 1) / kVerifyBlock;
    } else {
        if (L < q_len || L > max_ctx || (L + kVerifyBlock - 1) / kVerifyBlock > max_pages) {
            if (threadIdx.x == 0 && split == 0 && g == 0) atomicOr(err, kErrCtx);
            return;
        }
        int pb, pe;
        verify_split_pages(split, L, kVerifyBlock, kVerifyChunkPages, &pb, &pe);
        if (pb >= pe) return;  // this split lies beyond the request's context
        src.pb = pb;
        nblk = pe - pb;
    }

    constexpr int kS = kStagesOf<FP8>;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kS; ++s) {
            ptx::mbar_init(&sm.full[s], 1);
            ptx::mbar_init(&sm.empty[s], kConsumers);
        }
        sm.abort = ptx::prior_timeout(err) ? 1 : 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (sm.abort) return;  // an earlier launch timed out: do nothing

    if (warp == kConsumers) {
        // ------------------------------------------------ producer warp (TMA)
        if (lane == 0) {
            ptx::prefetch_tmap(&tmk);
            ptx::prefetch_tmap(&tmv);
        }
        const int32_t *pt = page_table + static_cast<long>(b) * max_pages;
        for (int base = 0; base < nblk; base += 32) {
            int my_page = 0;
            if (kind == 1 && base + lane < nblk) {
                my_page = pt[src.pb + base + lane];
                if (my_page < 0 || my_page >= num_pages) {
                    atomicOr(err, kErrPage);
                    my_page = 0;  // read a valid page; the request's result is void
                }
            }
            const int n = min(32, nblk - base);
            for (int j = 0; j < n; ++j) {
                const int blk = base + j;
                const int page = __shfl_sync(0xffffffffu, my_page, j);
                const int st = blk % kS;
                if (blk >= kS) {
                    if (!ptx::mbar_wait_warp(&sm.empty[st], ((blk / kS) - 1) & 1)) {
                        if (lane == 0) atomicOr(err, kErrWait);
                        return;
                    }
                }
                if (lane == 0) {
                    int c1, c2, c3;
                    if (kind == 0) { c1 = blk * kVerifyBlock; c2 = g; c3 = b; }
                    else           { c1 = 0;                  c2 = g; c3 = page; }
                    if constexpr (FP8) {  // one 8 KB box of codes each (128 codes per row)
                        ptx::mbar_arrive_expect_tx(&sm.full[st], 2 * kBlock8Bytes);
                        ptx::tma_load_4d(sm.k8[st], &tmk, 0, c1, c2, c3, &sm.full[st]);
                        ptx::tma_load_4d(sm.v8[st], &tmv, 0, c1, c2, c3, &sm.full[st]);
                    } else {
                        ptx::mbar_arrive_expect_tx(&sm.full[st], kStageBytes);
                        for (int hf = 0; hf < 2; ++hf) {
                            ptx::tma_load_4d(sm.k[st][hf], &tmk, hf * 64, c1, c2, c3, &sm.full[st]);
                            ptx::tma_load_4d(sm.v[st][hf], &tmv, hf * 64, c1, c2, c3, &sm.full[st]);
                        }
                    }
                }
                __syncwarp();
            }
        }
        return;
    }

    // ------------------------------------------------------ consumer warps
    // Q tile -> shared memory (swizzled like the K tiles), zero rows past q_len*G.
    for (int x = threadIdx.x; x < kVerifyRows * 16; x += kConsumers * 32) {
        const int r = x >> 4, c = x & 15;
        const int t = r / G, hh = r % G;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (t < q_len)
            val = *reinterpret_cast<const uint4 *>(
                q + (static_cast<long>(r0 + t) * Hq + g * G + hh) * kD + c * 8);
        if constexpr (FP8) {  // bf16 -> f16 operands
            const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&val);
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(p2[i]);
                w[i] = ptx::pack_f16x2(f.x, f.y);
            }
            val = make_uint4(w[0], w[1], w[2], w[3]);
        }
        *reinterpret_cast<uint4 *>(sm.q[c >> 3] + sw128(r, (c & 7) * 8)) = val;
    }
    ptx::named_bar_sync(1, kConsumers * 32);

    const int mt = warp & 1, kh = warp >> 1;
    const bool active = mt * 16 < q_len * G;  // this warp's rows hold real queries
    uint32_t qf[8][4];
    if (active) {
        if constexpr (FP8) {  // k positions {2c,2c+1 | 2c+8,2c+9} = d {4c,4c+1 | 4c+2,4c+3}
            const int c = lane & 3;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int d = kk * 16 + 4 * c;
                const uint8_t *half = sm.q[d >> 6];
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int row = mt * 16 + (lane >> 2) + 8 * h2;
                    const uint8_t *p = half + sw128(row, d & 56) + (d & 7) * 2;
                    qf[kk][h2] = *reinterpret_cast<const uint32_t *>(p);
                    qf[kk][2 + h2] = *reinterpret_cast<const uint32_t *>(p + 4);
                }
            }
        } else {
            const int row = mt * 16 + (lane & 15);
            for (int kk = 0; kk < 8; ++kk) {
                const int d = kk * 16 + (lane >> 4) * 8;
                ptx::ldsm_x4(ptx::smem_u32(sm.q[d >> 6]) + sw128(row, d & 63), qf[kk][0],
                             qf[kk][1], qf[kk][2], qf[kk][3]);
            }
        }
    }
    // query positions of this thread's two rows (-1: padding row, sees nothing)
    int qpos[2];
    for (int h2 = 0; h2 < 2; ++h2) {
        const int r = mt * 16 + (lane >> 2) + h2 * 8;
        const int t = r / G;
        qpos[h2] = (t < q_len) ? L - q_len + t : -1;
    }
    const int win = (kind == 0) ? window : 0;
    const float sl2 = scale * kLog2e * (FP8 ? k_scale[g] : 1.f);  // the K scale joins the score scale

    float oacc[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) oacc[n][0] = oacc[n][1] = oacc[n][2] = oacc[n][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

    for (int blk = 0; blk < nblk; ++blk) {
        const int st = blk % kS;
        if (!ptx::mbar_wait(&sm.full[st], (blk / kS) & 1)) {
            if (lane == 0) atomicOr(err, kErrWait);
            sm.abort = 1;
            break;
        }
        // ring: a warp whose 32 keys of this block all lie past the last slot skips it
        if (active && (kind != 0 || blk * kVerifyBlock + kh * 32 < R)) {
            // S = Q K^T for this warp's 16 rows x 32 keys
            float s[4][4];
#pragma unroll
            for (int n = 0; n < 4; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
            const int mi = lane >> 3;
            if constexpr (FP8) {
                // one ldmatrix per 16-d chunk: matrix j = keys 8j..8j+7 of this half
                const int key = kh * 32 + 8 * mi + (lane & 7);
                const uint32_t krow = ptx::smem_u32(sm.k8[st]) + key * 128;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    uint32_t r[4];
                    ptx::ldsm_x4(krow + (((kk ^ key) & 7) << 4), r[0], r[1], r[2], r[3]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t b0, b1;
                        ptx::e4m3x4_to_f16x2x2(r[j], b0, b1);
                        mma16816<true>(s[j], qf[kk], b0, b1);
                    }
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const int d = kk * 16 + (mi & 1) * 8;
                    const uint32_t kbase = ptx::smem_u32(sm.k[st][d >> 6]);
#pragma unroll
                    for (int np = 0; np < 2; ++np) {
                        const int key = kh * 32 + np * 16 + (mi >> 1) * 8 + (lane & 7);
                        uint32_t b0, b1, b2, b3;
                        ptx::ldsm_x4(kbase + sw128(key, d & 63), b0, b1, b2, b3);
                        mma16816<false>(s[2 * np], qf[kk], b0, b1);
                        mma16816<false>(s[2 * np + 1], qf[kk], b2, b3);
                    }
                }
            }
            // mask, scale to log2 units, online softmax.  A page that ends at or
            // before the first draft's position is visible to every query row:
            // only padding rows are masked there
            float mx[2] = {-INFINITY, -INFINITY};
            if (kind == 1 && (src.pb + blk + 1) * kVerifyBlock - 1 <= L - q_len) {
#pragma unroll
                for (int n = 0; n < 4; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float val = qpos[e >> 1] >= 0 ? s[n][e] * sl2 : -INFINITY;
                        s[n][e] = val;
                        mx[e >> 1] = fmaxf(mx[e >> 1], val);
                    }
            } else {
#pragma unroll
                for (int n = 0; n < 4; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = kh * 32 + n * 8 + 2 * (lane & 3) + (e & 1);
                        const int p = src.position(blk, c);
                        const float val = key_visible(qpos[e >> 1], p, win) ? s[n][e] * sl2 : -INFINITY;
                        s[n][e] = val;
                        mx[e >> 1] = fmaxf(mx[e >> 1], val);
                    }
            }
            // the running max is raised lazily: only when a row's block max
            // exceeds it by more than 2^8, so O is rarely rescaled and every
            // weight stays <= 2^8 (well inside bf16 / f16)
            bool grow = false;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                mx[h2] = fmaxf(mx[h2], __shfl_xor_sync(0xffffffffu, mx[h2], 1));
                mx[h2] = fmaxf(mx[h2], __shfl_xor_sync(0xffffffffu, mx[h2], 2));
                grow |= mx[h2] > mrow[h2] + kRescaleLog2;
            }
            if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const float mn = fmaxf(mrow[h2], mx[h2]);
                    const float alpha = ptx::exp2_approx(mrow[h2] - (mn == -INFINITY ? 0.f : mn));
                    mrow[h2] = mn;
                    lrow[h2] *= alpha;
#pragma unroll
                    for (int n = 0; n < 16; ++n) {
                        oacc[n][2 * h2] *= alpha;
                        oacc[n][2 * h2 + 1] *= alpha;
                    }
                }
            }
            float mbase[2];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) mbase[h2] = (mrow[h2] == -INFINITY) ? 0.f : mrow[h2];
#pragma unroll
            for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float pv = ptx::exp2_approx(s[n][e] - mbase[e >> 1]);
                    s[n][e] = pv;
                    lrow[e >> 1] += pv;
                }
            // O += P V  (P from registers as bf16 A fragments)
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
                uint32_t pa[4];
                pa[0] = pack16<FP8>(s[2 * k2][0], s[2 * k2][1]);
                pa[1] = pack16<FP8>(s[2 * k2][2], s[2 * k2][3]);
                pa[2] = pack16<FP8>(s[2 * k2 + 1][0], s[2 * k2 + 1][1]);
                pa[3] = pack16<FP8>(s[2 * k2 + 1][2], s[2 * k2 + 1][3]);
                const int key = kh * 32 + k2 * 16 + (mi & 1) * 8 + (lane & 7);
                if constexpr (FP8) {
                    // matrices: keys 0-7 / 8-15 of this chunk x d-chunks 2dp, 2dp+1
                    const uint32_t vrow = ptx::smem_u32(sm.v8[st]) + key * 128;
#pragma unroll
                    for (int dp = 0; dp < 4; ++dp) {
                        const int dch = 2 * dp + (mi >> 1);
                        uint32_t r[4];
                        ptx::ldsm_x4_t(vrow + (((dch ^ key) & 7) << 4), r[0], r[1], r[2], r[3]);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {  // d-chunk 2dp + h: registers 2h, 2h+1
                            const int nd = 2 * dp + h;
                            // bytes (0, 2) -> even d, bytes (1, 3) -> odd d: one permute, two converts
                            uint32_t e0, o0, e1, o1;
                            ptx::e4m3x4_to_f16x2x2(__byte_perm(r[2 * h], 0u, 0x3120u), e0, o0);
                            ptx::e4m3x4_to_f16x2x2(__byte_perm(r[2 * h + 1], 0u, 0x3120u), e1, o1);
                            mma16816<true>(oacc[2 * nd], pa, e0, e1);
                            mma16816<true>(oacc[2 * nd + 1], pa, o0, o1);
                        }
                    }
                } else {
#pragma unroll
                    for (int nd = 0; nd < 8; ++nd) {
                        const int d = nd * 16 + (mi >> 1) * 8;
                        uint32_t b0, b1, b2, b3;
                        ptx::ldsm_x4_t(ptx::smem_u32(sm.v[st][d >> 6]) + sw128(key, d & 63), b0,
                                       b1, b2, b3);
                        mma16816<false>(oacc[2 * nd], pa, b0, b1);
                        mma16816<false>(oacc[2 * nd + 1], pa, b2, b3);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.empty[st]);
    }

    // ---- merge the two key halves (warp kh=1 -> smem -> warp kh=0)
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        lrow[h2] += __shfl_xor_sync(0xffffffffu, lrow[h2], 1);
        lrow[h2] += __shfl_xor_sync(0xffffffffu, lrow[h2], 2);
    }
    ptx::named_bar_sync(1, kConsumers * 32);  // every warp is done with the stage buffers
    // rows padded to kMergeStride floats: float2 writes of 8 rows hit distinct banks
    float *mo = sm.merge() + mt * 16 * kMergeStride;
    if (kh == 1 && active) {
#pragma unroll
        for (int n = 0; n < 16; ++n)
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int rr = (lane >> 2) + h2 * 8, d = acc_d<FP8>(n, lane & 3);
                *reinterpret_cast<float2 *>(mo + rr * kMergeStride + d) =
                    make_float2(acc_x<FP8>(oacc, n, h2), acc_y<FP8>(oacc, n, h2));
            }
        if ((lane & 3) == 0)
            for (int h2 = 0; h2 < 2; ++h2) {
                sm.merge_ml[mt][(lane >> 2) + h2 * 8][0] = mrow[h2];
                sm.merge_ml[mt][(lane >> 2) + h2 * 8][1] = lrow[h2];
            }
    }
    ptx::named_bar_sync(1, kConsumers * 32);
    const bool lead = kh == 0 && active && !sm.abort;  // warps that hold the merged rows
    if (lead) {
        float sa[2], sb[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int rr = (lane >> 2) + h2 * 8;
            const float mb = sm.merge_ml[mt][rr][0], lb = sm.merge_ml[mt][rr][1];
            const float mm = merge_scale(mrow[h2], mb, &sa[h2], &sb[h2]);
            lrow[h2] = lrow[h2] * sa[h2] + lb * sb[h2];
            mrow[h2] = mm;
        }
#pragma unroll
        for (int n = 0; n < 16; ++n)
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int rr = (lane >> 2) + h2 * 8, d = acc_d<FP8>(n, lane & 3);
                const float2 x = *reinterpret_cast<const float2 *>(mo + rr * kMergeStride + d);
                float &ax = acc_x<FP8>(oacc, n, h2), &ay = acc_y<FP8>(oacc, n, h2);
                ax = ax * sa[h2] + x.x * sb[h2];
                ay = ay * sa[h2] + x.y * sb[h2];
            }
    }

    if (finalize) {
        // add the sink once; bf16 rows staged in shared memory (rows padded to
        // kStageRowBytes), then written with coalesced 16-byte stores
        uint8_t *ost = sm.ostage();
        if (lead) {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int r = mt * 16 + (lane >> 2) + h2 * 8;
                const int hh = r % G;
                const float sig = sink[g * G + hh];
                float inv;
                if (isinf(sig) && sig > 0.f) {
                    inv = 0.f;
                } else {
                    const float s2 = sig * kLog2e;
                    float ssa, ssb;
                    merge_scale(mrow[h2], s2, &ssa, &ssb);
                    const float z = lrow[h2] * ssa + ssb;
                    inv = ssa / z * (FP8 ? v_scale[g] : 1.f);  // the V scale joins the output
                }
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    const int d = acc_d<FP8>(n, lane & 3);
                    *reinterpret_cast<uint32_t *>(ost + r * kStageRowBytes + d * 2) =
                        ptx::pack_bf16x2(acc_x<FP8>(oacc, n, h2) * inv, acc_y<FP8>(oacc, n, h2) * inv);
                }
            }
        }
        ptx::named_bar_sync(1, kConsumers * 32);
        if (!sm.abort) {
            for (int x = threadIdx.x; x < kVerifyRows * 16; x += kConsumers * 32) {
                const int r = x >> 4, c = x & 15;
                if (r >= q_len * G) break;
                const int t = r / G, hh = r % G;
                *reinterpret_cast<uint4 *>(o + (static_cast<long>(r0 + t) * Hq + g * G + hh) * kD +
                                           c * 8) =
                    *reinterpret_cast<const uint4 *>(ost + r * kStageRowBytes + c * 16);
            }
        }
    } else if (lead) {
        // partial state of this split: m (log2 units), l, unnormalised o
        const long unit = (static_cast<long>(b) * Hkv + g) * nsplit + split;
        float *wo = ws_o + unit * kVerifyRows * kD;
        float *wml = ws_ml + unit * kVerifyRows * 2;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int r = mt * 16 + (lane >> 2) + h2 * 8;
            if ((lane & 3) == 0) {
                wml[r * 2 + 0] = mrow[h2];
                wml[r * 2 + 1] = lrow[h2];
            }
            const float vs = FP8 ? v_scale[g] : 1.f;  // the V scale joins the output
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                const int d = acc_d<FP8>(n, lane & 3);
                *reinterpret_cast<float2 *>(wo + r * kD + d) =
                    make_float2(acc_x<FP8>(oacc, n, h2) * vs, acc_y<FP8>(oacc, n, h2) * vs);
            }
        }
    }
}

// Split-KV merge for the paged cache: per (request, kv head), combine the
// splits' (m, l, o) by log-sum-exp and add the sink term once:
//   M = max(sigma, m_s),  o = sum_s 2^(m_s-M) o_s / (2^(sigma-M) + sum_s 2^(m_s-M) l_s)
// A split CTA whose pipeline wait ran out leaves its partials unwritten and
// sets ATTN_DEVERR_WAIT_TIMEOUT before this kernel starts (stream order), as
// does an earlier launch that timed out; the merge then writes nothing, so no
// output is ever made from scratch that this call did not write.
__global__ void __launch_bounds__(256)
    verify_combine_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_ml,
                          const int32_t *__restrict__ cu_q, const int32_t *__restrict__ seq_lens,
                          const float *__restrict__ sink, __nv_bfloat16 *__restrict__ o,
                          int nsplit, int Hq, int Hkv, int q_max, int max_ctx, int max_pages,
                          const unsigned *err) {
    if (ptx::prior_timeout(err)) return;
    const int g = blockIdx.x, b = blockIdx.y;
    const int G = Hq / Hkv;
    const int r0 = cu_q[b], q_len = cu_q[b + 1] - r0, L = seq_lens[b];
    if (q_len <= 0 || q_len > q_max || q_len * G > kVerifyRows || L < q_len || L > max_ctx ||
        (L + kVerifyBlock - 1) / kVerifyBlock > max_pages)
        return;  // the verify kernel already flagged the request
    const int ns = verify_num_splits((L + kVerifyBlock - 1) / kVerifyBlock, kVerifyChunkPages);
    const int r = threadIdx.x >> 3, part = threadIdx.x & 7;  // 32 rows x 8 parts of 16 d
    const int t = r / G, hh = r % G;
    if (t >= q_len) return;
    const long unit0 = (static_cast<long>(b) * Hkv + g) * nsplit;
    const float sig = sink[g * G + hh];
    __nv_bfloat16 *orow = o + (static_cast<long>(r0 + t) * Hq + g * G + hh) * kD + part * 16;
    if (isinf(sig) && sig > 0.f) {
        for (int d = 0; d < 16; d += 2)
            *reinterpret_cast<uint32_t *>(orow + d) = ptx::pack_bf16x2(0.f, 0.f);
        return;
    }
    float M = sig * kLog2e;
    for (int s = 0; s < ns; ++s) M = fmaxf(M, ws_ml[((unit0 + s) * kVerifyRows + r) * 2]);
    const float base = (M == -INFINITY) ? 0.f : M;
    float z = ptx::exp2_approx(sig * kLog2e - base);
    float acc[16];
#pragma unroll
    for (int d = 0; d < 16; ++d) acc[d] = 0.f;
    for (int s = 0; s < ns; ++s) {
        const float *ml = ws_ml + ((unit0 + s) * kVerifyRows + r) * 2;
        const float w = ptx::exp2_approx(ml[0] - base);
        z += w * ml[1];
        const float4 *src =
            reinterpret_cast<const float4 *>(ws_o + ((unit0 + s) * kVerifyRows + r) * kD + part * 16);
#pragma unroll
        for (int d4 = 0; d4 < 4; ++d4) {
            const float4 x = src[d4];
            acc[4 * d4 + 0] += w * x.x;
            acc[4 * d4 + 1] += w * x.y;
            acc[4 * d4 + 2] += w * x.z;
            acc[4 * d4 + 3] += w * x.w;
        }
    }
    const float inv = 1.f / z;
#pragma unroll
    for (int d = 0; d < 16; d += 2)
        *reinterpret_cast<uint32_t *>(orow + d) = ptx::pack_bf16x2(acc[d] * inv, acc[d + 1] * inv);
}

template <bool FP8>
size_t verify_smem_bytes() { return sizeof(VerifySmem<FP8>) + 1024; }

}  // namespace

cudaError_t launch_verify_ring(const VerifyMaps &maps, const void *q, const int32_t *cu_q,
                               const int32_t *seq_lens, const float *sink, void *o, int B, int Hq,
                               int Hkv, int window, int R, int q_max, float scale,
                               unsigned int *err, cudaStream_t s) {
    if (B == 0) return cudaSuccess;
    const size_t smem = verify_smem_bytes<false>();
    cudaError_t e = cudaFuncSetAttribute(verify_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    verify_kernel<false><<<dim3(1, Hkv, B), kThreads, smem, s>>>(
        maps.k, maps.v, static_cast<const __nv_bfloat16 *>(q), cu_q, seq_lens, nullptr, 0, 0, sink,
        static_cast<__nv_bfloat16 *>(o), nullptr, nullptr, 1, 0, Hq, Hkv, window, R, q_max, 0,
        scale, 1, nullptr, nullptr, err);
    return cudaGetLastError();
}

cudaError_t launch_verify_paged(const VerifyMaps &maps, const void *q, const int32_t *cu_q,
                                const int32_t *seq_lens, const int32_t *page_table, int max_pages,
                                int num_pages, const float *sink, void *o, float *ws_o,
                                float *ws_ml, int nsplit, int B, int Hq, int Hkv, int q_max,
                                int max_ctx, float scale, const float *k_scale,
                                const float *v_scale, unsigned int *err, cudaStream_t s) {
    if (B == 0) return cudaSuccess;
    const bool fp8 = k_scale != nullptr;
    const size_t smem = fp8 ? verify_smem_bytes<true>() : verify_smem_bytes<false>();
    auto kern = fp8 ? verify_kernel<true> : verify_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int finalize = (nsplit == 1) ? 1 : 0;
    // ordinary launches: a paged verify streams for a millisecond or more, and
    // letting the next kernel launch early measured slower here (the 8 x
    // 262144-token, 4-token call: 1.44 ms against 1.30 ms)
    kern<<<dim3(nsplit, Hkv, B), kThreads, smem, s>>>(
        maps.k, maps.v, static_cast<const __nv_bfloat16 *>(q), cu_q, seq_lens, page_table,
        max_pages, num_pages, sink, static_cast<__nv_bfloat16 *>(o), ws_o, ws_ml, nsplit, 1, Hq,
        Hkv, 0, 0, q_max, max_ctx, scale, finalize, k_scale, v_scale, err);
    e = cudaGetLastError();
    if (e != cudaSuccess || finalize) return e;
    verify_combine_kernel<<<dim3(Hkv, B), 256, 0, s>>>(ws_o, ws_ml, cu_q, seq_lens, sink,
                                                       static_cast<__nv_bfloat16 *>(o), nsplit, Hq,
                                                       Hkv, q_max, max_ctx, max_pages, err);
    return cudaGetLastError();
}

}  // namespace attn

// MTP verify against the SWA ring buffer on the 5th-generation tensor cores
// (sm_103a), bf16 in/out, fp32 accumulation, D = 128.
//
// The step (release announcement "小米开源 MiMo-V2-Flash", figure "Multi-Token
// Prediction"; technical-report summary, section "MTP加速"): every request
// scores its real token and up to three drafts in one pass, draft t seeing the
// history and drafts 0..t; the SWA layers read a fixed-size cache (section
// "将效率推向极限") -- here a ring of R = W + q_max - 1 slots per (request,
// kv head), position p in slot p mod R.
//
// A unit is one (request, kv head): its q_len x G query rows (G = 8 heads of
// the kv group, q_len <= 4 tokens) meet the whole ring in one pass.  The
// kernel is persistent: one CTA per SM walks its units u = cta, cta + grid,
// ... (at most 64) so that the cache reads of later units overlap the work on
// earlier ones, and two softmax warpgroups take alternate units so that two
// units' dependent chains (S, softmax, PV, store) run side by side:
//   - warp 0 loads Q (one box of 8 heads per token) and K of all R slots (one
//     box of 144 rows per D half; rows past the ring read 0) into a 3-stage
//     ring (44 KB per stage); warp 2 loads V into a 2-stage ring (36 KB);
//   - warp 1 issues, whichever is ready first, S = Q K^T of the next unit or
//     O = P V of the oldest unit whose P is written, into the TMEM slot of the
//     unit's warpgroup (256 columns each).  S is one tcgen05.mma group with
//     M = 128: the A descriptor's 8-row-group stride is 256 bytes, so MMA rows
//     32t..32t+7 read token t's 8 heads (one 1 KB swizzle atom) and the other
//     rows read unused data whose results are ignored; token t's scores land
//     in TMEM lane quarter t.  PV takes P from TMEM and V from shared memory;
//   - warps 4-7 (units 0, 2, 4, ..) and 8-11 (units 1, 3, ..): warp w serves
//     token t = w mod 4, the TMEM lane quarter it may access: four threads per
//     row through the 16-lane TMEM load/store shapes, the max seeded with the
//     sink logit, P (bf16) written over the S columns; then the unit's O is
//     normalised and stored.
// Each unit's request fields (and its 8 sink logits) are read once into
// shared memory after the wait on the preceding grid (programmatic dependent
// launch).  Before that wait a CTA only initialises its barriers and TMEM and
// asks L2 to prefetch the rings of its first units: a prefetch reads nothing
// into the SM, so it can never see stale data, and every global read and
// write of the kernel comes after the wait.
// Mask: slot s holds position ring_slot_position_r0(s, L, R, L mod R); it is
// visible from query position i iff that position is in [max(0, i-W+1), i],
// i.e. iff s lies in one of the two intervals of ring_visible_slots().
#include "index_math.cuh"
#include "internal.h"
#include "ptx_sm103.cuh"
#include "tc_tile.cuh"

#include <mutex>
#include <type_traits>

namespace attn {
namespace {
namespace vring {

using namespace tc;

// Bits of the slots [a, a + n) that fall in the 32-slot word starting at base.
ATTN_DEV uint32_t interval_bits(int a, int n, int base) {
    const int lo = max(a - base, 0), hi = min(a + n - base, 32);
    if (hi <= lo) return 0u;
    const uint32_t span = (hi - lo == 32) ? 0xffffffffu : ((1u << (hi - lo)) - 1u);
    return span << lo;
}

constexpr int kMaxTokens = 4;                     // q_max supported by this kernel
constexpr int kG = 8;                             // query heads per kv head
constexpr int kN = kVerifyRingKeys;               // key rows per D half (R rounded up to 16)
constexpr int kKHalf = kN * kHalfRowBytes;        // 18 KB
constexpr int kQHalf = kMaxTokens * kG * kHalfRowBytes;  // 4 KB
constexpr int kQKStages = 3, kVStages = 2;
constexpr int kThreads = 384;  // warps 0 (Q,K), 1 (MMA), 2 (V), 3 (spare), 4-11 two softmax groups
constexpr int kSlotCols = 256;                    // TMEM columns per softmax group
constexpr int kOCol = 96;                         // O accumulator column (P uses 0..71)
constexpr int kPrefetchUnits = 2;                 // rings per CTA asked of L2 before the wait
constexpr uint32_t kIdescPV = ptx::idesc_bf16(128, 128, false, true);
constexpr unsigned kErrCtx = 0x2u, kErrQlen = 0x4u;
static_assert(kN % 16 == 0 && kN <= 256 && kOCol >= kN / 2 && kOCol + 128 <= kSlotCols,
              "TMEM layout");
static_assert(kN == 8 * (8 + 8 + 2), "the softmax walks 18 repetitions of 8 columns: x8, x8, x2");

struct __align__(1024) QKStage {
    uint8_t q[2][kQHalf];  // [D half][token][head] rows of 128 B
    uint8_t k[2][kKHalf];  // [D half][slot] rows of 128 B
};
struct __align__(1024) VStage {
    uint8_t v[2][kKHalf];
};
struct UnitMeta {
    int b, g, r0, q_len, L;  // q_len = 0: nothing to compute or store for this unit
};

struct __align__(1024) Smem {
    QKStage qk[kQKStages];
    VStage v[kVStages];
    UnitMeta meta[kVerifyRingUnitsPerCta];          // this CTA's units, in order
    float msink[kVerifyRingUnitsPerCta][kG];        // their 8 sink logits
    uint64_t qk_full[kQKStages], qk_empty[kQKStages], v_full[kVStages], v_empty[kVStages];
    uint64_t s_full[2], p_full[2], o_full[2], tmem_empty[2];  // per softmax group
    uint64_t meta_ready, mma_done;
    uint32_t tmem_base;
    int abort;
};

// A unit's request: rows r0..r0+q_len-1 of q/o, L cached positions.  Returns
// 0 for a unit to compute, -1 for an empty request, else the error bits.
ATTN_DEV int unit_request(const int32_t *cu_q, const int32_t *seq_lens, int b, int q_max,
                          int q_rows, int &r0, int &q_len, int &L) {
    r0 = cu_q[b];
    q_len = cu_q[b + 1] - r0;
    L = seq_lens[b];
    if (q_len <= 0) return -1;
    if (q_len > q_max || q_len > kMaxTokens || r0 < 0 || r0 + q_len > q_rows) return kErrQlen;
    if (L < q_len) return kErrCtx;
    return 0;
}

ATTN_DEV bool aborted(const Smem &sm) {
    return *reinterpret_cast<const volatile int *>(&sm.abort) != 0;
}
ATTN_DEV void set_abort(Smem &sm, unsigned *err) {
    *reinterpret_cast<volatile int *>(&sm.abort) = 1;
    atomicOr(err, kErrWait);
}
// Waits until every copy armed on `full` (uses 0..uses-1) has landed (bounded).
ATTN_DEV void drain(uint64_t *full, int uses) {
    if (uses > 0) ptx::mbar_wait(full, (uses - 1) & 1);
}

__global__ void __launch_bounds__(kThreads, 1)
    verify_ring_tc_kernel(const __grid_constant__ CUtensorMap tmq,
                          const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tmv,
                          const int32_t *__restrict__ cu_q, const int32_t *__restrict__ seq_lens,
                          const float *__restrict__ sink, __nv_bfloat16 *__restrict__ o, int Hq,
                          int Hkv, int nunits, int window, int R, int q_max, int q_rows,
                          float scale, unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                         ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x, grid = gridDim.x;
    const int n = (nunits - cta + grid - 1) / grid;  // units of this CTA (<= kVerifyRingUnitsPerCta)

    // ---- prologue: nothing here reads or writes global memory
    if (threadIdx.x == 0) {
        for (int i = 0; i < kQKStages; ++i) {
            ptx::mbar_init(&sm.qk_full[i], 1);
            ptx::mbar_init(&sm.qk_empty[i], 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            ptx::mbar_init(&sm.v_full[i], 1);
            ptx::mbar_init(&sm.v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&sm.s_full[i], 1);
            ptx::mbar_init(&sm.p_full[i], 4);      // one arrival per warp of the group
            ptx::mbar_init(&sm.o_full[i], 1);
            ptx::mbar_init(&sm.tmem_empty[i], 4);  // one arrival per warp of the group
        }
        ptx::mbar_init(&sm.meta_ready, 1);
        ptx::mbar_init(&sm.mma_done, 1);
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(&sm.tmem_base, 2 * kSlotCols);
        ptx::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmq);
        ptx::prefetch_tmap(&tmk);
        ptx::prefetch_tmap(&tmv);
        for (int i = 0; i < kPrefetchUnits && i < n; ++i) {
            const int u = cta + i * grid;
            for (int hf = 0; hf < 2; ++hf) {
                ptx::tma_prefetch_l2_4d(&tmk, hf * 64, 0, u % Hkv, u / Hkv);
                ptx::tma_prefetch_l2_4d(&tmv, hf * 64, 0, u % Hkv, u / Hkv);
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    ptx::grid_dep_wait();
    ptx::grid_dep_launch_dependents();

    // Every unit of the CTA flows through the pipeline in order; a unit whose
    // request is empty or invalid is computed on whatever Q the stage holds
    // and stores nothing.  K and V depend only on the unit index, so their
    // first copies start before the request fields are read.
    if (warp == 0) {
        // ----------------- TMA of Q and K; this warp also reads the requests
        if (lane == 0)
            for (int k = 0; k < kQKStages && k < n; ++k) {
                const int u = cta + k * grid;
                ptx::mbar_expect_tx(&sm.qk_full[k], 2 * kKHalf);
                for (int hf = 0; hf < 2; ++hf)
                    ptx::tma_load_4d(sm.qk[k].k[hf], &tmk, hf * 64, 0, u % Hkv, u / Hkv,
                                     &sm.qk_full[k]);
            }
        for (int i = lane; i < n; i += 32) {
            const int u = cta + i * grid, b = u / Hkv, g = u % Hkv;
            int r0, q_len, L;
            const int st = unit_request(cu_q, seq_lens, b, q_max, q_rows, r0, q_len, L);
            if (st > 0 && g == 0) atomicOr(err, static_cast<unsigned>(st));
            sm.meta[i] = st == 0 ? UnitMeta{b, g, r0, q_len, L} : UnitMeta{b, g, 0, 0, 0};
#pragma unroll
            for (int hh = 0; hh < kG; ++hh) sm.msink[i][hh] = sink[g * kG + hh];
        }
        if (lane == 0) sm.abort = ptx::prior_timeout(err) ? 1 : 0;
        __syncwarp();
        if (lane == 0) {
            ptx::mbar_arrive(&sm.meta_ready);
            const bool skip = sm.abort != 0;  // an earlier launch timed out: do nothing more
            int k = 0;
            for (; k < n; ++k) {
                const UnitMeta m = sm.meta[k];
                const int s = k % kQKStages;
                const uint32_t qbytes = skip ? 0u : 2u * m.q_len * kG * kHalfRowBytes;
                if (k >= kQKStages) {
                    if (skip) break;
                    if (aborted(sm) || !ptx::mbar_wait(&sm.qk_empty[s], ((k / kQKStages) - 1) & 1)) {
                        set_abort(sm, err);
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(&sm.qk_full[s], 2 * kKHalf + qbytes);
                    for (int hf = 0; hf < 2; ++hf)
                        ptx::tma_load_4d(sm.qk[s].k[hf], &tmk, hf * 64, 0, m.g, m.b, &sm.qk_full[s]);
                } else {
                    ptx::mbar_arrive_expect_tx(&sm.qk_full[s], qbytes);  // K is already on its way
                }
                if (qbytes)
                    for (int tt = 0; tt < m.q_len; ++tt)
                        for (int hf = 0; hf < 2; ++hf)
                            ptx::tma_load_3d(sm.qk[s].q[hf] + tt * kG * kHalfRowBytes, &tmq, hf * 64,
                                             m.g * kG, m.r0 + tt, &sm.qk_full[s]);
            }
            // copies in flight land before the CTA may exit (bounded waits);
            // units 0..k-1 were armed (the first stages always are)
            for (int s = 0; s < kQKStages; ++s)
                drain(&sm.qk_full[s], (k - s + kQKStages - 1) / kQKStages);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------- TMA of V
        if (lane == 0) {
            int k = 0;
            for (; k < n; ++k) {
                const int u = cta + k * grid, s = k % kVStages;
                if (k >= kVStages) {
                    if (k == kVStages && (!ptx::mbar_wait(&sm.meta_ready, 0) || sm.abort)) break;
                    if (aborted(sm) || !ptx::mbar_wait(&sm.v_empty[s], ((k / kVStages) - 1) & 1)) {
                        set_abort(sm, err);
                        break;
                    }
                }
                ptx::mbar_arrive_expect_tx(&sm.v_full[s], 2 * kKHalf);
                for (int hf = 0; hf < 2; ++hf)
                    ptx::tma_load_4d(sm.v[s].v[hf], &tmv, hf * 64, 0, u % Hkv, u / Hkv, &sm.v_full[s]);
            }
            for (int s = 0; s < kVStages; ++s) drain(&sm.v_full[s], (k - s + kVStages - 1) / kVStages);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMAs
        if (lane == 0 && ptx::mbar_wait(&sm.meta_ready, 0) && !sm.abort && n > 0) {
            const uint32_t idS = ptx::idesc_bf16(128, kN, false, false);
            int nS = 0, nP = 0;  // next unit to score, next unit to aggregate
            uint64_t t_last = ptx::globaltimer();
            bool ok = true;
            for (uint32_t it = 0; nP < n; ++it) {
                bool progress = false;
                if (nP < nS) {  // O = P V of unit nP (P in TMEM columns 0..kN/2-1 of its slot)
                    const int j = nP & 1, vs = nP % kVStages;
                    if (ptx::mbar_poll(ptx::smem_u32(&sm.p_full[j]), (nP >> 1) & 1) &&
                        ptx::mbar_poll(ptx::smem_u32(&sm.v_full[vs]), (nP / kVStages) & 1)) {
                        ptx::tc_fence_after();
                        const uint32_t slot = tmem + j * kSlotCols;
                        for (int kk = 0; kk < kN / 16; ++kk)
                            ptx::mma_ts(slot + kOCol, slot + kk * 8, vmajor_desc(sm.v[vs].v[0], kk, kKHalf),
                                        kIdescPV, kk > 0 ? 1u : 0u);
                        ptx::tc_commit(&sm.o_full[j]);
                        ptx::tc_commit(&sm.v_empty[vs]);
                        ++nP;
                        progress = true;
                    }
                }
                if (nS < n && nS < nP + 2) {  // S = Q K^T of unit nS into its group's slot
                    const int j = nS & 1, s = nS % kQKStages;
                    if (ptx::mbar_poll(ptx::smem_u32(&sm.qk_full[s]), (nS / kQKStages) & 1) &&
                        (nS < 2 || ptx::mbar_poll(ptx::smem_u32(&sm.tmem_empty[j]), ((nS >> 1) - 1) & 1))) {
                        ptx::tc_fence_after();
                        // A rows 32t + i (i < 8) read token t, head i (8-row group
                        // stride 256 B, i.e. group 4t starts at t's 1 KB atom)
                        const QKStage &sg = sm.qk[s];
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t ad = ptx::sdesc_sw128(
                                ptx::smem_u32(sg.q[kk >> 2]) + (kk & 3) * 32, 16, 256);
                            ptx::mma_ss(tmem + j * kSlotCols, ad, kmajor_desc(sg.k[kk >> 2], kk & 3),
                                        idS, kk > 0 ? 1u : 0u);
                        }
                        ptx::tc_commit(&sm.s_full[j]);
                        ptx::tc_commit(&sm.qk_empty[s]);
                        ++nS;
                        progress = true;
                    }
                }
                if (progress) {
                    t_last = ptx::globaltimer();
                } else if ((it & 63u) == 0 &&
                           (aborted(sm) || ptx::globaltimer() - t_last > ptx::kWaitTimeoutNs)) {
                    ok = false;
                    break;
                }
            }
            if (!ok) set_abort(sm, err);
            if (nS > 0) {  // every MMA completes before TMEM is released (bounded)
                ptx::tc_commit(&sm.mma_done);
                ptx::mbar_wait(&sm.mma_done, 0);
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ---------------- softmax and epilogue: group j takes units j, j + 2, ..
        // Warp w may access TMEM lane quarter w mod 4, which holds token t's 8
        // heads in lanes 0..7.  The 16-lane TMEM shapes give each row to a
        // quad of threads: thread 4q + r holds columns 8k + 2r and 8k + 2r + 1
        // (k = 0, 1, ..) of row q (16x256b), and the bf16 pair of exactly those
        // two keys is P column 4k + r (16x128b).  Lanes 8..15 are read and
        // written but unused; lanes 16..31 are not touched.
        const int j = (warp - 4) >> 2, t = warp & 3, qrow = lane >> 2, r = lane & 3;
        const uint32_t tS = tmem + (static_cast<uint32_t>(t * 32) << 16) + j * kSlotCols;
        const uint32_t tO = tS + kOCol;
        const float sl2 = scale * kLog2e;
        bool ok = ptx::mbar_wait_warp(&sm.meta_ready, 0);
        const int nn = (ok && !sm.abort) ? n : 0;
        for (int k = j; k < nn; k += 2) {
            const UnitMeta m = sm.meta[k];
            const float sig = sm.msink[k][qrow];
            const int ph = (k >> 1) & 1;
            ok = !__any_sync(0xffffffffu, aborted(sm)) && ptx::mbar_wait_warp(&sm.s_full[j], ph);
            if (!ok) break;
            ptx::tc_fence_after();
            const int qpos = m.L - m.q_len + t;
            // visible slots: at most two intervals, the same for the whole
            // warp; as bitmask words pre-shifted by 2r, the two keys of
            // repetition k are bits 8(k%4) and 8(k%4)+1 of word k/4
            const RingVisible vis = ring_visible_slots(m.L, R, window, qpos);
            uint32_t vm[kN / 32 + 1];
#pragma unroll
            for (int w = 0; w <= kN / 32; ++w)
                vm[w] = (interval_bits(vis.a1, vis.n1, 32 * w) | interval_bits(vis.a2, vis.n2, 32 * w)) >>
                        (2 * r);
            auto vis_bit = [&](int kr, int e) { return ((vm[kr >> 2] >> (8 * (kr & 3) + e)) & 1u) != 0u; };
            // the 144 scores of this thread's quad row in one TMEM read: x8, x8
            // and x2 repetitions (columns 8k + 2r, 8k + 2r + 1 at v[4k], v[4k+1])
            uint32_t v[4 * 18];
            {
                uint32_t (&v0)[32] = *reinterpret_cast<uint32_t (*)[32]>(&v[0]);
                uint32_t (&v1)[32] = *reinterpret_cast<uint32_t (*)[32]>(&v[32]);
                uint32_t (&v2)[8] = *reinterpret_cast<uint32_t (*)[8]>(&v[64]);
                ptx::tmem_ld_16x256b_x8(tS, v0);
                ptx::tmem_ld_16x256b_x8(tS + 64, v1);
                ptx::tmem_ld_16x256b_x2(tS + 128, v2);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            }
            // masked max of the raw scores (scale > 0) over the quad
            float mx = -INFINITY;
#pragma unroll
            for (int kr = 0; kr < 18; ++kr)
                mx = fmax3(mx, vis_bit(kr, 0) ? __uint_as_float(v[4 * kr]) : -INFINITY,
                           vis_bit(kr, 1) ? __uint_as_float(v[4 * kr + 1]) : -INFINITY);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            // seeded with the sink logit; sigma = +inf gives m = +inf and every p = 0
            const float mfull = fmaxf(sig * kLog2e, mx * sl2);
            const float mb = (mfull == -INFINITY) ? 0.f : mfull;
            // P = 2^(s*scale*log2e - m); the pair of repetition k is P column
            // 4k + r (written over S columns already read)
            float ls = 0.f;
            uint32_t pw[2 * 18];
#pragma unroll
            for (int kr = 0; kr < 18; ++kr) {
                const float p0 = vis_bit(kr, 0)
                                     ? ptx::exp2_approx(fmaf(__uint_as_float(v[4 * kr]), sl2, -mb))
                                     : 0.f;
                const float p1 = vis_bit(kr, 1)
                                     ? ptx::exp2_approx(fmaf(__uint_as_float(v[4 * kr + 1]), sl2, -mb))
                                     : 0.f;
                ls += p0 + p1;
                pw[2 * kr] = ptx::pack_bf16x2(p0, p1);
                pw[2 * kr + 1] = 0u;  // lane q + 8: unused row
            }
            ptx::tmem_st_16x128b_x8(tS, *reinterpret_cast<uint32_t (*)[16]>(&pw[0]));
            ptx::tmem_st_16x128b_x8(tS + 32, *reinterpret_cast<uint32_t (*)[16]>(&pw[16]));
            ptx::tmem_st_16x128b_x2(tS + 64, *reinterpret_cast<uint32_t (*)[4]>(&pw[32]));
            ptx::tmem_st_wait();
            ls += __shfl_xor_sync(0xffffffffu, ls, 1);
            ls += __shfl_xor_sync(0xffffffffu, ls, 2);
            ptx::tc_fence_before();
            if (lane == 0) ptx::mbar_arrive(&sm.p_full[j]);
            // ---- epilogue of this unit once its PV has run
            ok = ptx::mbar_wait_warp(&sm.o_full[j], ph);
            if (!ok) break;
            ptx::tc_fence_after();
            const bool sink_all = isinf(sig) && sig > 0.f;
            if (!sink_all && !(isinf(sig) && sig < 0.f)) ls += ptx::exp2_approx(sig * kLog2e - mb);
            const float inv = sink_all ? 0.f : 1.f / ls;
            const bool real = t < m.q_len;
            // O row q: thread 4q + r holds columns 8k + 2r, +1 and stores them
            // as one bf16 pair
            uint32_t *dst = reinterpret_cast<uint32_t *>(
                                o + (static_cast<long>(m.r0 + t) * Hq + m.g * kG + qrow) * 128) + r;
            uint32_t ov[64];
            ptx::tmem_ld_16x256b_x8(tO, *reinterpret_cast<uint32_t (*)[32]>(&ov[0]));
            ptx::tmem_ld_16x256b_x8(tO + 64, *reinterpret_cast<uint32_t (*)[32]>(&ov[32]));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            if (real) {
#pragma unroll
                for (int kr = 0; kr < 16; ++kr)
                    dst[4 * kr] = ptx::pack_bf16x2(__uint_as_float(ov[4 * kr]) * inv,
                                                   __uint_as_float(ov[4 * kr + 1]) * inv);
            }
            ptx::tc_fence_before();
            if (lane == 0) ptx::mbar_arrive(&sm.tmem_empty[j]);
        }
        if (!ok && lane == 0) set_abort(sm, err);
    }
    // every warp reconverges before the CTA barrier (the roles above diverge
    // inside warps), so the barrier holds until the last role is done
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 2 * kSlotCols);
    }
}

// Streaming multiprocessors of the current device (cached per device).
int sm_count() {
    static int count[64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (!count[dev] &&
        cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        count[dev] = 148;
    return count[dev];
}

}  // namespace vring
}  // namespace

int verify_ring_tc_supported(int G, int R, int q_max) {
    return G == vring::kG && R >= 1 && R <= vring::kN && q_max >= 1 && q_max <= vring::kMaxTokens;
}

cudaError_t launch_verify_ring_tc(const VerifyMaps &maps, const int32_t *cu_q,
                                  const int32_t *seq_lens, const float *sink, void *o, int B,
                                  int Hq, int Hkv, int window, int R, int q_max, float scale,
                                  unsigned int *err, cudaStream_t s) {
    if (B == 0) return cudaSuccess;
    const size_t smem = sizeof(vring::Smem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(vring::verify_ring_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int nunits = B * Hkv;
    // one CTA per SM, more when a CTA would get over kVerifyRingUnitsPerCta units
    int grid = nunits < vring::sm_count() ? nunits : vring::sm_count();
    const int need = (nunits + kVerifyRingUnitsPerCta - 1) / kVerifyRingUnitsPerCta;
    if (grid < need) grid = need;
    return launch_pdl(vring::verify_ring_tc_kernel, dim3(grid), dim3(vring::kThreads), smem, s,
                      maps.q, maps.k, maps.v, cu_q, seq_lens, sink,
                      static_cast<__nv_bfloat16 *>(o), Hq, Hkv, nunits, window, R, q_max,
                      B * q_max, scale, err);
}

}  // namespace attn

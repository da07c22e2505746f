// Streaming sliding-window sink-attention prefill on the 5th-generation tensor
// cores (sm_103a), bf16 in/out, fp32 accumulation.
//
// What it computes (technical-report summary, fanfer.top "MiMo-V2", sections
// "MiMo-V2-Flash Model Architecture": SWA layers with window W = 128, and
// "Hybrid Sliding Window Attention Architecture": a learnable gpt-oss-style
// sink per head): for every query row, softmax over the scores of its W most
// recent keys plus one sink column (logit sigma_h, no value), times V.
//
// Tiling: a tile is 16 consecutive tokens x the 8 query heads that share one
// kv head (GQA packing, row r = 8*t + hh), i.e. 128 rows, against the 144 keys
// key0 = i0 - 128 .. i0 + 15 that cover every key its rows can see.  A batch
// is B sequences, of T tokens each or packed by cu_seqlens; every sequence
// starts its own tile grid at its first token (positions are relative to the
// sequence, and keys before it are masked like keys before position 0).  Each
// persistent CTA walks a contiguous run of tiles in (b, g, token block) order
// (swa_stream_range), so consecutive tiles share 128 of their 144 keys: K and
// V live in a ring of 16-key blocks in shared memory and a tile loads one new
// block of each (8 KB) besides its 32 KB of Q.  With one CTA per SM every
// byte of Q, K and V is read from HBM once and O is written once; that is the
// roofline of this kernel (HBM-bound: 114 FLOP per byte at W = 128).
//
// Roles (352 threads):
//   warps 0-3 / 4-7  softmax + epilogue of the tiles in TMEM slot 0 / slot 1
//                    (thread = row = TMEM lane);
//   warp 8           TMA producer of Q (3-stage ring) and K blocks (a K block
//                    in ring slot 0..7 is loaded twice: slot and mirror);
//   warp 10          TMA producer of V blocks;
//   warp 9           one thread issues tcgen05.mma: S = Q K^T (bf16 operands
//                    in 128-byte-swizzled shared memory, fp32 S in TMEM; the
//                    K blocks of ring slots 0..7 are also kept at slots
//                    12..19, so a tile's nine blocks are always contiguous
//                    and S is one N = 144 MMA per k-step) and
//                    O = P V (P as bf16 in TMEM over the S columns), choosing
//                    whichever of the next S and the next PV is ready.
// Per TMEM slot (256 columns): S in columns 0..143, P (bf16 pairs) in 0..71,
// O in 96..223.  The epilogue moves O into registers and releases the slot
// before it normalises and stores O, so the next S starts early.
//
// Every wait is bounded (2 s); on expiry the kernel records
// ATTN_DEVERR_WAIT_TIMEOUT, stops issuing, waits (bounded) for its own copies
// and MMAs in flight, frees TMEM and returns.
#include "index_math.cuh"
#include "internal.h"
#include "ptx_sm103.cuh"
#include "tc_tile.cuh"

namespace attn {
namespace {
namespace swa {

using namespace tc;

constexpr int kG = kSwaHeads;                  // query heads per kv head
constexpr int kTT = kSwaTokens;                // tokens per tile
constexpr int kN = kSwaKeys;                   // keys per tile
constexpr int kNB = kSwaTileBlocks;            // key blocks per tile
constexpr int kRing = kSwaRingBlocks;          // K/V ring blocks
constexpr int kQStages = 3;
constexpr int kQHalf = 128 * kHalfRowBytes;    // 16 KB: 128 rows of one D half
constexpr int kBlkHalf = kSwaBlockKeys * kHalfRowBytes;  // 2 KB: one block, one D half
constexpr int kRingHalf = kRing * kBlkHalf;    // one D half of the ring
constexpr int kKRingHalf = (kRing + kNB - 1) * kBlkHalf;  // K ring with its mirror
constexpr int kThreads = 352;
constexpr int kOCol = 96;                      // O accumulator column in a slot
constexpr uint32_t kIdescS = ptx::idesc_bf16(128, kN, false, false);
constexpr uint32_t kIdescPV = ptx::idesc_bf16(128, 128, false, true);
static_assert(kOCol >= kN / 2 && kOCol + 128 <= 256, "slot TMEM layout");
static_assert(kRing >= kNB + 1, "ring must hold a tile's window plus one block");

struct __align__(1024) Smem {
    uint8_t q[kQStages][2][kQHalf];   // [stage][D half]
    uint8_t k[2][kKRingHalf];         // [D half][ring block (+ mirror of 0..7)][16 rows]
    uint8_t v[2][kRingHalf];
    uint64_t q_full[kQStages], q_empty[kQStages];
    uint64_t k_full[kRing], k_empty[kRing], v_full[kRing], v_empty[kRing];
    uint64_t s_full[2], p_full[2], o_full[2], tmem_free[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
    SwaTileCursor first;  // the CTA's first tile
    int ntile;            // and the number of tiles in its run
};
static_assert(sizeof(Smem) + 1024 <= 227 * 1024, "shared memory of one CTA");

// Warp-cooperative forms of the tile order (swa_total_tiles and
// swa_cursor_at; every lane returns the same): the number of tiles of the
// batch, with *bad set when a packed span is invalid, and the cursor of tile u.
ATTN_DEV int count_tiles_warp(const int32_t *cu, int B, int T, int total, int Hkv, int lane,
                              bool *bad) {
    *bad = false;
    if (!cu) return B * Hkv * swa_seq_blocks(T);
    int n = 0;
    bool ok = true;
    for (int b = lane; b < B; b += 32) {
        const SeqSpan sp = seq_span(cu, b, T, total);
        n += swa_seq_blocks(sp.len) * Hkv;
        ok &= sp.ok;
    }
    for (int off = 16; off > 0; off >>= 1) n += __shfl_xor_sync(0xffffffffu, n, off);
    *bad = !__all_sync(0xffffffffu, ok);
    return n;
}
ATTN_DEV SwaTileCursor cursor_at_warp(const int32_t *cu, int B, int T, int total, int Hkv, int u,
                                      int lane) {
    SwaTileCursor c;
    c.g = c.blk = 0;
    if (!cu) {
        c.nblk = swa_seq_blocks(T);
        const int bg = u / c.nblk;
        c.blk = u - bg * c.nblk;
        c.b = bg / Hkv;
        c.g = bg - c.b * Hkv;
        c.start = c.b * T;
        c.len = T;
        return c;
    }
    int acc = 0;  // tiles of the sequences before this chunk of 32
    for (int c0 = 0; c0 < B; c0 += 32) {
        const int b = c0 + lane;
        const int nt = b < B ? swa_seq_blocks(seq_span(cu, b, T, total).len) * Hkv : 0;
        int incl = nt;
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, acc + incl > u);
        if (hit) {  // the first such lane holds tile u (and has tiles)
            const int src = __ffs(static_cast<int>(hit)) - 1;
            const int excl = __shfl_sync(0xffffffffu, incl - nt, src);
            c.b = c0 + src;
            swa_cursor_seq(c, cu, T, total);
            const int rem = u - acc - excl;
            c.g = rem / c.nblk;
            c.blk = rem - c.g * c.nblk;
            return c;
        }
        acc += __shfl_sync(0xffffffffu, incl, 31);
    }
    c.b = B;
    c.nblk = c.start = c.len = 0;
    return c;
}

// Per-tile state of the MMA issuer: the tile, its ring blocks and the blocks
// it releases after use.
struct Issue {
    SwaRingCursor cur;
    SwaTileCursor t;      // the tile
    int k = 0;            // tile index within the CTA's run
    int rel_end = 0;      // blocks [cur.base, rel_end) are released after this tile
    int waited = -1;      // highest block sequence number whose full barrier was seen
    __device__ void advance(int n, int Hkv) {
        swa_ring_step(cur, t.b * Hkv + t.g, kNB);
        const bool next_same = (k + 1 < n) && (t.blk + 1 < t.nblk);
        rel_end = swa_ring_release_end(cur.base, next_same, kNB);
    }
};

// Non-blocking check that blocks up to `last` have landed (full barriers).
ATTN_DEV bool blocks_ready(uint64_t *full, int &waited, int last) {
    while (waited < last) {
        const int n = waited + 1;
        if (!ptx::mbar_test(ptx::smem_u32(&full[n % kRing]), (n / kRing) & 1)) return false;
        waited = n;
    }
    return true;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_swa_stream_kernel(const __grid_constant__ CUtensorMap tmq,
                              const __grid_constant__ CUtensorMap tmk,
                              const __grid_constant__ CUtensorMap tmv,
                              __nv_bfloat16 *__restrict__ out, const float *__restrict__ sink,
                              float *__restrict__ lse, const int32_t *__restrict__ cu, int B,
                              int T, int total, int Hq, int Hkv, int window, float scale,
                              float vscale, unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                         ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kQStages; ++s) {
            ptx::mbar_init(&sm.q_full[s], 1);
            ptx::mbar_init(&sm.q_empty[s], 1);
        }
        for (int s = 0; s < kRing; ++s) {
            ptx::mbar_init(&sm.k_full[s], 1);
            ptx::mbar_init(&sm.k_empty[s], 1);
            ptx::mbar_init(&sm.v_full[s], 1);
            ptx::mbar_init(&sm.v_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&sm.s_full[s], 1);
            ptx::mbar_init(&sm.p_full[s], 128);
            ptx::mbar_init(&sm.o_full[s], 1);
            ptx::mbar_init(&sm.tmem_free[s], 128);
        }
        ptx::mbar_init(&sm.mma_done, 1);
        sm.abort = ptx::prior_timeout(err) ? 1 : 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0) {  // this CTA's run of tiles
        bool bad;
        const int ntiles = count_tiles_warp(cu, B, T, total, Hkv, lane, &bad);
        int u0, u1;
        swa_stream_range(static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), ntiles, &u0,
                         &u1);
        SwaTileCursor c;
        c.b = B;
        c.g = c.blk = c.nblk = c.start = c.len = 0;
        if (u0 < u1) c = cursor_at_warp(cu, B, T, total, Hkv, u0, lane);
        if (lane == 0) {
            sm.first = c;
            sm.ntile = u1 - u0;
            if (bad && blockIdx.x == 0) atomicOr(err, kErrSeqlens);
        }
    }
    if (warp == 9) {
        ptx::tmem_alloc(&sm.tmem_base, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const bool skip = sm.abort != 0;  // an earlier launch timed out: do nothing
    const int n = sm.ntile;
    const SwaTileCursor first = sm.first;

    if (warp == 8 || warp == 10) {
        // --------------------------------------------- TMA producers
        if (lane == 0 && !skip) {
            const bool qk = (warp == 8);
            if (qk) {
                ptx::prefetch_tmap(&tmq);
                ptx::prefetch_tmap(&tmk);
            } else {
                ptx::prefetch_tmap(&tmv);
            }
            uint64_t *full = qk ? sm.k_full : sm.v_full;
            uint64_t *empty = qk ? sm.k_empty : sm.v_empty;
            uint8_t *ring = qk ? sm.k[0] : sm.v[0];
            const CUtensorMap *map = qk ? &tmk : &tmv;
            SwaRingCursor cur;
            SwaTileCursor t = first;
            bool ok = true;
            int last_q = -1, last_s = -1;  // last Q tile and ring block issued
            for (int k = 0; ok && k < n; ++k) {
                if (k > 0) swa_cursor_next(t, cu, B, T, total, Hkv);
                const int i0 = t.blk * kTT;
                const int key0 = i0 + kTT - kN;
                swa_ring_step(cur, t.b * Hkv + t.g, kNB);
                if (qk) {
                    const int st = k % kQStages;
                    if (k >= kQStages && !ptx::mbar_wait(&sm.q_empty[st], ((k / kQStages) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(&sm.q_full[st], 2 * kQHalf);
                    for (int hf = 0; hf < 2; ++hf)
                        ptx::tma_load_3d(sm.q[st][hf], &tmq, hf * 64, t.g * kG, t.start + i0,
                                         &sm.q_full[st]);
                    last_q = k;
                }
                for (int s = cur.first_new; s < cur.first_new + cur.n_new; ++s) {
                    const int slot = s % kRing;
                    if (s >= kRing && !ptx::mbar_wait(&empty[slot], ((s / kRing) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    const bool mirror = qk && slot < kNB - 1;
                    const int half = qk ? kKRingHalf : kRingHalf;
                    ptx::mbar_arrive_expect_tx(&full[slot], (mirror ? 4 : 2) * kBlkHalf);
                    const int kp = key0 + kSwaBlockKeys * (s - cur.base);
                    for (int hf = 0; hf < 2; ++hf) {
                        ptx::tma_load_3d(ring + hf * half + slot * kBlkHalf, map, hf * 64, t.g,
                                         t.start + kp, &full[slot]);
                        if (mirror)
                            ptx::tma_load_3d(ring + hf * half + (slot + kRing) * kBlkHalf, map,
                                             hf * 64, t.g, t.start + kp, &full[slot]);
                    }
                    last_s = s;
                }
            }
            if (!ok) atomicOr(err, kErrWait);
            // copies still in flight land before the CTA may exit (bounded;
            // immediate on the normal path, where every copy was consumed)
            for (int k = (last_q - kQStages + 1 > 0 ? last_q - kQStages + 1 : 0); k <= last_q; ++k)
                ptx::mbar_wait(&sm.q_full[k % kQStages], (k / kQStages) & 1);
            for (int s = (last_s - kRing + 1 > 0 ? last_s - kRing + 1 : 0); s <= last_s; ++s)
                ptx::mbar_wait(&full[s % kRing], (s / kRing) & 1);
        }
        __syncwarp();
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA
        if (lane == 0 && !skip) {
            Issue is, ip;  // next S, next PV
            is.t = ip.t = first;
            if (n > 0) {
                is.advance(n, Hkv);
                ip.advance(n, Hkv);
            }
            const uint32_t kbase[2] = {ptx::smem_u32(sm.k[0]), ptx::smem_u32(sm.k[1])};
            const uint32_t vbase = ptx::smem_u32(sm.v[0]);
            bool ok = true, issued = false;
            uint64_t t_last = ptx::globaltimer();
            uint32_t spins = 0;
            while (ip.k < n) {
                bool prog = false;
                // O = P V for tile ip.k: needs its P and its V blocks
                if (ip.k < is.k) {
                    const int s = ip.k & 1;
                    if (ptx::mbar_test(ptx::smem_u32(&sm.p_full[s]), (ip.k >> 1) & 1) &&
                        blocks_ready(sm.v_full, ip.waited, ip.cur.base + kNB - 1)) {
                        ptx::tc_fence_after();
                        const uint32_t tS = tmem + 256 * s;
                        for (int j = 0; j < kNB; ++j) {
                            const int slot = (ip.cur.base + j) % kRing;
                            const uint64_t bd =
                                ptx::sdesc_sw128(vbase + slot * kBlkHalf, kRingHalf, 1024);
                            ptx::mma_ts(tS + kOCol, tS + j * 8, bd, kIdescPV, j > 0 ? 1u : 0u);
                        }
                        ptx::tc_commit(&sm.o_full[s]);
                        for (int b = ip.cur.base; b < ip.rel_end; ++b)
                            ptx::tc_commit(&sm.v_empty[b % kRing]);
                        issued = true;
                        prog = true;
                        if (++ip.k < n) {
                            swa_cursor_next(ip.t, cu, B, T, total, Hkv);
                            ip.advance(n, Hkv);
                        }
                    }
                }
                // S = Q K^T for tile is.k: needs Q, its K blocks and a free slot
                if (!prog && is.k < n && is.k <= ip.k + 1) {
                    const int s = is.k & 1, st = is.k % kQStages;
                    if (ptx::mbar_test(ptx::smem_u32(&sm.q_full[st]), (is.k / kQStages) & 1) &&
                        blocks_ready(sm.k_full, is.waited, is.cur.base + kNB - 1) &&
                        (is.k < 2 ||
                         ptx::mbar_test(ptx::smem_u32(&sm.tmem_free[s]), ((is.k >> 1) - 1) & 1))) {
                        ptx::tc_fence_after();
                        const uint32_t tS = tmem + 256 * s;
                        const int r = is.cur.base % kRing;  // blocks r..r+8: contiguous (mirror)
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t ad = kmajor_desc(sm.q[st][kk >> 2], kk & 3);
                            const uint32_t kb = kbase[kk >> 2] + (kk & 3) * 32;
                            ptx::mma_ss(tS, ad, ptx::sdesc_sw128(kb + r * kBlkHalf, 16, 1024), kIdescS,
                                        kk > 0 ? 1u : 0u);
                        }
                        ptx::tc_commit(&sm.s_full[s]);
                        ptx::tc_commit(&sm.q_empty[st]);
                        for (int b = is.cur.base; b < is.rel_end; ++b)
                            ptx::tc_commit(&sm.k_empty[b % kRing]);
                        issued = true;
                        prog = true;
                        if (++is.k < n) {
                            swa_cursor_next(is.t, cu, B, T, total, Hkv);
                            is.advance(n, Hkv);
                        }
                    }
                }
                if (prog) {
                    spins = 0;
                } else if ((++spins & 63u) == 0) {
                    const uint64_t now = ptx::globaltimer();
                    if (spins == 64) t_last = now;
                    else if (now - t_last > ptx::kWaitTimeoutNs) { ok = false; break; }
                }
            }
            if (!ok) atomicOr(err, kErrWait);
            if (issued) {  // every MMA issued completes before TMEM is freed
                ptx::tc_commit(&sm.mma_done);
                ptx::mbar_wait(&sm.mma_done, 0);
            }
        }
        __syncwarp();
    } else if (!skip) {
        // ------------------------------------------ softmax + epilogue
        // Thread = row = TMEM lane.  Failure decisions are warp-uniform and
        // there is no barrier inside the loop.
        const int s = warp >> 2;
        const int row = threadIdx.x & 127;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + 256 * s + lane_off, tO = tS + kOCol;
        const int t_in = row / kG, hh = row % kG;
        const float sl2 = scale * kLog2e;
        const bool out32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;  // 32-byte stores
        SwaTileCursor t = first;
        if (s == 1 && n > 1) swa_cursor_next(t, cu, B, T, total, Hkv);
        for (int k = s; k < n; k += 2) {
            if (k > s) {  // two tiles on: this slot takes every other tile
                swa_cursor_next(t, cu, B, T, total, Hkv);
                swa_cursor_next(t, cu, B, T, total, Hkv);
            }
            const int ph = (k >> 1) & 1;
            const int i0 = t.blk * kTT;
            const int key0 = i0 + kTT - kN;
            const int qpos = i0 + t_in, h = t.g * kG + hh;
            int c_lo, c_hi;
            swa_row_cols(qpos, key0, window, &c_lo, &c_hi);
            const bool interior = key0 >= 0;  // uniform over the tile
            const float sig = sink[h];
            if (!ptx::mbar_wait_warp(&sm.s_full[s], ph)) {
                if (lane == 0) atomicOr(err, kErrWait);
                break;
            }
            ptx::tc_fence_after();
            float x[kN];
            tmem_load_row<kN>(tS, x);
            // selects, not conditional stores: a branch per column costs
            // far more than the compare
            if (interior) {
#pragma unroll
                for (int c = 0; c < kN; ++c) x[c] = swa_col_admitted(c, c_lo, c_hi, true) ? x[c] : -INFINITY;
            } else {
#pragma unroll
                for (int c = 0; c < kN; ++c) x[c] = swa_col_admitted(c, c_lo, c_hi, false) ? x[c] : -INFINITY;
            }
            // row max of the raw scores (scale > 0 commutes with max), seeded
            // with the sink logit; four independent partial maxima
            float m4[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // accumulator j takes columns j, j+4, j+8, ...
                m4[j] = fmaxf(x[j], x[j + 4]);
#pragma unroll
                for (int c = j + 8; c < kN; c += 8) m4[j] = fmax3(m4[j], x[c], x[c + 4]);
            }
            const float m = fmaxf(sig * kLog2e, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl2);
            // sigma = +inf: m = +inf, every p is 0 and o is 0
            const float mb = (m == -INFINITY) ? 0.f : m;
            // P = 2^(x*scale*log2e - mb), written as bf16 pairs over the S
            // columns; paired fp32 arithmetic, four partial sums
            const uint64_t sl2x2 = f2(sl2, sl2), nmb = f2(-mb, -mb);
            uint64_t l2[4] = {0, 0, 0, 0};
#pragma unroll
            for (int c = 0; c < kN; c += 2) {
                const float2 a = f2_split(f2_fma(f2(x[c], x[c + 1]), sl2x2, nmb));
                x[c] = ptx::exp2_approx(a.x);
                x[c + 1] = ptx::exp2_approx(a.y);
                l2[(c >> 1) & 3] = f2_add(l2[(c >> 1) & 3], f2(x[c], x[c + 1]));
            }
            tmem_store_p<kN>(tS, x);
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&sm.p_full[s]);
            const float2 ls = f2_split(f2_add(f2_add(l2[0], l2[1]), f2_add(l2[2], l2[3])));
            float l = ls.x + ls.y;
            const bool sink_all = isinf(sig) && sig > 0.f;
            if (!sink_all && !(isinf(sig) && sig < 0.f)) l += ptx::exp2_approx(sig * kLog2e - mb);

            if (!ptx::mbar_wait_warp(&sm.o_full[s], ph)) {
                if (lane == 0) atomicOr(err, kErrWait);
                break;
            }
            ptx::tc_fence_after();
            float o[128];
            tmem_load_row<128>(tO, o);
            ptx::tc_fence_before();
            ptx::mbar_arrive(&sm.tmem_free[s]);  // the slot may take the next S now
            const float inv = sink_all ? 0.f : vscale / l;  // the value scale rides on 1/l
            if (qpos < t.len) {
                const uint64_t inv2 = f2(inv, inv);
                uint4 *dst = reinterpret_cast<uint4 *>(
                    out + (static_cast<long>(t.start + qpos) * Hq + h) * 128);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    uint32_t w[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int c = 16 * i + 2 * j;
                        const float2 y = f2_split(f2_mul(f2(o[c], o[c + 1]), inv2));
                        w[j] = ptx::pack_bf16x2(y.x, y.y);
                    }
                    if (out32) {  // one 32-byte store: a whole sector of the row
                        ptx::st_global_v8(dst + 2 * i, w);
                    } else {
                        dst[2 * i] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[2 * i + 1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
                if (lse)
                    lse[lse_index(cu, t.b, h, qpos, t.start, T, total, Hq)] =
                        sink_all ? INFINITY : (mb + log2f(l)) * kLn2;
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

}  // namespace swa

int sm_count() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

}  // namespace

int prefill_swa_tc_supported(int G, int window) {
    return G == swa::kG && swa_pack_keys(G, window) == swa::kN;
}

int prefill_swa_grid(long max_tiles) {
    return static_cast<int>(max_tiles < sm_count() ? max_tiles : sm_count());
}

cudaError_t launch_prefill_swa_tc(const PrefillMaps &maps, const float *sink, float *lse,
                                  const PrefillBatch &pb, int Hq, int Hkv, int window, float scale,
                                  float vscale, unsigned int *err, cudaStream_t s) {
    if (pb.B == 0 || pb.total == 0) return cudaSuccess;
    // tiles: exact for equal lengths, an upper bound for a packed batch
    const long max_tiles =
        static_cast<long>(Hkv) * (pb.cu ? pb.total / swa::kTT + pb.B
                                        : static_cast<long>(pb.B) * swa_seq_blocks(pb.T));
    const size_t smem = sizeof(swa::Smem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(swa::prefill_swa_stream_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    swa::prefill_swa_stream_kernel<<<prefill_swa_grid(max_tiles), swa::kThreads, smem, s>>>(
        maps.q, maps.k, maps.v, static_cast<__nv_bfloat16 *>(maps.out), sink, lse, pb.cu, pb.B,
        pb.T, pb.total, Hq, Hkv, window, scale, vscale, err);
    return cudaGetLastError();
}

}  // namespace attn

// Host-side replay of the streaming SWA prefill schedule, built from the same
// index functions the kernel runs (index_math.cuh compiled as host code), so
// that the CPU test suite checks the run partition, the ring bookkeeping and
// the column masks without a GPU, for batches of equal length (cu = NULL) and
// packed batches (cu[B+1], T >= the longest sequence).  visits [B*Hkv, T, T+1]
// by position within the sequence; column T counts admitted keys outside the
// sequence.  Returns the largest number of blocks that are
// live (loaded and not yet released) at any point of a run.
#include "index_math.cuh"

extern "C" int swa_stream_visits_host(int32_t *visits, const int32_t *cu, int B, int T,
                                      int total, int Hkv, int window, int grid) {
    using namespace attn;
    const int ntiles = swa_total_tiles(cu, B, T, total, Hkv);
    int max_live = 0;
    for (int cta = 0; cta < grid; ++cta) {
        int u0, u1;
        swa_stream_range(cta, grid, ntiles, &u0, &u1);
        if (u0 >= u1) continue;
        SwaRingCursor cur;
        SwaTileCursor t = swa_cursor_at(cu, B, T, total, Hkv, u0);
        int slot_key[kSwaRingBlocks];
        for (int s = 0; s < kSwaRingBlocks; ++s) slot_key[s] = -(1 << 30);
        int released = 0;  // blocks [0, released) were released
        for (int u = u0; u < u1; ++u) {
            if (u > u0) swa_cursor_next(t, cu, B, T, total, Hkv);
            const int bg = t.b * Hkv + t.g, i0 = t.blk * kSwaTokens;
            const int key0 = i0 + kSwaTokens - kSwaKeys;
            swa_ring_step(cur, bg, kSwaTileBlocks);
            for (int s = cur.first_new; s < cur.first_new + cur.n_new; ++s)
                slot_key[s % kSwaRingBlocks] = key0 + kSwaBlockKeys * (s - cur.base);
            if (cur.seq_next - released > max_live) max_live = cur.seq_next - released;
            const bool interior = key0 >= 0;
            for (int tt = 0; tt < kSwaTokens && i0 + tt < t.len; ++tt) {
                const int qpos = i0 + tt;
                int c_lo, c_hi;
                swa_row_cols(qpos, key0, window, &c_lo, &c_hi);
                int32_t *row = visits + (static_cast<long>(bg) * T + qpos) * (T + 1);
                for (int j = 0; j < kSwaTileBlocks; ++j) {
                    const int kb = slot_key[(cur.base + j) % kSwaRingBlocks];
                    for (int cc = 0; cc < kSwaBlockKeys; ++cc) {
                        if (!swa_col_admitted(j * kSwaBlockKeys + cc, c_lo, c_hi, interior)) continue;
                        const int key = kb + cc;
                        row[(key >= 0 && key < t.len) ? key : T] += 1;
                    }
                }
            }
            const bool next_same = (u + 1 < u1) && (t.blk + 1 < t.nblk);
            released = swa_ring_release_end(cur.base, next_same, kSwaTileBlocks);
        }
    }
    return max_live;
}

// Ring visibility as the tensor-core verify kernel computes it: out[s] = the
// position held by slot s if visible from query position qpos, else -1.
extern "C" void ring_visible_host(int32_t *out, int L, int R, int window, int qpos) {
    using namespace attn;
    const RingVisible vis = ring_visible_slots(L, R, window, qpos);
    for (int s = 0; s < R; ++s) out[s] = vis.contains(s) ? ring_slot_position(s, L, R) : -1;
}

// Block order of the GA-tiled prefill: out[3*bid .. 3*bid+2] = (pair, head, sequence).
extern "C" void ga_block_coords_host(int32_t *out, int nblocks, int npairs, int Hq, int Hkv) {
    using namespace attn;
    for (int bid = 0; bid < nblocks; ++bid) {
        int pair, h, b;
        ga_block_coords(bid, npairs, Hq, Hkv, &pair, &h, &b);
        out[3 * bid] = pair;
        out[3 * bid + 1] = h;
        out[3 * bid + 2] = b;
    }
}

// Integer index arithmetic shared by every kernel of the library and by the
// index-dump kernels, so that a bit-exact dump tests the code the kernels run.
//
// Visibility (MiMo-V2-Flash technical-report summary, section "MiMo-V2-Flash
// Model Architecture": sliding window W = 128 for SWA layers, full causal
// attention for GA layers): key position j is visible from query position i
// iff 0 <= j <= i and, for SWA, j >= i - W + 1.
//
// SWA ring (release announcement "小米开源 MiMo-V2-Flash", section "将效率推向极限":
// fixed-size SWA KV cache): R = W + q_max - 1 slots, position p in slot p mod R.
//
// GA paged cache: position p in page page_table[b][p / P] at offset p % P.
#pragma once

#include <stdint.h>

#define ATTN_HD __host__ __device__ __forceinline__

namespace attn {

// (bitwise operators: no branch per element in the kernels' unrolled masks)
ATTN_HD bool key_visible(int i, int j, int window) {
    return (j >= 0) & (j <= i) & ((window <= 0) | (j > i - window));
}

// The position held by ring slot `s` once positions 0..L-1 were written into
// a ring of R slots: the unique p in [L-R, L) with p = s (mod R), or -1.
// With r0 = L mod R (computed once per request), slots r0..R-1 hold
// L-R .. L-R+(R-1-r0) and slots 0..r0-1 hold L-r0 .. L-1.
ATTN_HD int ring_slot_position_r0(int s, int L, int R, int r0) {
    const int p = s + (s >= r0 ? L - R - r0 : L - r0);
    return p >= 0 ? p : -1;
}
ATTN_HD int ring_slot_position(int s, int L, int R) {
    return ring_slot_position_r0(s, L, R, L % R);
}
// The ring slots visible from query position qpos (window W) once positions
// 0..L-1 were written: those holding positions in [max(0, qpos-W+1), qpos].
// Since slots r0..R-1 and 0..r0-1 each hold increasing positions, they are at
// most two intervals [a1, a1+n1) and [a2, a2+n2).  contains() is two unsigned
// compares and a bitwise OR: no branch per slot.
struct RingVisible {
    int a1, n1, a2, n2;
    ATTN_HD bool contains(int s) const {
        return (static_cast<unsigned>(s - a1) < static_cast<unsigned>(n1)) |
               (static_cast<unsigned>(s - a2) < static_cast<unsigned>(n2));
    }
};
ATTN_HD RingVisible ring_visible_slots(int L, int R, int window, int qpos) {
    const int r0 = L % R;
    int lo = qpos - window + 1;
    if (lo < 0) lo = 0;
    const int a1 = lo - (L - R - r0) > r0 ? lo - (L - R - r0) : r0;
    const int b1 = qpos - (L - R - r0) < R - 1 ? qpos - (L - R - r0) : R - 1;
    const int a2 = lo - (L - r0) > 0 ? lo - (L - r0) : 0;
    const int b2 = qpos - (L - r0) < r0 - 1 ? qpos - (L - r0) : r0 - 1;
    RingVisible v;
    v.a1 = a1;
    v.n1 = b1 >= a1 ? b1 - a1 + 1 : 0;
    v.a2 = a2;
    v.n2 = b2 >= a2 ? b2 - a2 + 1 : 0;
    return v;
}

// ---- prefill batches: sequence b covers the tokens [start, start + len) of
// the flattened token axis.  cu == nullptr: B sequences of T tokens each
// (start = b*T); otherwise the packed layout cu[b] .. cu[b+1] with
// cu[B] = total and T >= every length.  A span outside [0, total), longer
// than T or with a negative length is invalid: it holds no tokens and the
// kernels report it.
struct SeqSpan {
    int start, len;
    bool ok;
};
ATTN_HD SeqSpan seq_span(const int32_t *cu, int b, int T, int total) {
    SeqSpan s;
    if (!cu) {
        s.start = b * T;
        s.len = T;
        s.ok = true;
        return s;
    }
    s.start = cu[b];
    const int e = cu[b + 1];
    s.ok = (s.start >= 0) & (e >= s.start) & (e <= total) & (e - s.start <= T);
    s.len = s.ok ? e - s.start : 0;
    return s;
}
// Index of the LSE of (sequence b, head h, position i): [B, Hq, T] for
// batches of equal length, [Hq, total] for packed batches.
ATTN_HD long lse_index(const int32_t *cu, int b, int h, int i, int start, int T, int total,
                       int Hq) {
    return cu ? static_cast<long>(h) * total + start + i
              : (static_cast<long>(b) * Hq + h) * T + i;
}

// ---- GA prefill tiling: BM query rows per tile, BN keys per key tile.
constexpr int kTileM = 128;
constexpr int kTileN = 128;

// Key tiles [first, last] that a query tile starting at q0 (rows q0..q0+BM-1,
// clipped to T) must visit; window <= 0 is full causal.
ATTN_HD void ga_key_tiles(int q0, int T, int window, int *first, int *last) {
    int qhi = q0 + kTileM - 1;
    if (qhi > T - 1) qhi = T - 1;
    *last = qhi / kTileN;
    int lo = (window > 0) ? q0 - window + 1 : 0;
    if (lo < 0) lo = 0;
    *first = lo / kTileN;
}

// Block order of the GA-tiled prefill: block -> (256-row pair, query head,
// sequence).  The G = Hq/Hkv heads that share a kv head vary fastest, then
// the pair (latest, i.e. heaviest under causal masking, first), then the kv
// head, then the sequence: the CTAs resident at one time read one kv head's
// K/V (16.8 MB at T = 32768, D = 128), which L2 then serves to all of them.
ATTN_HD void ga_block_coords(int bid, int npairs, int Hq, int Hkv, int *pair, int *h, int *b) {
    const int G = Hq / Hkv;
    const int hh = bid % G, rest = bid / G;
    *pair = npairs - 1 - rest % npairs;
    const int rest2 = rest / npairs;
    *h = (rest2 % Hkv) * G + hh;
    *b = rest2 / Hkv;
}

// True when some (row, key) pair of the key tile `j` is invisible from the
// query tile starting at q0, i.e. the tile needs the element mask; interior
// tiles skip it.
ATTN_HD bool ga_tile_needs_mask(int q0, int j, int window) {
    const int k_lo = j * kTileN, k_hi = j * kTileN + kTileN - 1;
    if (k_hi > q0) return true;                                   // crosses the diagonal
    if (window > 0 && k_lo < q0 + kTileM - 1 - window + 1) return true;  // crosses the window edge
    return false;
}

// ---- backward tiling.  The dK/dV kernel owns keys j0..j0+bk-1 and visits the
// query tiles of bq rows [first, last] holding a row that sees one of them;
// the dQ kernel owns query rows i0..i0+bq-1 and visits the key tiles of bk
// keys [first, last] holding a key one of its rows sees (window <= 0: causal).
ATTN_HD void bwd_kv_query_tiles(int j0, int T, int window, int bk, int bq, int *first, int *last) {
    *first = j0 / bq;
    int hi = T - 1;
    if (window > 0 && j0 + bk - 1 + window - 1 < hi) hi = j0 + bk - 1 + window - 1;
    *last = hi / bq;
}
ATTN_HD void bwd_q_key_tiles(int i0, int T, int window, int bq, int bk, int *first, int *last) {
    int lo = window > 0 ? i0 - window + 1 : 0;
    if (lo < 0) lo = 0;
    *first = lo / bk;
    int hi = i0 + bq - 1;
    if (hi > T - 1) hi = T - 1;
    *last = hi / bk;
}
// True when every pair of query rows [i0, i0+nq) and keys [j0, j0+nk) is
// visible, so the tile needs no element mask.
ATTN_HD bool tile_all_visible(int i0, int nq, int j0, int nk, int window) {
    if (j0 + nk - 1 > i0) return false;                      // some key after some row
    if (window > 0 && j0 <= i0 + nq - 1 - window) return false;  // some key out of a window
    return true;
}

// ---- packed SWA prefill tiling: a tile holds TT = 128/G consecutive query
// tokens of the G query heads that share one kv head (row r = t*G + hh), and
// one key tile of N = round_up(TT + W - 1, 16) keys starting at
// key0 = i0 + TT - N, which covers every key any of its rows can see.
ATTN_HD int swa_pack_tokens(int G) { return kTileM / G; }
ATTN_HD int swa_pack_keys(int G, int window) {
    int need = swa_pack_tokens(G) + window - 1;
    return (need + 15) & ~15;
}
ATTN_HD int swa_pack_key0(int i0, int G, int window) {
    return i0 + swa_pack_tokens(G) - swa_pack_keys(G, window);
}

// ---- streaming SWA prefill (G = 8, 16 tokens x 8 heads per tile, N = 144):
// a CTA walks a contiguous run of tiles in (b, g, token block) order
// and keeps the keys of the current window in a ring of 16-key blocks in
// shared memory, so each tile loads one new K/V block (nine after a change of
// (b, g) or at the start of the run).
constexpr int kSwaBlockKeys = 16;                 // keys per ring block
constexpr int kSwaHeads = 8;                      // query heads per kv head (G)
constexpr int kSwaTokens = 16;                    // tokens per tile (128 / G)
constexpr int kSwaKeys = 144;                     // keys per tile
constexpr int kSwaTileBlocks = kSwaKeys / kSwaBlockKeys;  // 9
constexpr int kSwaRingBlocks = 12;                // ring capacity in blocks

// Tiles [*u0, *u1) of CTA `cta` of `grid` (balanced contiguous runs).
ATTN_HD void swa_stream_range(int cta, int grid, int ntiles, int *u0, int *u1) {
    *u0 = static_cast<int>((static_cast<long long>(cta) * ntiles) / grid);
    *u1 = static_cast<int>((static_cast<long long>(cta + 1) * ntiles) / grid);
}

// A tile of the streaming order: sequence b, kv head g, token block blk of
// the nblk blocks of sequence b (tokens start + 16*blk ..).  Tiles run in
// (b, g, blk) order over the sequences that hold tokens.
struct SwaTileCursor {
    int b, g, blk, nblk, start, len;
};
ATTN_HD int swa_seq_blocks(int len) { return (len + kSwaTokens - 1) / kSwaTokens; }
ATTN_HD void swa_cursor_seq(SwaTileCursor &c, const int32_t *cu, int T, int total) {
    const SeqSpan s = seq_span(cu, c.b, T, total);
    c.start = s.start;
    c.len = s.len;
    c.nblk = swa_seq_blocks(s.len);
}
// The next tile of the order (past the last tile: b == B).
ATTN_HD void swa_cursor_next(SwaTileCursor &c, const int32_t *cu, int B, int T, int total,
                             int Hkv) {
    if (++c.blk < c.nblk) return;
    c.blk = 0;
    if (++c.g < Hkv) return;
    c.g = 0;
    while (++c.b < B) {
        swa_cursor_seq(c, cu, T, total);
        if (c.nblk > 0) return;
    }
}
// Serial reference of the order: the number of tiles, and tile u.
ATTN_HD int swa_total_tiles(const int32_t *cu, int B, int T, int total, int Hkv) {
    int n = 0;
    for (int b = 0; b < B; ++b) n += swa_seq_blocks(seq_span(cu, b, T, total).len) * Hkv;
    return n;
}
ATTN_HD SwaTileCursor swa_cursor_at(const int32_t *cu, int B, int T, int total, int Hkv, int u) {
    SwaTileCursor c;
    c.g = c.blk = c.nblk = c.start = c.len = 0;
    for (c.b = 0; c.b < B; ++c.b) {
        swa_cursor_seq(c, cu, T, total);
        const int nt = c.nblk * Hkv;
        if (u < nt) {
            c.g = u / c.nblk;
            c.blk = u - c.g * c.nblk;
            return c;
        }
        u -= nt;
    }
    return c;
}

// Block bookkeeping in load order: every block a CTA loads gets the next
// sequence number n and lives in ring slot n mod ring.  A tile reads the
// blocks base .. base+nb-1, whose keys start at key0 + 16*(n - base).
struct SwaRingCursor {
    int seq_next = 0;   // sequence number of the next block to load
    int prev_bg = -1;   // (b*Hkv + g) of the previous tile
    int base = 0;       // first block of the current tile
    int first_new = 0;  // first block loaded for the current tile
    int n_new = 0;      // blocks loaded for the current tile (nb or 1)
};
ATTN_HD void swa_ring_step(SwaRingCursor &c, int bg, int nb) {
    c.first_new = c.seq_next;
    if (bg != c.prev_bg) {
        c.n_new = nb;
        c.base = c.seq_next;
    } else {
        c.n_new = 1;
        c.base = c.seq_next + 1 - nb;
    }
    c.seq_next += c.n_new;
    c.prev_bg = bg;
}
// End of the blocks [base, end) that the current tile is the last to read:
// one block when the next tile continues the same (b, g), all nb otherwise.
ATTN_HD int swa_ring_release_end(int base, bool next_same_bg, int nb) {
    return next_same_bg ? base + 1 : base + nb;
}

// Visible key columns [*c_lo, *c_hi] of the row at query position qpos in a
// key tile starting at key0.
ATTN_HD void swa_row_cols(int qpos, int key0, int window, int *c_lo, int *c_hi) {
    int lo = qpos - window + 1;
    if (lo < 0) lo = 0;
    *c_lo = lo - key0;
    *c_hi = qpos - key0;
}
// Whether the streaming kernel admits column c of such a row.  Interior tiles
// (key0 >= 0, window in [114, 129]) test only columns < 32 against c_lo and
// columns > 128 against c_hi: every other column is visible to all 128 rows.
ATTN_HD bool swa_col_admitted(int c, int c_lo, int c_hi, bool interior) {
    if (interior) {
        if (c < 32) return c >= c_lo;
        if (c > 128) return c <= c_hi;
        return true;
    }
    return (c >= c_lo) & (c <= c_hi);
}

// ---- verify split-KV geometry (GA paged): each split covers a fixed number
// of whole pages; split s covers positions [s*chunk, (s+1)*chunk).
ATTN_HD int verify_num_splits(int max_ctx, int chunk) { return (max_ctx + chunk - 1) / chunk; }
// Page-table indices [*pb, *pe) that split s reads for a request of L positions.
ATTN_HD void verify_split_pages(int s, int L, int page_size, int chunk_pages, int *pb, int *pe) {
    const int npages = (L + page_size - 1) / page_size;
    *pb = s * chunk_pages;
    *pe = (*pb + chunk_pages < npages) ? *pb + chunk_pages : npages;
}

}  // namespace attn

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

ATTN_HD bool key_visible(int i, int j, int window) {
    return j >= 0 && j <= i && (window <= 0 || j > i - window);
}

// The position held by ring slot `s` once positions 0..L-1 were written into
// a ring of R slots: the unique p in [L-R, L) with p = s (mod R), or -1.
ATTN_HD int ring_slot_position(int s, int L, int R) {
    int base = L - R;
    int r = (s - base) % R;
    if (r < 0) r += R;
    int p = base + r;
    return p >= 0 ? p : -1;
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

// True when some (row, key) pair of the key tile `j` is invisible from the
// query tile starting at q0, i.e. the tile needs the element mask; interior
// tiles skip it.
ATTN_HD bool ga_tile_needs_mask(int q0, int j, int window) {
    const int k_lo = j * kTileN, k_hi = j * kTileN + kTileN - 1;
    if (k_hi > q0) return true;                                   // crosses the diagonal
    if (window > 0 && k_lo < q0 + kTileM - 1 - window + 1) return true;  // crosses the window edge
    return false;
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

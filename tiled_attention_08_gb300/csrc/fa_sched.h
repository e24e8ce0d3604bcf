// fa_sched.h -- tile bounds under the causal mask, round order of persistent grids and the grid
// rules of the three attention passes (host and device).
#pragma once

namespace fa {

// Queries and keys may differ in length.  Under the causal mask the queries are the last Lq
// positions of the key sequence: query row i sees key j iff j <= i + (Lk - Lq).

// Key tiles that query tile qt (rows [128 qt, min(128 qt + 128, Lq))) sees: all of them, or
// under the causal mask those holding a key at or before the tile's last row; 0 when even the
// last row sees no key.
__host__ __device__ __forceinline__ int q_tile_kv(int qt, int Lq, int Lk, bool causal) {
    const int n_k = (Lk + 127) / 128;
    if (!causal) return n_k;
    const int last_row = (qt * 128 + 127 < Lq - 1) ? qt * 128 + 127 : Lq - 1;
    const int last_key = last_row + (Lk - Lq);
    if (last_key < 0) return 0;
    return (last_key / 128 + 1 < n_k) ? last_key / 128 + 1 : n_k;
}

// First query tile that sees key tile kt (every later query tile sees it too).
__host__ __device__ __forceinline__ int k_tile_q0(int kt, int Lq, int Lk, bool causal) {
    if (!causal) return 0;
    const int first_row = kt * 128 - (Lk - Lq);  // first row that sees key 128 kt
    return first_row <= 0 ? 0 : first_row / 128;
}

// Whether tile (query tile qt, key tile kt) needs the element mask: some key of it lies after
// what the tile's first row may see (causal), or past the last key, or its rows run past Lq.
__host__ __device__ __forceinline__ bool tile_masked(int qt, int kt, int Lq, int Lk, bool causal) {
    return (causal && kt * 128 + 127 > qt * 128 + (Lk - Lq)) || (kt * 128 + 128 > Lk) ||
           (qt * 128 + 128 > Lq);
}

// Of `grid` persistent CTAs, CTA `cta` takes in round r the tile id r*grid + cta for even r and
// r*grid + (grid-1-cta) for odd r (-1 once the ids run out).  Ids are heaviest-first inside a
// head group (tile_coords), so every CTA alternates between the heavy and the light end of
// consecutive rounds and the per-CTA totals stay even under the causal mask.
__host__ __device__ __forceinline__ int persistent_tile(int round, int cta, int grid, int total) {
    const int b = (round & 1) ? (grid - 1 - cta) : cta;
    const long long id = (long long)round * grid + b;
    return id < (long long)total ? (int)id : -1;
}

// Grid of a pass over `items` work items per head-batch whose rows hold `row_tiles` tiles in
// all (summed over the items of one head).  Persistent (one CTA per SM) when the items see at
// most `max_mean` tiles on average and there are more items than SMs; otherwise one CTA per
// item.  The fixed cost of a CTA is worth hiding only for short rows; for long rows the
// one-CTA-per-item kernels run each tile a little faster than the persistent ones, and that
// outweighs it.  (The forward's persistent CTAs take fixed rounds, persistent_tile; the
// backward's take the next item from a counter, fa_queue.cuh.)
constexpr int kPersistMaxKv = 32;
__host__ __device__ __forceinline__ int persistent_grid(int items_per_head, long long row_tiles,
                                                        int BH, int max_mean, int n_sm) {
    const long long items = (long long)items_per_head * BH;
    const bool short_rows = row_tiles <= (long long)max_mean * items_per_head;
    return (n_sm > 0 && n_sm < items && short_rows) ? n_sm : (int)items;
}

// Grid of the dQ pass: one item per query tile.
__host__ __device__ __forceinline__ int dq_grid(int Lq, int Lk, int BH, bool causal, int n_sm) {
    const int n_q = (Lq + 127) / 128;
    long long kv = 0;
    for (int qt = 0; qt < n_q; ++qt) kv += q_tile_kv(qt, Lq, Lk, causal);
    return persistent_grid(n_q, kv, BH, kPersistMaxKv, n_sm);
}

// Grid of the dK/dV pass: one item per key tile.  Its persistent kernel carries per-item state
// across the query-tile loop in elementwise warps at the 96-register limit of an 18-warp CTA
// (a few spilled bytes at D = 128), so per query tile it is a little slower than the
// one-CTA-per-item kernel; with items taken from the work counter it wins up to a mean of
// kDkdvPersistMaxKv query tiles per key tile (measured: B8 H32 L4096 causal, mean 16.5, 1.534
// against 1.597 ms at D = 128 and 1.092 against 1.190 ms at D = 64; B1 H16 L16384 D64 causal,
// mean 64.5, 0.991 against 0.987 ms).
constexpr int kDkdvPersistMaxKv = 32;
__host__ __device__ __forceinline__ int dkdv_grid(int Lq, int Lk, int BH, bool causal,
                                                  int n_sm) {
    const int n_q = (Lq + 127) / 128, n_k = (Lk + 127) / 128;
    long long rows = 0;
    for (int kt = 0; kt < n_k; ++kt) rows += n_q - k_tile_q0(kt, Lq, Lk, causal);
    return persistent_grid(n_k, rows, BH, kDkdvPersistMaxKv, n_sm);
}

// Grid of the forward: one item per pair of query tiles (2p, 2p+1), which streams the key tiles
// of its heavier tile.
__host__ __device__ __forceinline__ int fwd_grid(int Lq, int Lk, int BH, bool causal, int n_sm) {
    const int n_q = (Lq + 127) / 128, n_pairs = (n_q + 1) / 2;
    long long kv = 0;
    for (int p = 0; p < n_pairs; ++p)
        kv += q_tile_kv(2 * p + 1 < n_q ? 2 * p + 1 : 2 * p, Lq, Lk, causal);
    return persistent_grid(n_pairs, kv, BH, kPersistMaxKv, n_sm);
}

}  // namespace fa

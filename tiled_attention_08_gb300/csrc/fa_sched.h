// fa_sched.h -- round order of persistent grids (host and device).
#pragma once

namespace fa {

// Of `grid` persistent CTAs, CTA `cta` takes in round r the tile id r*grid + cta for even r and
// r*grid + (grid-1-cta) for odd r (-1 once the ids run out).  Ids are heaviest-first inside a
// head group (tile_coords), so every CTA alternates between the heavy and the light end of
// consecutive rounds and the per-CTA totals stay even under the causal mask.
__host__ __device__ __forceinline__ int persistent_tile(int round, int cta, int grid, int total) {
    const int b = (round & 1) ? (grid - 1 - cta) : cta;
    const long long id = (long long)round * grid + b;
    return id < (long long)total ? (int)id : -1;
}

// Grid of a pass over `items` work items that see `mean_kv2` / 2 key tiles on average.
// Persistent (one CTA per SM) when the items see at most kPersistMaxKv key tiles on average and
// there are more items than SMs; otherwise one CTA per item.  The fixed cost of a CTA is worth
// hiding only for short rows; for long rows the hardware's own block scheduling balances the
// causal items better than fixed rounds.
constexpr int kPersistMaxKv = 32;
__host__ __device__ __forceinline__ int persistent_grid(int items, int mean_kv2, int n_sm) {
    return (n_sm > 0 && n_sm < items && mean_kv2 <= 2 * kPersistMaxKv) ? n_sm : items;
}

// Grid of the dQ pass: one item per query tile, which sees tile+1 key tiles under the causal
// mask (mean (n_tiles+1)/2) and every key tile otherwise.
__host__ __device__ __forceinline__ int dq_grid(int n_tiles, int BH, bool causal, int n_sm) {
    return persistent_grid(n_tiles * BH, causal ? n_tiles + 1 : 2 * n_tiles, n_sm);
}

// Grid of the dK/dV pass: one item per key tile, which sees n_tiles - tile query tiles under the
// causal mask (mean (n_tiles+1)/2) and every query tile otherwise.  Its persistent kernel carries
// per-item state across the query-tile loop in elementwise warps already at the 96-register
// limit of an 18-warp CTA, so it costs a few percent per query tile against the one-CTA-per-item
// kernel; it is used only for rows of at most kDkdvPersistMaxKv query tiles on average, where
// the saved fixed cost is larger (measured: B1 H32 L2048 causal, mean 8.5, +2.3%; B16 H32 L512
// and L1024, +3 to +13%; B8 H32 L4096 causal, mean 16.5, -2.8%).
constexpr int kDkdvPersistMaxKv = 12;
__host__ __device__ __forceinline__ int dkdv_grid(int n_tiles, int BH, bool causal, int n_sm) {
    const int mean_kv2 = causal ? n_tiles + 1 : 2 * n_tiles;
    return mean_kv2 <= 2 * kDkdvPersistMaxKv ? persistent_grid(n_tiles * BH, mean_kv2, n_sm)
                                             : n_tiles * BH;
}

// Grid of the forward: one item per pair of query tiles (2p, 2p+1), which sees
// min(2p+2, n_tiles) key tiles under the causal mask (mean about n_tiles/2 + 1) and every key
// tile otherwise.
__host__ __device__ __forceinline__ int fwd_grid(int n_pairs, int n_tiles, int BH, bool causal,
                                                 int n_sm) {
    return persistent_grid(n_pairs * BH, causal ? n_tiles + 2 : 2 * n_tiles, n_sm);
}

}  // namespace fa

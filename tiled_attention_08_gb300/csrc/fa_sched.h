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

// Grid of the dQ pass.  Persistent (one CTA per SM) when query tiles see at most kPersistMaxKv
// key tiles on average and there are more tiles than SMs; otherwise one CTA per tile.  The
// fixed cost of a CTA is worth hiding only for short rows; for long rows the hardware's own
// block scheduling balances the causal tiles better than fixed rounds.
constexpr int kPersistMaxKv = 32;
__host__ __device__ __forceinline__ int dq_grid(int n_tiles, int BH, bool causal, int n_sm) {
    const int total = n_tiles * BH;
    const int mean_kv2 = causal ? n_tiles + 1 : 2 * n_tiles;  // twice the mean
    return (n_sm > 0 && n_sm < total && mean_kv2 <= 2 * kPersistMaxKv) ? n_sm : total;
}

}  // namespace fa

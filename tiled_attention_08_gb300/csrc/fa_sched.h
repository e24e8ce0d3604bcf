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

}  // namespace fa

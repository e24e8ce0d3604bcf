// Host-side check of the kernels' tile schedule (tile_coords): every (head, tile) is visited
// exactly once, and inside each head group the tiles come heaviest first; of the persistent
// round order (persistent_tile): every tile id taken exactly once; and of the grid rules of the
// dQ pass, the dK/dV pass and the forward (dq_grid, dkdv_grid, fwd_grid).
#include <cstdio>
#include <vector>

#include "fa_internal.h"
#include "fa_sched.h"

int main() {
    const int cases[][3] = {{1, 1, 1}, {1, 16, 1}, {32, 16, 32}, {256, 32, 24}, {256, 32, 32},
                            {16, 128, 6}, {512, 8, 96}, {7, 5, 3}, {3, 9, 7}, {64, 1, 5}};
    int failures = 0;
    for (const auto& c : cases) {
        const int BH = c[0], T = c[1], G = c[2];
        std::vector<int> seen(BH * T, 0);
        int prev_group = -1, prev_rank = -1;
        for (int tid = 0; tid < BH * T; ++tid) {
            int bh = -1, rank = -1;
            fa::tile_coords(tid, BH, T, G, bh, rank);
            if (bh < 0 || bh >= BH || rank < 0 || rank >= T) {
                std::printf("FAIL out of range BH=%d T=%d G=%d tid=%d -> (%d,%d)\n", BH, T, G, tid,
                            bh, rank);
                ++failures;
                continue;
            }
            ++seen[bh * T + rank];
            const int group = bh / G;
            if (group == prev_group && rank < prev_rank) {
                std::printf("FAIL order BH=%d T=%d G=%d tid=%d\n", BH, T, G, tid);
                ++failures;
            }
            if (group < prev_group) {
                std::printf("FAIL group order BH=%d T=%d G=%d tid=%d\n", BH, T, G, tid);
                ++failures;
            }
            prev_group = group;
            prev_rank = rank;
        }
        for (int i = 0; i < BH * T; ++i)
            if (seen[i] != 1) {
                std::printf("FAIL coverage BH=%d T=%d G=%d tile=%d seen=%d\n", BH, T, G, i, seen[i]);
                ++failures;
            }
    }
    // Persistent grids: across all CTAs and rounds every tile id is taken exactly once, a
    // CTA's ids end at its first -1, and no CTA takes more than one tile more than another.
    const int pcases[][2] = {{1, 1}, {5, 5}, {16, 152}, {152, 152}, {153, 152}, {512, 152},
                             {8192, 152}, {1000, 7}, {2048, 152}, {999, 152}};
    for (const auto& c : pcases) {
        const int total = c[0];
        const int grid = total < c[1] ? total : c[1];
        std::vector<int> seen(total, 0);
        int most = 0, least = total + 1;
        for (int cta = 0; cta < grid; ++cta) {
            int mine = 0;
            bool ended = false;
            for (int round = 0; round * grid < total + grid; ++round) {
                const int id = fa::persistent_tile(round, cta, grid, total);
                if (id < 0) {
                    ended = true;
                    continue;
                }
                if (ended || id >= total) {
                    std::printf("FAIL persistent order total=%d grid=%d cta=%d round=%d\n", total,
                                grid, cta, round);
                    ++failures;
                    continue;
                }
                ++seen[id];
                ++mine;
            }
            most = mine > most ? mine : most;
            least = mine < least ? mine : least;
        }
        for (int i = 0; i < total; ++i)
            if (seen[i] != 1) {
                std::printf("FAIL persistent coverage total=%d grid=%d id=%d seen=%d\n", total,
                            grid, i, seen[i]);
                ++failures;
            }
        if (most - least > 1) {
            std::printf("FAIL persistent balance total=%d grid=%d (%d..%d tiles)\n", total, grid,
                        least, most);
            ++failures;
        }
    }
    // The dQ pass's grid: persistent (152 CTAs) for short rows with more tiles than SMs, one
    // CTA per tile otherwise.  {n_tiles, BH, causal, n_sm, expected}
    const int gcases[][5] = {{32, 256, 1, 152, 152},    // B8 H32 L4096 causal: mean 16.5
                             {16, 32, 1, 152, 152},     // B1 H32 L2048 causal: mean 8.5
                             {128, 16, 1, 152, 2048},   // B1 H16 L16384 causal: mean 64.5
                             {4, 512, 0, 152, 152},     // B16 H32 L512: mean 4
                             {32, 64, 0, 152, 152},     // non-causal L4096: mean 32 (limit)
                             {33, 64, 0, 152, 2112},    // non-causal, mean 33
                             {63, 64, 1, 152, 152},     // causal, mean 32
                             {64, 64, 1, 152, 4096},    // causal, mean 32.5
                             {1, 1, 0, 152, 1},         // fewer tiles than SMs
                             {32, 256, 1, 0, 8192}};    // SM count unknown
    for (const auto& c : gcases) {
        const int got = fa::dq_grid(c[0], c[1], c[2] != 0, c[3]);
        if (got != c[4]) {
            std::printf("FAIL dq_grid(%d,%d,%d,%d) = %d, want %d\n", c[0], c[1], c[2], c[3], got,
                        c[4]);
            ++failures;
        }
    }
    // The dK/dV pass: persistent only up to a mean of 12 query tiles per key tile.
    const int kcases[][5] = {{32, 256, 1, 152, 8192},   // B8 H32 L4096 causal: mean 16.5
                             {16, 32, 1, 152, 152},     // B1 H32 L2048 causal: mean 8.5
                             {128, 16, 1, 152, 2048},   // B1 H16 L16384 causal: mean 64.5
                             {4, 512, 0, 152, 152},     // B16 H32 L512: mean 4
                             {8, 512, 0, 152, 152},     // B16 H32 L1024: mean 8
                             {12, 64, 0, 152, 152},     // non-causal, mean 12 (limit)
                             {13, 64, 0, 152, 832},     // non-causal, mean 13
                             {23, 64, 1, 152, 152},     // causal, mean 12
                             {24, 64, 1, 152, 1536},    // causal, mean 12.5
                             {1, 1, 0, 152, 1},         // fewer tiles than SMs
                             {4, 512, 0, 0, 2048}};     // SM count unknown
    for (const auto& c : kcases) {
        const int got = fa::dkdv_grid(c[0], c[1], c[2] != 0, c[3]);
        if (got != c[4]) {
            std::printf("FAIL dkdv_grid(%d,%d,%d,%d) = %d, want %d\n", c[0], c[1], c[2], c[3], got,
                        c[4]);
            ++failures;
        }
    }
    // The forward's grid over query-tile pairs: {n_pairs, n_tiles, BH, causal, n_sm, expected}.
    const int fcases[][6] = {{16, 32, 256, 1, 152, 152},    // B8 H32 L4096 causal: mean 17
                             {8, 16, 32, 1, 152, 152},      // B1 H32 L2048 causal: mean 9
                             {64, 128, 16, 1, 152, 1024},   // B1 H16 L16384 causal: mean 65
                             {2, 4, 512, 0, 152, 152},      // B16 H32 L512: mean 4
                             {16, 32, 64, 0, 152, 152},     // non-causal L4096: mean 32 (limit)
                             {17, 33, 64, 0, 152, 1088},    // non-causal, mean 33
                             {31, 62, 64, 1, 152, 152},     // causal, mean 32
                             {32, 63, 64, 1, 152, 2048},    // causal, mean 32.5
                             {1, 1, 1, 0, 152, 1},          // fewer pairs than SMs
                             {16, 32, 256, 1, 0, 4096}};    // SM count unknown
    for (const auto& c : fcases) {
        const int got = fa::fwd_grid(c[0], c[1], c[2], c[3] != 0, c[4]);
        if (got != c[5]) {
            std::printf("FAIL fwd_grid(%d,%d,%d,%d,%d) = %d, want %d\n", c[0], c[1], c[2], c[3],
                        c[4], got, c[5]);
            ++failures;
        }
    }
    std::printf(failures ? "FAILED %d\n" : "OK\n", failures);
    return failures ? 1 : 0;
}

// Host-side check of the kernels' tile schedule (tile_coords): every (head, tile) is visited
// exactly once, and inside each head group the tiles come heaviest first; and of the persistent
// round order (persistent_tile): every tile id taken exactly once.
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
    std::printf(failures ? "FAILED %d\n" : "OK\n", failures);
    return failures ? 1 : 0;
}

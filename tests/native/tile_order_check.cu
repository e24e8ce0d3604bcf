// Host-side check of the kernels' tile schedule (tile_coords): every (head, tile) is visited
// exactly once, and inside each head group the tiles come heaviest first.
#include <cstdio>
#include <vector>

#include "fa_internal.h"

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
    std::printf(failures ? "FAILED %d\n" : "OK\n", failures);
    return failures ? 1 : 0;
}

// Host-side check of the kernels' tile schedule (tile_coords): every (head, tile) is visited
// exactly once, and inside each head group the tiles come heaviest first; of the persistent
// round order (persistent_tile): every tile id taken exactly once; of the tile bounds under the
// causal mask with Lq != Lk (q_tile_kv, k_tile_q0, tile_masked) against the per-element
// definition; and of the grid rules of the dQ pass, the dK/dV pass and the forward.
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
    // Tile bounds under the causal mask against the per-element definition (query row i sees key
    // j iff j <= i + Lk - Lq), on square and rectangular shapes with ragged tails.
    const int shapes[][2] = {{1, 1},     {128, 128}, {129, 129}, {300, 300}, {384, 1000},
                             {1000, 384}, {5, 700},   {700, 5},   {256, 128}, {128, 256},
                             {200, 77},  {77, 200},  {513, 129}, {129, 513}};
    for (const auto& sh : shapes) {
        const int Lq = sh[0], Lk = sh[1];
        const int n_q = (Lq + 127) / 128, n_k = (Lk + 127) / 128;
        for (int causal = 0; causal < 2; ++causal) {
            for (int qt = 0; qt < n_q; ++qt) {
                int want_kv = 0;  // key tiles holding a key some row of the tile sees
                for (int kt = 0; kt < n_k; ++kt) {
                    bool seen = false, all = true;
                    for (int i = qt * 128; i < qt * 128 + 128; ++i)
                        for (int j = kt * 128; j < kt * 128 + 128; ++j) {
                            const bool vis = i < Lq && j < Lk && (!causal || j <= i + Lk - Lq);
                            seen = seen || vis;
                            all = all && vis;
                        }
                    if (seen) want_kv = kt + 1;
                    if (seen && fa::tile_masked(qt, kt, Lq, Lk, causal != 0) == all) {
                        std::printf("FAIL tile_masked(%d,%d,%d,%d,%d)\n", qt, kt, Lq, Lk, causal);
                        ++failures;
                    }
                    const bool q0_says = qt >= fa::k_tile_q0(kt, Lq, Lk, causal != 0);
                    if (kt * 128 < Lk && seen != q0_says) {
                        std::printf("FAIL k_tile_q0(%d,%d,%d,%d) vs qt=%d\n", kt, Lq, Lk, causal,
                                    qt);
                        ++failures;
                    }
                }
                if (fa::q_tile_kv(qt, Lq, Lk, causal != 0) != want_kv) {
                    std::printf("FAIL q_tile_kv(%d,%d,%d,%d) = %d, want %d\n", qt, Lq, Lk, causal,
                                fa::q_tile_kv(qt, Lq, Lk, causal != 0), want_kv);
                    ++failures;
                }
            }
        }
    }
    // The dQ pass's grid: persistent (152 CTAs) for short rows with more tiles than SMs, one
    // CTA per tile otherwise.  {Lq, Lk, BH, causal, n_sm, expected}
    const int gcases[][6] = {{4096, 4096, 256, 1, 152, 152},    // B8 H32 L4096 causal: mean 16.5
                             {2048, 2048, 32, 1, 152, 152},     // B1 H32 L2048 causal: mean 8.5
                             {16384, 16384, 16, 1, 152, 2048},  // B1 H16 L16384 causal: mean 64.5
                             {512, 512, 512, 0, 152, 152},      // B16 H32 L512: mean 4
                             {4096, 4096, 64, 0, 152, 152},     // non-causal L4096: mean 32 (limit)
                             {4224, 4224, 64, 0, 152, 2112},    // non-causal, mean 33
                             {8064, 8064, 64, 1, 152, 152},     // causal, mean 32
                             {8192, 8192, 64, 1, 152, 4096},    // causal, mean 32.5
                             {128, 128, 1, 0, 152, 1},          // fewer tiles than SMs
                             {4096, 4096, 256, 1, 0, 8192},     // SM count unknown
                             {512, 8192, 64, 1, 152, 256},      // 512 queries after 7680 keys: 62.5
                             {1024, 640, 256, 1, 152, 152}};    // Lq > Lk: 3 tiles see no key
    for (int i = 0; i < (int)(sizeof(gcases) / sizeof(gcases[0])); ++i) {
        const auto& c = gcases[i];
        const int got = fa::dq_grid(c[0], c[1], c[2], c[3] != 0, c[4]);
        if (got != c[5]) {
            std::printf("FAIL dq_grid(%d,%d,%d,%d,%d) = %d, want %d\n", c[0], c[1], c[2], c[3],
                        c[4], got, c[5]);
            ++failures;
        }
    }
    // The dK/dV pass: persistent only up to a mean of 32 query tiles per key tile.
    const int kcases[][6] = {{4096, 4096, 256, 1, 152, 152},    // B8 H32 L4096 causal: mean 16.5
                             {2048, 2048, 32, 1, 152, 152},     // B1 H32 L2048 causal: mean 8.5
                             {16384, 16384, 16, 1, 152, 2048},  // B1 H16 L16384 causal: mean 64.5
                             {512, 512, 512, 0, 152, 152},      // B16 H32 L512: mean 4
                             {1024, 1024, 512, 0, 152, 152},    // B16 H32 L1024: mean 8
                             {4096, 4096, 64, 0, 152, 152},     // non-causal, mean 32 (limit)
                             {4224, 4224, 64, 0, 152, 2112},    // non-causal, mean 33
                             {8064, 8064, 64, 1, 152, 152},     // causal, mean 32
                             {8192, 8192, 64, 1, 152, 4096},    // causal, mean 32.5
                             {128, 128, 1, 0, 152, 1},          // fewer tiles than SMs
                             {512, 512, 512, 0, 0, 2048}};      // SM count unknown
    for (const auto& c : kcases) {
        const int got = fa::dkdv_grid(c[0], c[1], c[2], c[3] != 0, c[4]);
        if (got != c[5]) {
            std::printf("FAIL dkdv_grid(%d,%d,%d,%d,%d) = %d, want %d\n", c[0], c[1], c[2], c[3],
                        c[4], got, c[5]);
            ++failures;
        }
    }
    // The forward's grid over query-tile pairs.
    const int fcases[][6] = {{4096, 4096, 256, 1, 152, 152},    // B8 H32 L4096 causal: mean 17
                             {2048, 2048, 32, 1, 152, 152},     // B1 H32 L2048 causal: mean 9
                             {16384, 16384, 16, 1, 152, 1024},  // B1 H16 L16384 causal: mean 65
                             {512, 512, 512, 0, 152, 152},      // B16 H32 L512: mean 4
                             {4096, 4096, 64, 0, 152, 152},     // non-causal L4096: mean 32 (limit)
                             {4224, 4224, 64, 0, 152, 1088},    // non-causal, mean 33
                             {7936, 7936, 64, 1, 152, 152},     // causal, 62 tiles: mean 32
                             {8064, 8064, 64, 1, 152, 2048},    // causal, 63 tiles: mean 33
                             {128, 128, 1, 0, 152, 1},          // fewer pairs than SMs
                             {4096, 4096, 256, 1, 0, 4096}};    // SM count unknown
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

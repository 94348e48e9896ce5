// Host check of the key-stationary backward's CTA order (grouped_tile_order):
// for every size given, the linear block indices 0 .. BH * n_tiles - 1 visit each
// (head, key tile) pair exactly once, heads of one group before the next group,
// and inside a group the tile index never decreases (heaviest tiles first).
// Usage: tile_order_check BH n_tiles group [BH n_tiles group ...]; with no
// arguments it sweeps small sizes and every group from 1 to BH.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "common.cuh"

static bool check(int64_t BH, int n_tiles, int group) {
    std::vector<unsigned char> seen((size_t)BH * n_tiles, 0);
    int prev_group = -1, prev_tile = -1;
    for (int64_t idx = 0; idx < BH * n_tiles; ++idx) {
        int bh = -1, tile = -1;
        relation::grouped_tile_order((unsigned)idx, BH, n_tiles, group, bh, tile);
        if (bh < 0 || bh >= BH || tile < 0 || tile >= n_tiles) {
            std::printf("out of range: BH=%lld n_tiles=%d group=%d idx=%lld -> bh=%d tile=%d\n", (long long)BH,
                        n_tiles, group, (long long)idx, bh, tile);
            return false;
        }
        unsigned char& s = seen[(size_t)bh * n_tiles + tile];
        if (s) {
            std::printf("visited twice: BH=%lld n_tiles=%d group=%d bh=%d tile=%d\n", (long long)BH, n_tiles, group,
                        bh, tile);
            return false;
        }
        s = 1;
        const int g = bh / group;
        if (g < prev_group || (g == prev_group && tile < prev_tile)) {
            std::printf("order: BH=%lld n_tiles=%d group=%d idx=%lld (group %d tile %d after group %d tile %d)\n",
                        (long long)BH, n_tiles, group, (long long)idx, g, tile, prev_group, prev_tile);
            return false;
        }
        if (g != prev_group) prev_tile = -1;
        prev_group = g;
        prev_tile = tile;
    }
    return true;  // BH * n_tiles distinct in-range pairs: every pair once
}

int main(int argc, char** argv) {
    long cases = 0;
    if (argc > 1) {
        if ((argc - 1) % 3 != 0) return 2;
        for (int a = 1; a + 2 < argc; a += 3) {
            if (!check(std::atoll(argv[a]), std::atoi(argv[a + 1]), std::atoi(argv[a + 2]))) return 1;
            ++cases;
        }
    } else {
        for (int BH = 1; BH <= 40; ++BH)
            for (int n_tiles = 1; n_tiles <= 12; ++n_tiles)
                for (int group = 1; group <= BH; ++group, ++cases)
                    if (!check(BH, n_tiles, group)) return 1;
    }
    std::printf("ok %ld\n", cases);
    return 0;
}

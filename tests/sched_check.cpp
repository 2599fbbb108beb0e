// Host-side brute-force check of the scheduling arithmetic in tile_schedule.h
// (compiled and run by test_host_logic.py with the system C++ compiler).
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "tile_schedule.h"

static int fail(const char* what, long long a, long long b, long long c) {
    std::printf("FAIL %s %lld %lld %lld\n", what, a, b, c);
    return 1;
}

int main() {
    // tile_coord is a bijection onto [0, tiles_m) x [0, tiles_n)
    const int shapes[][3] = {{1, 1, 16}, {64, 112, 16}, {3, 7, 16}, {17, 5, 16}, {33, 9, 8},
                             {16, 16, 16}, {5, 100, 4}, {100, 3, 1}};
    for (auto& s : shapes) {
        const int tm = s[0], tn = s[1], g = s[2] < tm ? s[2] : tm;
        std::vector<int> seen(static_cast<size_t>(tm) * tn, 0);
        for (int t = 0; t < tm * tn; ++t) {
            tg::TileCoord c = tg::tile_coord(t, tm, tn, g);
            if (c.m_blk < 0 || c.m_blk >= tm || c.n_blk < 0 || c.n_blk >= tn)
                return fail("tile_coord range", t, c.m_blk, c.n_blk);
            if (seen[static_cast<size_t>(c.m_blk) * tn + c.n_blk]++)
                return fail("tile_coord duplicate", t, c.m_blk, c.n_blk);
        }
    }
    // unit ranges tile [0, U) and unit_owner inverts unit_begin
    for (long long U = 1; U <= 400; ++U) {
        for (long long G = 1; G <= U && G <= 160; ++G) {
            if (tg::unit_begin(0, G, U) != 0 || tg::unit_begin(G, G, U) != U)
                return fail("unit_begin ends", U, G, 0);
            for (long long c = 0; c < G; ++c) {
                const long long b = tg::unit_begin(c, G, U), e = tg::unit_begin(c + 1, G, U);
                if (e - b < U / G || e - b > U / G + 1) return fail("unit range length", U, G, c);
                for (long long u = b; u < e; ++u)
                    if (tg::unit_owner(u, G, U) != c) return fail("unit_owner", U, G, u);
            }
        }
    }
    // large sizes without overflow (skinny workload: 128 tiles x 128 k-blocks over 152 CTAs)
    {
        const long long U = 128LL * 128, G = 152;
        for (long long c = 0; c < G; ++c)
            for (long long u = tg::unit_begin(c, G, U); u < tg::unit_begin(c + 1, G, U); ++u)
                if (tg::unit_owner(u, G, U) != c) return fail("unit_owner big", U, G, u);
        const long long U2 = 16777215LL * 33554431LL, G2 = 152;
        if (tg::unit_begin(G2, G2, U2) != U2) return fail("unit_begin overflow", U2, G2, 0);
        if (tg::unit_owner(U2 - 1, G2, U2) != G2 - 1) return fail("unit_owner overflow", U2, G2, 0);
    }
    std::printf("OK\n");
    return 0;
}

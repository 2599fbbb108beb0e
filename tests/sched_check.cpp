// Host-side brute-force check of the scheduling arithmetic in tile_schedule.h
// and of the 2:4 kernel choice in sparse_plan.h (compiled and run by
// test_abi.py with the system C++ compiler).
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "sparse_plan.h"
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
    // pair work items: every (tile, column half, k block) exactly once; cuts
    // only in the last wave; either at most kPairMaxSplit k-pieces, each at
    // least kPairMinPieceBlocks long, or two column halves over all of k;
    // R·S·H <= P and P <= pairs; KB = 0 rules out k-pieces
    for (int T = 1; T <= 700; T += (T < 160 ? 1 : 37)) {
        for (int pairs : {1, 2, 7, 38, 74, 76}) {
            for (int KB : {0, 1, 7, 8, 16, 32, 33, 64, 65, 96, 97, 128}) {
                int P = 0, S = 0, H = 0;
                tg::pair_launch_shape(T, pairs, KB, &P, &S, &H);
                if (P < 1 || P > pairs || S < 1 || S > tg::kPairMaxSplit || H < 1 || H > 2)
                    return fail("pair_launch_shape range", T, pairs, KB);
                if (S > 1 && H > 1) return fail("pair both cuts", T, pairs, KB);
                if (S > 1 && KB / S < tg::kPairMinPieceBlocks)
                    return fail("pair piece length", T, pairs, KB);
                const int W = T / P, R = T - W * P;
                if (R * S * H > P) return fail("pair tail items", T, P, S * H);
                if (KB == 0) continue;
                std::vector<int> seen(static_cast<size_t>(T) * 2 * KB, 0);
                for (int c = 0; c < P; ++c) {
                    const int n = tg::pair_item_count(c, T, P, S, H);
                    for (int i = 0; i < n; ++i) {
                        int tile = -1, kb0 = -1, kb1 = -1, half = -2;
                        tg::pair_item(c, i, T, P, S, H, KB, &tile, &kb0, &kb1, &half);
                        if (tile < 0 || tile >= T || kb0 < 0 || kb1 > KB || kb0 >= kb1 ||
                            half < -1 || half > 1)
                            return fail("pair_item range", T, c, i);
                        if ((kb0 != 0 || kb1 != KB || half >= 0) && tile < W * P)
                            return fail("pair cut outside the last wave", T, c, i);
                        if (half >= 0 && (kb0 != 0 || kb1 != KB))
                            return fail("pair half with a k range", T, c, i);
                        for (int h = 0; h < 2; ++h) {
                            if (half >= 0 && h != half) continue;
                            for (int kb = kb0; kb < kb1; ++kb)
                                if (seen[(static_cast<size_t>(tile) * 2 + h) * KB + kb]++)
                                    return fail("pair_item duplicate", T, tile, kb);
                        }
                    }
                }
                for (size_t u = 0; u < seen.size(); ++u)
                    if (seen[u] != 1) return fail("pair_item missing", T, P, static_cast<long long>(u));
            }
        }
    }
    // the choice between the two cuts: column halves on the 4096^3 shape and
    // the 8192x28672x4096 MLP shape (76 pairs), k-pieces once K is long
    {
        int P, S, H;
        tg::pair_launch_shape(256, 76, 32, &P, &S, &H);
        if (P != 76 || S != 1 || H != 2) return fail("4096^3 tail", P, S, H);
        tg::pair_launch_shape(3584, 76, 32, &P, &S, &H);
        if (P != 76 || S != 1 || H != 2) return fail("MLP tail", P, S, H);
        tg::pair_launch_shape(4, 76, 128, &P, &S, &H);
        if (P != 16 || S != 4 || H != 1) return fail("long-k tail", P, S, H);
        tg::pair_launch_shape(80, 76, 32, &P, &S, &H);  // 4 tail tiles, k too short to pay
        if (P != 76 || S != 1 || H != 2) return fail("short-k tail", P, S, H);
        tg::pair_launch_shape(256, 76, 128, &P, &S, &H);  // 4096x4096x16384
        if (P != 76 || S != 2 || H != 1) return fail("long-k two pieces", P, S, H);
    }
    // the 2:4 kernel choice on 152 SMs with 76 resident pairs, at the shapes
    // it was measured on (1: CTA pairs)
    const long long sp[][4] = {{8192, 28672, 4096, 1}, {2048, 2048, 4096, 1}, {2048, 2048, 1024, 1},
                               {512, 512, 8192, 1},    {1024, 1024, 4096, 1}, {256, 2048, 4096, 1},
                               {256, 256, 16384, 1},   {1024, 2048, 2048, 1}, {1024, 1024, 2048, 0},
                               {1024, 1024, 1024, 0},  {2048, 1024, 512, 0},  {512, 512, 512, 0},
                               {128, 4096, 8192, 0},   {96, 160, 192, 0}};
    for (auto& c : sp) {
        const bool pair = tg::sp24_use_pairs(c[0], c[1], c[2], 76, 152);
        if (pair != (c[3] == 1)) return fail("sp24 kernel choice", c[0], c[1], c[2]);
    }
    if (tg::sp24_use_pairs(8192, 28672, 4096, 0, 152)) return fail("sp24 no pairs", 0, 0, 0);
    std::printf("OK\n");
    return 0;
}

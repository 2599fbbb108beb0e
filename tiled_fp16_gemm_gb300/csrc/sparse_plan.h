// Which 2:4 sparse kernel runs a problem: the host planner's rule, in a header
// of its own so that host tests compile it.
#pragma once

#include <cstdint>

namespace tg {

// The CTA-pair kernel (256×256 tiles) runs once its tiles fill every resident
// pair at least once, and also below that when K ≥ 1024 and one-CTA tiles
// would occupy more than half the SMs (measured on GB300: 2048×2048×4096 22.7
// µs against 37.8 µs, 1536×1536×4096 20.8 against 22.7 µs, 2048×2048×1024 12.4
// against 14.5 µs; a tie at K = 512), and for K ≥ 4096 with M > 128 whatever
// the tile count: per k block a pair moves a 256×256 tile in less time than a
// one-CTA kernel moves a 128×128 one (512×512×8192 28.2 against 32.3 µs,
// 1024×1024×4096 17.0 against 17.9 µs).  Smaller problems take the one-CTA
// kernel (128×128 tiles, four times the tiles in flight: 1024³ 7.1 against
// 8.4 µs, 2048×1024×512 5.5 against 7.0 µs).  max_pairs: the CTA pairs of the
// pair kernel that fit on the device at once (0: none).
inline bool sp24_use_pairs(int64_t M, int64_t N, int64_t K, int32_t max_pairs, int32_t num_sms) {
    if (max_pairs < 1) return false;
    const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
    const int64_t cta_tiles = ((M + 127) / 128) * ((N + 127) / 128);
    return pair_tiles >= max_pairs || (K >= 1024 && 2 * cta_tiles > num_sms) ||
           (K >= 4096 && M > 128);
}

}  // namespace tg

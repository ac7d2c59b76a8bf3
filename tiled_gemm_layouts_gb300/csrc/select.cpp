// select.cpp -- deterministic per-shape tile / stage selector.
//
// The policy is a fixed scoring rule, not an autotuner (the same stance as
// the deterministic dot thread-shape policy of pbelevich.github.io "My Triton
// From Scratch Part 16: Register Tiles", section "Choosing the physical thread
// shape"); tile sizes stay a property of the chosen layout (ninetoothed.org
// "Named layouts", section "Contract").
#include "select.h"

#include <cstdio>
#include <cstdlib>
#include <cstring>

namespace tg {

namespace {

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Relative MMA-pipe efficiency of a 128 x bn tile: narrower tiles re-read the
// 128-row operand from shared memory more often per flop.
double tile_efficiency(int bn) {
    switch (bn) {
        case 256: return 1.0;
        case 128: return 0.92;
        case 64: return 0.75;
        default: return 0.55;
    }
}

void apply_override(KernelConfig& c) {
    const char* env = std::getenv("TG_FORCE_CONFIG");
    if (!env || !*env) return;
    char buf[256];
    std::snprintf(buf, sizeof(buf), "%s", env);
    for (char* tok = std::strtok(buf, ", "); tok; tok = std::strtok(nullptr, ", ")) {
        int v = 0;
        if (std::sscanf(tok, "bn=%d", &v) == 1 && (v == 32 || v == 64 || v == 128 || v == 256))
            c.bn = v;
        else if (std::sscanf(tok, "swap=%d", &v) == 1 && (v == 0 || v == 1))
            c.swap = v;
        else if (std::sscanf(tok, "group_m=%d", &v) == 1 && v >= 1 && v <= 64)
            c.group_m = v;
        else if (std::sscanf(tok, "grid=%d", &v) == 1 && v >= 1)
            c.grid = v;
    }
}

}  // namespace

KernelConfig select_config(int64_t M, int64_t N, int64_t K, int /*dtype*/, int permA, int permB,
                           bool /*has_epilogue*/, int sms) {
    KernelConfig c{};
    // Operand swap: when M cannot fill the 128 accumulator lanes but N can,
    // compute C^T = B^T A^T so that N runs along the lanes.
    c.swap = (M <= 64 && N > M) ? 1 : 0;
    c.bm = 128;
    c.pair = 0;
    c.group_m = 8;
    c.grid = 0;
    apply_override(c);
    const int forced_bn = c.bn;

    const int64_t Mk = c.swap ? N : M, Nk = c.swap ? M : N;
    // Q (the kernel's column operand) is MN-major when its storage runs along
    // the kernel's columns; such tiles are fetched in 64-column swizzle atoms.
    const bool q_mn = c.swap ? (permA == 1) : (permB == 0);
    if (!forced_bn) {
        double best = -1.0;
        for (int bn : {256, 128, 64, 32}) {
            if (bn == 32 && q_mn) continue;
            const int64_t tiles = cdiv(Mk, 128) * cdiv(Nk, bn);
            const int64_t waves = cdiv(tiles, sms);
            const double util = (double)Mk * (double)Nk / ((double)waves * sms * 128.0 * bn);
            const double score = util * tile_efficiency(bn);
            if (score > best + 1e-9) {
                best = score;
                c.bn = bn;
            }
        }
    } else if (forced_bn == 32 && q_mn) {
        c.bn = 64;
    }
    const int64_t tiles_m = cdiv(Mk, 128);
    const int64_t tiles = tiles_m * cdiv(Nk, c.bn);
    c.tiles = (int)tiles;
    if (c.group_m > tiles_m) c.group_m = (int)tiles_m;
    if (c.grid <= 0 || c.grid > sms) c.grid = sms;
    if (c.grid > tiles) c.grid = (int)tiles;
    c.stages = gemm_stages(c.bn);
    (void)K;
    return c;
}

std::string describe_config(const KernelConfig& c) {
    char buf[256];
    std::snprintf(buf, sizeof(buf),
                  "swap=%d bm=%d bn=%d pair=%d stages=%d group_m=%d grid=%d tiles=%d", c.swap,
                  c.bm, c.bn, c.pair, c.stages, c.group_m, c.grid, c.tiles);
    return buf;
}

}  // namespace tg

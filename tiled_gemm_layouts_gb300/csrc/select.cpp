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

// Relative tensor-pipe efficiency of a tile in steady state, indexed by the
// B columns it stages.  A single-CTA 128 x BN tile stages 16 KB of A and
// BN*128 bytes of B per 64-deep K block and the tensor core reads the same
// bytes back, so narrower tiles move more shared-memory bytes per flop and
// stall on shared-memory bandwidth; a CTA pair (256 x BN on two SMs) halves
// the B bytes each SM stages.  Calibrated on GB300 sweeps of this kernel over
// every compiled tile at 4096^3 and 8192 x 8192 x 4096 (fp16, row-major).
double tile_efficiency(int cols, int pair) {
    if (pair) {
        if (cols >= 256) return 0.88;
        if (cols >= 224) return 0.83;
        if (cols >= 192) return 0.75;
        if (cols >= 128) return 0.49;
        return 0.3;
    }
    if (cols >= 256) return 0.79;
    if (cols >= 224) return 0.74;
    if (cols >= 192) return 0.675;
    if (cols >= 128) return 0.49;
    if (cols >= 64) return 0.26;
    return 0.15;
}

// B columns a tile actually stages: MN-major B arrives in whole 64-column
// swizzle atoms per CTA.
int staged_columns(int bn, int pair, bool q_mn) {
    if (!q_mn) return bn;
    const int per_cta = pair ? bn / 2 : bn;
    return ((per_cta + 63) / 64) * 64 * (pair ? 2 : 1);
}

struct Choice {
    int swap, pair, bn;
    double score;
};

void apply_override(KernelConfig& c, bool& forced_bn, bool& forced_pair, bool& forced_swap,
                    bool& forced_no_sk, bool& forced_sk, bool& forced_group) {
    const char* env = std::getenv("TG_FORCE_CONFIG");
    if (!env || !*env) return;
    // Tokens are split by hand (no strtok: this runs on every call, possibly
    // from several host threads at once).
    std::string spec(env);
    for (size_t i = 0; i < spec.size();) {
        const size_t j = spec.find_first_of(", ", i);
        const std::string word = spec.substr(i, j == std::string::npos ? std::string::npos : j - i);
        i = j == std::string::npos ? spec.size() : j + 1;
        if (word.empty()) continue;
        const char* tok = word.c_str();
        int v = 0;
        if (std::sscanf(tok, "bn=%d", &v) == 1 && gemm_stages(v, 0) > 0) {
            c.bn = v;
            forced_bn = true;
        } else if (std::sscanf(tok, "swap=%d", &v) == 1 && (v == 0 || v == 1)) {
            c.swap = v;
            forced_swap = true;
        } else if (std::sscanf(tok, "pair=%d", &v) == 1 && (v == 0 || v == 1)) {
            c.pair = v;
            forced_pair = true;
        } else if (std::sscanf(tok, "group_m=%d", &v) == 1 && v >= 1 && v <= 64) {
            c.group_m = v;
            forced_group = true;
        } else if (std::sscanf(tok, "grid=%d", &v) == 1 && v >= 1) {
            c.grid = v;
        } else if (std::sscanf(tok, "sk=%d", &v) == 1 && (v == 0 || v == 1)) {
            forced_no_sk = v == 0;
            forced_sk = v == 1;
        }
    }
}

}  // namespace

// Waves a tile count costs on `slots` workers: whole waves when every tile is
// computed by one worker; with stream-K the tiles of the last waves are
// shared out in equal K-ranges, at a small price for the partial sums.
double effective_waves(int64_t tiles, int slots, bool allow_sk) {
    const double whole = (double)cdiv(tiles, slots);
    if (!allow_sk) return whole;
    const double fill = (double)tiles / (whole * slots);
    if (tiles <= slots || fill >= 0.9) return whole;
    return (double)tiles / slots + 0.25;
}

KernelConfig select_config(int64_t M, int64_t N, int64_t K, int /*dtype*/, int permA, int permB,
                           bool /*has_epilogue*/, int sms, bool allow_sk) {
    KernelConfig c{};
    // Tiles run in groups of group_m tile rows, column after column, so the
    // 76 concurrent 256-row tiles share few B panels; 16 measured 1.6 % over
    // 8 at 8192 x 8192 x 4096 (less B re-read from DRAM) and 0.6 % at 4096^3.
    c.group_m = 16;
    bool forced_bn = false, forced_pair = false, forced_swap = false, forced_no_sk = false,
         forced_sk = false, forced_group = false;
    apply_override(c, forced_bn, forced_pair, forced_swap, forced_no_sk, forced_sk, forced_group);

    // Stream-K only deals out tails of tiles at least 32 K-blocks deep (see
    // below), so only then may the wave estimate count on it.
    const bool sk_possible = allow_sk && (K + 63) / 64 >= 32;
    const bool shallow = (K + 63) / 64 < 32;
    Choice best{0, 0, 0, -1.0};
    for (int swap = 0; swap < 2; ++swap) {
        if (forced_swap && swap != c.swap) continue;
        const int64_t Mk = swap ? N : M, Nk = swap ? M : N;
        // Q (the kernel's column operand) is MN-major when its storage runs
        // along the kernel's columns; such tiles are fetched in 64-column atoms.
        const bool q_mn = swap ? (permA == 1) : (permB == 0);
        for (int pair = 0; pair < 2; ++pair) {
            if (forced_pair && pair != c.pair) continue;
            for (int bn : {256, 224, 192, 128, 64, 32}) {
                if (forced_bn && bn != c.bn) continue;
                if (gemm_stages(bn, pair) <= 0) continue;
                if (bn == 32 && q_mn) continue;  // MN-major atoms are 64 columns wide
                const int bm = pair ? 256 : 128;
                const int slots = pair ? sms / 2 : sms;
                const int64_t tiles = cdiv(Mk, bm) * cdiv(Nk, bn);
                const double waves = effective_waves(tiles, slots, sk_possible);
                const int cols = staged_columns(bn, pair, q_mn);
                double score = (double)Mk * (double)Nk / (waves * slots * bm * cols) *
                               tile_efficiency(cols, pair);
                // A one-tile-wide problem is bandwidth bound: the narrowest tile
                // that covers it streams the other operand once per SM.
                if (Nk <= 32 && bn == 32 && !pair) score = 2.0;
                // Swapping pays only when M cannot fill the 128 accumulator
                // lanes: the transposed output path stores one 2-byte element
                // per lane and measured 12% slower at 4096^3.
                const bool small_m = M <= 64 && N > M;
                if (swap != (small_m ? 1 : 0) && !forced_swap) continue;
                // Equal modelled cost (same waves, same staged columns) with
                // a shallow K, where the ring hides most loads and tensor
                // work sets a tile's time: the narrower tile computes fewer
                // columns (4000 x 3000 x 1000, B row-major: 256 x 224
                // measured 5 % faster than 256 x 256, both three whole
                // waves).  Deep tiles are load-bound: keep the wider one.
                if (score > best.score + 1e-9 ||
                    (shallow && score > best.score - 1e-9 && pair == best.pair && bn < best.bn))
                    best = Choice{swap, pair, bn, score};
            }
        }
    }
    if (best.score < 0) {  // an impossible forced combination: fall back to the plain default
        best = Choice{0, 0, 128, 0.0};
    }
    c.swap = best.swap;
    c.pair = best.pair;
    c.bn = best.bn;
    c.bm = c.pair ? 256 : 128;
    const int64_t Mk = c.swap ? N : M, Nk = c.swap ? M : N;
    const int64_t tiles_m = cdiv(Mk, c.bm);
    const int64_t tiles = tiles_m * cdiv(Nk, c.bn);
    c.tiles = (int)tiles;
    if (c.group_m > tiles_m) c.group_m = (int)tiles_m;
    const int slots = c.pair ? sms / 2 : sms;
    int clusters = c.grid > 0 ? (c.pair ? c.grid / 2 : c.grid) : slots;
    if (clusters > slots) clusters = slots;
    // With few tile columns a group of 16 tile rows holds less than one wave:
    // each wave then spans two groups and its A panels outgrow L2 before the
    // next wave reuses them.  Widen the group to a whole wave of tiles
    // (16384 x 1024 x 8192: 4 columns, groups of 19 rows, measured 4.5 %
    // faster than 16, with 2.4x less A re-read from DRAM).
    const int64_t tiles_n = cdiv(Nk, c.bn);
    if (!forced_group && tiles_n * c.group_m < clusters) c.group_m = (int)cdiv(clusters, tiles_n);
    if (c.group_m > tiles_m) c.group_m = (int)tiles_m;
    c.stages = gemm_stages(c.bn, c.pair);

    // Stream-K for the tail: the last partial wave plus one whole wave are
    // dealt out as equal K-ranges when that beats whole waves.
    c.sk_tiles = 0;
    c.sk_cmax = 0;
    c.ws_bytes = 0;
    const int64_t num_kb = cdiv(K, 64);
    // Measured on GB300: the split pays when whole waves leave at least 10 %
    // of the SM-time idle, every worker also has whole tiles, and tiles are
    // at least 32 K-blocks deep (the partial sums cost about half a tile).
    // A problem with fewer tiles than workers is not split: dealing every
    // tile out over all workers measured slower on GB300 (32 x 16384 x 16384
    // on 152 instead of 128 SMs: 5.05 against 5.31 TB/s; 2048 x 2048 x 4096:
    // 729 against 1049 TFLOP/s) -- every tile then ends in a fix-up, all at
    // the end of the launch.
    const double wave_fill = (double)tiles / ((double)cdiv(tiles, clusters) * clusters);
    const bool want_sk = forced_sk ? tiles % clusters != 0
                                   : (tiles > clusters && wave_fill < 0.9 && num_kb >= 32);
    if (allow_sk && !forced_no_sk && want_sk) {
        const int64_t sk_tiles = tiles > clusters ? clusters + tiles % clusters : tiles;
        const int64_t iters = sk_tiles * num_kb;
        if (iters >= 2 * (int64_t)clusters) {
            const int64_t per = iters / clusters;  // shortest range
            int64_t cmax = (num_kb - 1) / per + 2;
            if (cmax > clusters) cmax = clusters;
            c.sk_tiles = (int)sk_tiles;
            c.sk_cmax = (int)cmax;
            c.ws_bytes = sk_workspace_bytes(clusters, (int)cmax, c.bm, c.bn);
        }
    }
    if (c.sk_tiles == 0 && clusters > tiles) clusters = (int)tiles;
    if (clusters < 1) clusters = 1;
    c.grid = c.pair ? 2 * clusters : clusters;
    return c;
}

long long sk_counter_bytes(int workers) { return ((long long)workers * 2 * 4 + 255) / 256 * 256; }

long long sk_workspace_bytes(int workers, int cmax, int bm, int bn) {
    return sk_counter_bytes(workers) + (long long)workers * cmax * bm * bn * 4;
}

std::string describe_config(const KernelConfig& c) {
    char buf[256];
    std::snprintf(buf, sizeof(buf),
                  "swap=%d bm=%d bn=%d pair=%d stages=%d group_m=%d grid=%d tiles=%d sk_tiles=%d "
                  "sk_cmax=%d ws_bytes=%lld",
                  c.swap, c.bm, c.bn, c.pair, c.stages, c.group_m, c.grid, c.tiles, c.sk_tiles,
                  c.sk_cmax, c.ws_bytes);
    return buf;
}

}  // namespace tg

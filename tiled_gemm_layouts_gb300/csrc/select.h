// select.h -- deterministic per-shape tile / stage selector.
#pragma once

#include <cstdint>
#include <string>

#include "gemm_params.h"

namespace tg {

// Chooses operand swap, tile width, CTA pairing, raster group and grid for a
// problem on a device with `sms` SMs.  Deterministic: the same arguments give
// the same configuration; TG_FORCE_CONFIG (e.g. "bn=128,swap=0,group_m=8")
// overrides single fields for experiments.
// allow_sk: a stream-K workspace is available, so the tail waves may be
// shared out in K-ranges (the config then reports the workspace it needs).
KernelConfig select_config(int64_t M, int64_t N, int64_t K, int dtype, int permA, int permB,
                           bool has_epilogue, int sms, bool allow_sk);

// Workspace bytes of a stream-K split: arrival counters, then the partial
// accumulator slots.
long long sk_workspace_bytes(int workers, int cmax, int bm, int bn);

std::string describe_config(const KernelConfig& c);

}  // namespace tg

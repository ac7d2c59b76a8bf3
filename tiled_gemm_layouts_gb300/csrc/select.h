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

// Bytes of the arrival counters at the start of a split's workspace (two
// ints per worker, rounded up to 256 bytes); they are zero between calls.
long long sk_counter_bytes(int workers);

std::string describe_config(const KernelConfig& c);

// Bytes of stream-K arrival counters that tg_gemm_ws would use at the start
// of its workspace for these arguments on the current device (0 when the
// selector runs whole tiles only).  Status as tg_gemm_workspace_size.
int split_counter_bytes(int64_t M, int64_t N, int64_t K, int dtype, int permA, int permB,
                        bool has_epilogue, size_t* bytes);

}  // namespace tg

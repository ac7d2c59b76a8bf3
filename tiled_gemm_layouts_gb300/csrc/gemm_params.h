// gemm_params.h -- what the host side hands to the tcgen05 GEMM kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace tg {

// Device status word values (the kernel records the first failure it sees).
enum : int {
    DEV_OK = 0,
    DEV_TIMEOUT_PRODUCER = 0x100,   // + which wait
    DEV_TIMEOUT_MMA = 0x200,
    DEV_TIMEOUT_EPILOGUE = 0x300,
};

// The kernel computes D = P * Q over a (Mk x Nk) output in tiles of
// BM x BN, contracting over K in blocks of 64.  Without operand swap P = A,
// Q = B and D = C; with swap P = B^T, Q = A^T and D = C^T (the output is then
// written transposed, so C is still M x N row-major).
struct alignas(128) GemmParams {
    CUtensorMap map_p;   // P operand: K-major box {64, BM} or MN-major box {64, 64}
    CUtensorMap map_q;   // Q operand: K-major box {64, BN} or MN-major box {64, 64}
    CUtensorMap map_c;   // C for tensor stores: box {32 columns, 32 rows}, 64-byte swizzle
    // Two consecutive K-blocks of an operand as one box (valid when p_2k / q_2k):
    // P K-major {64, BM rows, 2 blocks}; Q MN-major {64, 64, atoms, 2 blocks}
    CUtensorMap map_p2;
    CUtensorMap map_q2;
    int Mk, Nk, K;       // kernel-side problem (after the optional swap)
    int num_kb;          // ceil(K / 64)
    int tiles_m, tiles_n, num_tiles;
    int group_m;         // raster: tile rows per group
    uint32_t idesc;      // tcgen05 instruction descriptor (dtype, majors, N, M)
    int p_mn_major;      // 1: P tile stored MN-major in shared memory
    int q_mn_major;
    int p_3d, q_3d;      // 1: an MN-major stage arrives as one 3-D box (all its 64-wide atoms)
    int p_2k, q_2k;      // 1: map_p2 / map_q2 load two K-blocks (K a multiple of 64)
    int swap;            // 1: D is C^T
    int bf16;            // element type of every operand: 0 fp16, 1 bf16
    // epilogue, in C's (m, n) coordinates
    int M, N;            // C is M x N
    int n_tma;           // columns [0, n_tma) of C go through tensor stores (N rounded down to 8)
    void* C;
    long long ldc;
    const void* bias_n;  // [N] or null
    const void* scale_m; // [M] or null
    const void* resid;   // [M, ldr] or null
    long long ldr;
    int relu;
    // Work split over the persistent workers (clusters of a pair, or CTAs).
    // Tiles [0, dp_tiles) in raster order are computed whole, worker w taking
    // w, w + workers, ...  The remaining sk_tiles are cut into
    // sk_tiles * num_kb K-block iterations dealt out in equal contiguous
    // ranges ("stream-K"); a tile whose range is split is finished by the
    // contributor that arrives last, summing the partials in K order.
    int workers;
    int dp_tiles;
    int sk_tiles;
    int sk_cmax;           // partial slots per split tile
    long long sk_iters;    // sk_tiles * num_kb
    float* ws_partial;     // [workers][sk_cmax][BM][BN] fp32 partial accumulators
    int* ws_count;         // [workers][2] arrival counters, zero between calls
    // watchdog
    long long timeout_cycles;
    int* status;         // device status word
    int inject_skip_load;// test hook: producer never arms this k-block (-1 = off)
};

// Tile / pipeline configuration chosen by the selector.
struct KernelConfig {
    int swap;       // compute C^T = B^T A^T
    int bm;         // 128 (one CTA) or 256 (CTA pair)
    int bn;         // tile columns: 32..256, a compiled value (see gemm_launch.cuh)
    int pair;       // 1: cta_group::2 on a 2-CTA cluster
    int stages;
    int group_m;
    int grid;       // persistent CTAs
    int tiles;
    int sk_tiles;   // tiles computed stream-K (0: every tile whole)
    int sk_cmax;    // partial slots per split tile
    long long ws_bytes;  // workspace the stream-K part needs
};

// Launches one persistent GEMM; returns a cudaError_t.
cudaError_t launch_gemm(const GemmParams& p, const KernelConfig& cfg, int num_sms,
                        cudaStream_t stream);

// Dynamic shared memory (bytes) and ring depth of a configuration; -1 if the
// (bn, pair) combination is not compiled.
int gemm_smem_bytes(int bn, int pair);
int gemm_stages(int bn, int pair);

}  // namespace tg

// gemm_launch.cuh -- the set of compiled tile configurations and their launch.
#pragma once

#include <atomic>

#include "gemm_kernel.cuh"

// Every (BN, PAIR) the library is compiled for: single-CTA 128 x BN tiles and
// CTA-pair 256 x BN tiles.
#define TG_FOR_EACH_CONFIG(X)                                                   \
    X(32, false) X(64, false) X(128, false) X(192, false) X(224, false)        \
    X(256, false) X(128, true) X(192, true) X(224, true) X(256, true)

namespace tg {

template <int BN, bool PAIR, bool AUX, bool SK>
cudaError_t launch_config(const GemmParams& p, const KernelConfig& cfg, cudaStream_t stream);

// Explicit instantiation of one configuration (in gemm_inst_*.cu).
#define TG_INSTANTIATE(B, P, X, S)                                                        \
    template <>                                                                           \
    cudaError_t launch_config<B, P, X, S>(const GemmParams& p, const KernelConfig& cfg,    \
                                          cudaStream_t stream) {                          \
        using TS = TileShape<B, P>;                                                       \
        auto kern = gemm_kernel<B, P, X, S>;                                              \
        static std::atomic<unsigned long long> attr_set{0}; /* one bit per device */     \
        int dev = 0;                                                                      \
        cudaError_t e = cudaGetDevice(&dev);                                              \
        if (e != cudaSuccess) return e;                                                   \
        const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;                    \
        if (!(attr_set.load(std::memory_order_acquire) & bit)) {                          \
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,   \
                                     TS::kSmemBytes);                                     \
            if (e != cudaSuccess) return e;                                               \
            attr_set.fetch_or(bit, std::memory_order_release);                            \
        }                                                                                 \
        cudaLaunchConfig_t lc = {};                                                       \
        cudaLaunchAttribute attr[1];                                                      \
        lc.gridDim = dim3(cfg.grid, 1, 1);                                                \
        lc.blockDim = dim3(kThreads, 1, 1);                                               \
        lc.dynamicSmemBytes = TS::kSmemBytes;                                             \
        lc.stream = stream;                                                               \
        if (P) {                                                                          \
            attr[0].id = cudaLaunchAttributeClusterDimension;                             \
            attr[0].val.clusterDim.x = 2;                                                 \
            attr[0].val.clusterDim.y = 1;                                                 \
            attr[0].val.clusterDim.z = 1;                                                 \
            lc.attrs = attr;                                                              \
            lc.numAttrs = 1;                                                              \
        }                                                                                 \
        return cudaLaunchKernelEx(&lc, kern, p);                                          \
    }

}  // namespace tg

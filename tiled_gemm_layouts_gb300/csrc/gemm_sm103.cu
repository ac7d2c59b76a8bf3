// gemm_sm103.cu -- instantiations and launch of the persistent tcgen05 GEMM.
#include "gemm_kernel.cuh"

namespace tg {

namespace {

template <int BN>
constexpr int stages_for() {
    // Fill ~192 KB of the 227 KB opt-in shared memory with stages (at most 8).
    return (192 * 1024 / TileShape<BN>::kStage) > 8 ? 8 : (192 * 1024 / TileShape<BN>::kStage);
}

template <int BN, int STAGES>
constexpr int smem_bytes() {
    return 1024 /* alignment slack */ + STAGES * TileShape<BN>::kStage +
           (2 * STAGES + 5) * 8 /* barriers */ + 16 /* tmem slot, abort flag */;
}

template <int BN>
cudaError_t launch_bn(const GemmParams& p, const KernelConfig& cfg, cudaStream_t stream) {
    constexpr int S = stages_for<BN>();
    constexpr int bytes = smem_bytes<BN, S>();
    auto kern = gemm_kernel<BN, S>;
    // Cheap and idempotent; keeps the attribute right on every device.
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(cfg.grid, 1, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.dynamicSmemBytes = bytes;
    lc.stream = stream;
    return cudaLaunchKernelEx(&lc, kern, p);
}

}  // namespace

int gemm_smem_bytes(int bn, int /*stages*/, int /*pair*/) {
    switch (bn) {
        case 32: return smem_bytes<32, stages_for<32>()>();
        case 64: return smem_bytes<64, stages_for<64>()>();
        case 128: return smem_bytes<128, stages_for<128>()>();
        case 256: return smem_bytes<256, stages_for<256>()>();
        default: return -1;
    }
}

int gemm_stages(int bn) {
    switch (bn) {
        case 32: return stages_for<32>();
        case 64: return stages_for<64>();
        case 128: return stages_for<128>();
        case 256: return stages_for<256>();
        default: return -1;
    }
}

cudaError_t launch_gemm(const GemmParams& p, const KernelConfig& cfg, int /*num_sms*/,
                        cudaStream_t stream) {
    switch (cfg.bn) {
        case 32: return launch_bn<32>(p, cfg, stream);
        case 64: return launch_bn<64>(p, cfg, stream);
        case 128: return launch_bn<128>(p, cfg, stream);
        case 256: return launch_bn<256>(p, cfg, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace tg

// gemm_sm103.cu -- launch of the persistent tcgen05 GEMM (instantiations live
// in gemm_inst_*.cu so they compile in parallel).
#include "gemm_launch.cuh"

namespace tg {

int gemm_smem_bytes(int bn, int pair) {
#define TG_CASE(B, P) \
    if (bn == B && pair == P) return TileShape<B, P>::kSmemBytes;
    TG_FOR_EACH_CONFIG(TG_CASE)
#undef TG_CASE
    return -1;
}

int gemm_stages(int bn, int pair) {
#define TG_CASE(B, P) \
    if (bn == B && pair == P) return TileShape<B, P>::kStages;
    TG_FOR_EACH_CONFIG(TG_CASE)
#undef TG_CASE
    return -1;
}

cudaError_t launch_gemm(const GemmParams& p, const KernelConfig& cfg, int /*num_sms*/,
                        cudaStream_t stream) {
    const bool aux = p.bias_n != nullptr || p.resid != nullptr;
    const bool sk = p.sk_tiles > 0;
#define TG_CASE(B, P)                                                                      \
    if (cfg.bn == B && cfg.pair == P)                                                      \
        return aux ? (sk ? launch_config<B, P, true, true>(p, cfg, stream)                 \
                         : launch_config<B, P, true, false>(p, cfg, stream))               \
                   : (sk ? launch_config<B, P, false, true>(p, cfg, stream)                \
                         : launch_config<B, P, false, false>(p, cfg, stream));
    TG_FOR_EACH_CONFIG(TG_CASE)
#undef TG_CASE
    return cudaErrorInvalidValue;
}

}  // namespace tg

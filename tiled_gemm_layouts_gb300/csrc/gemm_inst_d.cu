// gemm_inst_d.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
#define X(B, P) TG_INSTANTIATE(B, P)
X(224, true) X(256, true)
#undef X
}  // namespace tg

// gemm_inst_a.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
#define X(B, P) TG_INSTANTIATE(B, P)
X(32, false) X(64, false) X(128, false)
#undef X
}  // namespace tg

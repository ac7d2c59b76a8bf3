// gemm_inst_b.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
#define X(B, P) TG_INSTANTIATE(B, P)
X(192, false) X(224, false) X(256, false)
#undef X
}  // namespace tg

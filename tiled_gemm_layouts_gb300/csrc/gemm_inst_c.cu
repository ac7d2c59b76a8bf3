// gemm_inst_c.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
#define X(B, P) TG_INSTANTIATE(B, P)
X(128, true) X(192, true)
#undef X
}  // namespace tg

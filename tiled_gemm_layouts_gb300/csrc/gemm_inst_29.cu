// gemm_inst_29.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(224, true, false, false)
}  // namespace tg

// gemm_inst_14.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(224, false, false, true)
}  // namespace tg

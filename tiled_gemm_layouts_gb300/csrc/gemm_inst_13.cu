// gemm_inst_13.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(224, false, false, false)
}  // namespace tg

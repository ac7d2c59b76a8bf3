// gemm_inst_3.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(192, false, false)
TG_INSTANTIATE(224, false, false)
}  // namespace tg

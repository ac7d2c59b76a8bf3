// gemm_inst_4.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(192, false, true)
TG_INSTANTIATE(224, false, true)
}  // namespace tg

// gemm_inst_8.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(128, true, true)
TG_INSTANTIATE(192, true, true)
}  // namespace tg

// gemm_inst_12.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(192, false, true, true)
}  // namespace tg

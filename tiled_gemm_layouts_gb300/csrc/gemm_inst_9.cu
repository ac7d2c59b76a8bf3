// gemm_inst_9.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(192, false, false, false)
}  // namespace tg

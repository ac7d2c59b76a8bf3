// gemm_inst_25.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(192, true, false, false)
}  // namespace tg

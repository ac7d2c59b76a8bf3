// gemm_inst_8.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(128, false, true, true)
}  // namespace tg

// gemm_inst_1.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(32, false, false, false)
TG_INSTANTIATE(64, false, false, false)
}  // namespace tg

// gemm_inst_2.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(32, false, false, true)
TG_INSTANTIATE(64, false, false, true)
}  // namespace tg

// gemm_inst_3.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(32, false, true, false)
TG_INSTANTIATE(64, false, true, false)
}  // namespace tg

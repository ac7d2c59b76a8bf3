// gemm_inst_4.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(32, false, true, true)
TG_INSTANTIATE(64, false, true, true)
}  // namespace tg

// gemm_inst_6.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(128, false, false, true)
}  // namespace tg

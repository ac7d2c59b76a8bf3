// gemm_inst_5.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(128, false, false, false)
}  // namespace tg

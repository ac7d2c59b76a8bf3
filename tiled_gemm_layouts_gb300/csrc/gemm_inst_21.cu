// gemm_inst_21.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(128, true, false, false)
}  // namespace tg

// gemm_inst_7.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(128, false, true, false)
}  // namespace tg

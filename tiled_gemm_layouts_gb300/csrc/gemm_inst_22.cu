// gemm_inst_22.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(128, true, false, true)
}  // namespace tg

// gemm_inst_33.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(256, true, false, false)
}  // namespace tg

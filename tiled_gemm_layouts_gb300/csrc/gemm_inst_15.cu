// gemm_inst_15.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(224, false, true, false)
}  // namespace tg

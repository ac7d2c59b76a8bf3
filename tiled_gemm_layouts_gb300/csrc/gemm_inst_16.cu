// gemm_inst_16.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(224, false, true, true)
}  // namespace tg

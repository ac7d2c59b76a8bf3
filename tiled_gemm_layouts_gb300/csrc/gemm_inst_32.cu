// gemm_inst_32.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(224, true, true, true)
}  // namespace tg

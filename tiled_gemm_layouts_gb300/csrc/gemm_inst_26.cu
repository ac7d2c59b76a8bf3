// gemm_inst_26.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(192, true, false, true)
}  // namespace tg

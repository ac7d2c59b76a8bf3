// gemm_inst_28.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(192, true, true, true)
}  // namespace tg

// gemm_inst_11.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(192, false, true, false)
}  // namespace tg

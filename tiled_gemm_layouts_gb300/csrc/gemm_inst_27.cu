// gemm_inst_27.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(192, true, true, false)
}  // namespace tg

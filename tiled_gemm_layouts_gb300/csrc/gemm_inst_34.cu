// gemm_inst_34.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(256, true, false, true)
}  // namespace tg

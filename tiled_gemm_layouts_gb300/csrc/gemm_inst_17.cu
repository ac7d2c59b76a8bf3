// gemm_inst_17.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(256, false, false, false)
}  // namespace tg

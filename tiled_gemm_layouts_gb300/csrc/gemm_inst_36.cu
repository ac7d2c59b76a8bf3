// gemm_inst_36.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(256, true, true, true)
}  // namespace tg

// gemm_inst_24.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(128, true, true, true)
}  // namespace tg

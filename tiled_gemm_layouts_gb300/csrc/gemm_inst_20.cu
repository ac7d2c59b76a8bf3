// gemm_inst_20.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(256, false, true, true)
}  // namespace tg

// gemm_inst_35.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(256, true, true, false)
}  // namespace tg

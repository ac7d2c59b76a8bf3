// gemm_inst_19.cu -- explicit instantiations of some tile configurations.
#include "gemm_launch.cuh"

namespace tg {
TG_INSTANTIATE(256, false, true, false)
}  // namespace tg

// pointwise.h -- parameters of the pointwise kernels (pointwise.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace tg {

struct PwParams {
    int M, N;
    const uint16_t* X;
    long long ldx;        // X(m, n) = X[m*ldx + n], or X[n*ldx + m] when permuted
    uint16_t* C;
    long long ldc;
    const uint16_t* scale;  // [M] or null
    const uint16_t* bias;   // [N] or null
    const uint16_t* R;      // [M, ldr] or null
    long long ldr;
    int relu;
};

cudaError_t launch_pointwise(const PwParams& p, bool transposed, bool bf16, int sms,
                             cudaStream_t stream);

}  // namespace tg

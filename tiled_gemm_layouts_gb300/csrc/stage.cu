// stage.cu -- row copies for operands the tensor maps cannot describe.
//
// A TMA tensor map needs a 16-byte-aligned base and row strides that are whole
// 16-byte units.  Positive strides of any size are valid arguments all the
// same (ninetoothed.org "Named layouts", section "Runtime and compilation"),
// so tg_gemm_ws copies such an operand into an aligned dense buffer in the
// caller's workspace first, and copies an unaligned C out of one afterwards.
// The copy is a plain bandwidth-bound kernel: one thread moves 8 consecutive
// elements of a row, with one 16-byte access on a side that is aligned and
// element accesses otherwise.
#include <cuda_runtime.h>

#include <cstdint>

namespace tg {

namespace {

__global__ void copy_rows_kernel(const uint16_t* __restrict__ src, long long lds,
                                 uint16_t* __restrict__ dst, long long ldd, long long rows,
                                 long long cols) {
    const long long vecs = (cols + 7) / 8;
    const long long total = rows * vecs;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long r = i / vecs, c0 = (i - r * vecs) * 8;
        const uint16_t* s = src + r * lds + c0;
        uint16_t* d = dst + r * ldd + c0;
        const int n = (int)(cols - c0 < 8 ? cols - c0 : 8);
        uint16_t v[8];
        if (n == 8 && (reinterpret_cast<uintptr_t>(s) & 15u) == 0) {
            *reinterpret_cast<uint4*>(v) = *reinterpret_cast<const uint4*>(s);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < n) v[j] = s[j];
        }
        if (n == 8 && (reinterpret_cast<uintptr_t>(d) & 15u) == 0) {
            *reinterpret_cast<uint4*>(d) = *reinterpret_cast<const uint4*>(v);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < n) d[j] = v[j];
        }
    }
}

}  // namespace

// Copies rows x cols 16-bit elements from (src, lds) to (dst, ldd), both
// strides in elements, asynchronously on `stream`.
cudaError_t launch_copy_rows(const void* src, long long lds, void* dst, long long ldd,
                             long long rows, long long cols, cudaStream_t stream) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    const long long work = rows * ((cols + 7) / 8);
    const long long blocks = (work + 255) / 256;
    copy_rows_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(
        static_cast<const uint16_t*>(src), lds, static_cast<uint16_t*>(dst), ldd, rows, cols);
    return cudaGetLastError();
}

}  // namespace tg

// pointwise.cu -- the named-layout pointwise programs: an M x N output
// computed element by element from an M x N input, with missing-axis
// broadcasting and an explicit reordering of the input
// (ninetoothed.org "Named layouts": this version supports pointwise work,
// missing-axis broadcasting, reordering and same-output-domain
// bias/ReLU/residual postprocessing).
//
//     C[m, n] = relu?( X(m, n) * scale_m[m] + bias_n[n] ) + R[m, n]
//
// with the GEMM epilogue's operands and order; scale_m has axes ("m") and
// bias_n axes ("n"), so each broadcasts along the axis it lacks.  X(m, n) is
// X[m*ldx + n], or X[n*ldx + m] when the input is given permuted (storage
// N x M).  Values are fp16/bf16, arithmetic fp32, rounding to nearest even.
//
// The work is HBM-bound (one read of every input byte and one write of C),
// so the kernels are plain coalesced streaming kernels: the row-major input
// moves 8 consecutive elements per thread with 16-byte accesses where
// aligned; a permuted input with 16-byte-aligned rows is transposed in
// 8 x 8 register blocks (16-byte loads and stores on both sides), any other
// permuted input through a 64 x 64 shared-memory tile so that both its reads
// (along m) and C's writes (along n) stay coalesced.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pointwise.h"

namespace tg {

namespace {

template <bool BF>
__device__ __forceinline__ float f32_of(uint16_t h) {
    if constexpr (BF)
        return __bfloat162float(__ushort_as_bfloat16(h));
    else
        return __half2float(__ushort_as_half(h));
}

template <bool BF>
__device__ __forceinline__ uint16_t bits_of(float x) {
    if constexpr (BF)
        return __bfloat16_as_ushort(__float2bfloat16_rn(x));
    else
        return __half_as_ushort(__float2half_rn(x));
}

__device__ __forceinline__ bool aligned16(const void* p) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// y[0..cnt) = p[0..cnt) as floats (one 16-byte load when possible).
template <bool BF>
__device__ __forceinline__ void load8(const uint16_t* p, int cnt, float (&y)[8]) {
    uint16_t v[8];
    if (cnt == 8 && aligned16(p)) {
        *reinterpret_cast<uint4*>(v) = __ldg(reinterpret_cast<const uint4*>(p));
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = j < cnt ? p[j] : 0;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) y[j] = f32_of<BF>(v[j]);
}

template <bool BF>
__device__ __forceinline__ void store8(uint16_t* p, int cnt, const float (&y)[8]) {
    uint16_t v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = bits_of<BF>(y[j]);
    if (cnt == 8 && aligned16(p)) {
        *reinterpret_cast<uint4*>(p) = *reinterpret_cast<const uint4*>(v);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < cnt) p[j] = v[j];
    }
}

// Row-major input: thread i handles C(m, n0 .. n0+7).
template <bool BF>
__global__ void __launch_bounds__(256) pointwise_rows_kernel(const PwParams p) {
    const long long vecs = (p.N + 7) / 8;
    const long long total = (long long)p.M * vecs;
    for (long long i = blockIdx.x * 256LL + threadIdx.x; i < total; i += gridDim.x * 256LL) {
        const int m = (int)(i / vecs);
        const int n0 = (int)(i - (long long)m * vecs) * 8;
        const int cnt = p.N - n0 < 8 ? p.N - n0 : 8;
        float y[8];
        load8<BF>(p.X + (long long)m * p.ldx + n0, cnt, y);
        if (p.scale) {
            const float s = f32_of<BF>(p.scale[m]);
#pragma unroll
            for (int j = 0; j < 8; ++j) y[j] *= s;
        }
        if (p.bias) {
            float b[8];
            load8<BF>(p.bias + n0, cnt, b);
#pragma unroll
            for (int j = 0; j < 8; ++j) y[j] += b[j];
        }
        if (p.relu) {
#pragma unroll
            for (int j = 0; j < 8; ++j) y[j] = fmaxf(y[j], 0.0f);
        }
        if (p.R) {
            float r[8];
            load8<BF>(p.R + (long long)m * p.ldr + n0, cnt, r);
#pragma unroll
            for (int j = 0; j < 8; ++j) y[j] += r[j];
        }
        store8<BF>(p.C + (long long)m * p.ldc + n0, cnt, y);
    }
}

// Permuted input (X(m, n) = X[n*ldx + m]): 64 x 64 tiles through shared
// memory; 32 x 8 threads, each with 16 loads in flight (enough bytes in
// flight per SM to cover HBM latency) and 16 stores.  Reads run along m
// (storage rows), C's writes along n, each a 64-byte run per warp access.
template <bool BF>
__global__ void __launch_bounds__(256) pointwise_transposed_kernel(const PwParams p) {
    __shared__ float tile[64][65];  // [n - n0][m - m0]
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int tiles_m = (p.M + 63) / 64, tiles_n = (p.N + 63) / 64;
    const long long tiles = (long long)tiles_m * tiles_n;
    for (long long t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int m0 = (int)(t % tiles_m) * 64, n0 = (int)(t / tiles_m) * 64;
        uint16_t v[16];
#pragma unroll
        for (int r = 0; r < 8; ++r) {  // storage rows n, coalesced along m
            const int n = n0 + ty + 8 * r;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int m = m0 + tx + 32 * h;
                v[2 * r + h] = (n < p.N && m < p.M) ? p.X[(long long)n * p.ldx + m] : 0;
            }
        }
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int h = 0; h < 2; ++h) tile[ty + 8 * r][tx + 32 * h] = f32_of<BF>(v[2 * r + h]);
        __syncthreads();
#pragma unroll
        for (int r = 0; r < 8; ++r) {  // C rows m, coalesced along n
            const int m = m0 + ty + 8 * r;
            if (m >= p.M) continue;
            const float s = p.scale ? f32_of<BF>(p.scale[m]) : 1.0f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int n = n0 + tx + 32 * h;
                if (n >= p.N) continue;
                float y = tile[tx + 32 * h][ty + 8 * r];
                if (p.scale) y *= s;
                if (p.bias) y += f32_of<BF>(p.bias[n]);
                if (p.relu) y = fmaxf(y, 0.0f);
                if (p.R) y += f32_of<BF>(p.R[(long long)m * p.ldr + n]);
                p.C[(long long)m * p.ldc + n] = bits_of<BF>(y);
            }
        }
        __syncthreads();
    }
}

// The permuted input when X's rows, C's rows, R's rows and bias all start on
// 16-byte boundaries: no shared memory.  Each thread loads an 8 x 8 block of
// elements -- 8 storage rows n .. n+7, 8 consecutive m each, one 16-byte
// load per row -- and transposes it in registers: output row m+c, columns
// n .. n+7, is 4 words, word w taking element c of storage rows 2w and 2w+1
// (one byte permute each).  A warp covers 64 storage rows x 32 columns:
// lane (a, b) = (lane / 4, lane % 4) owns rows n0 + 8a and columns m0 + 8b,
// so each load instruction reads 8 storage rows x 64 contiguous bytes and
// each store instruction writes 4 rows of C x 128 contiguous bytes.  Items
// are dealt out grid-stride with m fastest, so concurrent warps read whole
// storage rows and write neighbouring runs of the same C rows.  With an
// epilogue (EPI), the block's 8 scales and 8 biases -- and with a residual
// (RES) its 8 rows of R -- are loaded together with X, so that no load waits
// behind another; the residual's registers cost a resident block per SM, so
// it is a separate instance.
template <bool BF>
__device__ __forceinline__ void raw8(const uint16_t* p, int cnt, uint32_t (&w)[4]) {
    if (cnt == 8 && aligned16(p)) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
        w[0] = v.x;
        w[1] = v.y;
        w[2] = v.z;
        w[3] = v.w;
    } else {
        uint16_t e[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) e[j] = j < cnt ? p[j] : 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) w[k] = (uint32_t)e[2 * k] | ((uint32_t)e[2 * k + 1] << 16);
    }
}

template <bool BF>
__device__ __forceinline__ float half_of(uint32_t w, int hi) {
    return f32_of<BF>((uint16_t)(hi ? w >> 16 : w & 0xffffu));
}

template <bool BF, bool EPI, bool RES>
__global__ void __launch_bounds__(256, RES ? 2 : 3) pointwise_transposed_reg_kernel(const PwParams p) {
    const int lane = threadIdx.x & 31;
    const int a = lane >> 2, b = lane & 3;
    const int items_m = (p.M + 31) / 32, items_n = (p.N + 63) / 64;
    const long long items = (long long)items_m * items_n;
    const long long stride = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long it = blockIdx.x * (long long)(blockDim.x >> 5) + (threadIdx.x >> 5); it < items;
         it += stride) {
        const int m = (int)(it % items_m) * 32 + 8 * b;
        const int n = (int)(it / items_m) * 64 + 8 * a;
        const int mc = p.M - m, nc = p.N - n;  // columns / rows of the block inside X
        if (mc <= 0 || nc <= 0) continue;
        const int mcnt = mc < 8 ? mc : 8, cnt = nc < 8 ? nc : 8;
        uint32_t x[8][4];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            if (r < nc) {
                raw8<BF>(p.X + (long long)(n + r) * p.ldx + m, mcnt, x[r]);
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) x[r][k] = 0;
            }
        }
        uint32_t rr[8][4];
        float sc[8], bi[8];
        if constexpr (EPI) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                if (RES && c < mc) {
                    raw8<BF>(p.R + (long long)(m + c) * p.ldr + n, cnt, rr[c]);
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k) rr[c][k] = 0;
                }
            }
            if (p.scale) {
                load8<BF>(p.scale + m, mcnt, sc);
            } else {
#pragma unroll
                for (int c = 0; c < 8; ++c) sc[c] = 1.0f;
            }
            if (p.bias) {
                load8<BF>(p.bias + n, cnt, bi);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) bi[j] = 0.0f;
            }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            if (c >= mc) break;
            uint32_t y[4];
#pragma unroll
            for (int w = 0; w < 4; ++w)
                y[w] = __byte_perm(x[2 * w][c >> 1], x[2 * w + 1][c >> 1],
                                   (c & 1) ? 0x7632u : 0x5410u);
            if constexpr (EPI) {
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    float v0 = half_of<BF>(y[w], 0), v1 = half_of<BF>(y[w], 1);
                    if (p.scale) {  // each step only with its operand (a -0 stays -0)
                        v0 *= sc[c];
                        v1 *= sc[c];
                    }
                    if (p.bias) {
                        v0 += bi[2 * w];
                        v1 += bi[2 * w + 1];
                    }
                    if (p.relu) {
                        v0 = fmaxf(v0, 0.0f);
                        v1 = fmaxf(v1, 0.0f);
                    }
                    if (RES) {
                        v0 += half_of<BF>(rr[c][w], 0);
                        v1 += half_of<BF>(rr[c][w], 1);
                    }
                    y[w] = (uint32_t)bits_of<BF>(v0) | ((uint32_t)bits_of<BF>(v1) << 16);
                }
            }
            uint16_t* dst = p.C + (long long)(m + c) * p.ldc + n;
            if (cnt == 8) {
                *reinterpret_cast<uint4*>(dst) = make_uint4(y[0], y[1], y[2], y[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j < cnt) dst[j] = (uint16_t)(y[j >> 1] >> (16 * (j & 1)));
            }
        }
    }
}

}  // namespace

cudaError_t launch_pointwise(const PwParams& p, bool transposed, bool bf16, int sms,
                             cudaStream_t stream) {
    auto rows16 = [](const void* base, long long ld) {
        return base == nullptr ||
               ((reinterpret_cast<uintptr_t>(base) & 15u) == 0 && (ld * 2) % 16 == 0);
    };
    const bool vec = rows16(p.X, p.ldx) && rows16(p.C, p.ldc) && rows16(p.R, p.ldr) &&
                     rows16(p.bias, 8);
    if (transposed && vec) {
        // resident blocks of 8 warps per SM (no shared memory): 3 (at most
        // 85 registers a thread), 2 with a residual (128); each warp works
        // through several items, so the last round leaves few SMs idle
        const bool epi = p.scale || p.bias || p.relu || p.R, res = p.R != nullptr;
        const long long warps = (long long)((p.M + 31) / 32) * ((p.N + 63) / 64);
        const long long blocks = (warps + 7) / 8, cap = (long long)sms * (res ? 2 : 3);
        const unsigned grid = (unsigned)(blocks < cap ? blocks : cap);
        auto k = bf16 ? (res ? pointwise_transposed_reg_kernel<true, true, true>
                             : epi ? pointwise_transposed_reg_kernel<true, true, false>
                                   : pointwise_transposed_reg_kernel<true, false, false>)
                      : (res ? pointwise_transposed_reg_kernel<false, true, true>
                             : epi ? pointwise_transposed_reg_kernel<false, true, false>
                                   : pointwise_transposed_reg_kernel<false, false, false>);
        k<<<grid, 256, 0, stream>>>(p);
        return cudaGetLastError();
    }
    const long long cap = (long long)sms * 8;  // 8 blocks of 256 threads per SM
    long long blocks;
    if (transposed) {
        blocks = (long long)((p.M + 63) / 64) * ((p.N + 63) / 64);
    } else {
        blocks = ((long long)p.M * ((p.N + 7) / 8) + 255) / 256;
    }
    const unsigned grid = (unsigned)(blocks < cap ? blocks : cap);
    if (transposed) {
        if (bf16)
            pointwise_transposed_kernel<true><<<grid, 256, 0, stream>>>(p);
        else
            pointwise_transposed_kernel<false><<<grid, 256, 0, stream>>>(p);
    } else {
        if (bf16)
            pointwise_rows_kernel<true><<<grid, 256, 0, stream>>>(p);
        else
            pointwise_rows_kernel<false><<<grid, 256, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace tg

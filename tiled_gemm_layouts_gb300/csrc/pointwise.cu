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
// aligned; the permuted input goes through a 64 x 64 shared-memory tile so
// that both its reads (along m) and C's writes (along n) stay coalesced.
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

// The same with 16-byte accesses, when X's rows, C's rows, R's rows and bias
// all start on 16-byte boundaries: each thread moves two 8-element vectors
// of storage rows in, and writes two 8-element vectors of C rows out.  The
// next tile's loads are issued before the current tile's stores, so a load
// phase and a store phase are always in flight together.
template <bool BF>
__device__ __forceinline__ void load_tile_vec(const PwParams& p, int m0, int n0, int t,
                                              float (&in)[2][8]) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {  // storage row n, elements m .. m+7
        const int idx = t + 256 * i, row = idx >> 3, seg = idx & 7;
        const int n = n0 + row, m = m0 + seg * 8;
        const int cnt = n < p.N ? (p.M - m < 8 ? p.M - m : 8) : 0;
        if (cnt > 0) {
            load8<BF>(p.X + (long long)n * p.ldx + m, cnt, in[i]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) in[i][j] = 0.0f;
        }
    }
}

template <bool BF>
__global__ void __launch_bounds__(256) pointwise_transposed_vec_kernel(const PwParams p) {
    __shared__ float tile[64][65];  // [n - n0][m - m0]
    const int t = threadIdx.x;
    const int tiles_m = (p.M + 63) / 64, tiles_n = (p.N + 63) / 64;
    const long long tiles = (long long)tiles_m * tiles_n;
    float in[2][8];
    long long u = blockIdx.x;
    if (u < tiles) load_tile_vec<BF>(p, (int)(u % tiles_m) * 64, (int)(u / tiles_m) * 64, t, in);
    for (; u < tiles; u += gridDim.x) {
        const int m0 = (int)(u % tiles_m) * 64, n0 = (int)(u / tiles_m) * 64;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int idx = t + 256 * i, row = idx >> 3, seg = idx & 7;
#pragma unroll
            for (int j = 0; j < 8; ++j) tile[row][seg * 8 + j] = in[i][j];
        }
        __syncthreads();
        const long long nxt = u + gridDim.x;  // its loads overlap this tile's stores
        if (nxt < tiles)
            load_tile_vec<BF>(p, (int)(nxt % tiles_m) * 64, (int)(nxt / tiles_m) * 64, t, in);
#pragma unroll
        for (int i = 0; i < 2; ++i) {  // C row m, elements n .. n+7
            const int idx = t + 256 * i, mrow = idx >> 3, seg = idx & 7;
            const int m = m0 + mrow, n = n0 + seg * 8;
            if (m >= p.M || n >= p.N) continue;
            const int cnt = p.N - n < 8 ? p.N - n : 8;
            float y[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) y[j] = tile[seg * 8 + j][mrow];
            if (p.scale) {
                const float s = f32_of<BF>(p.scale[m]);
#pragma unroll
                for (int j = 0; j < 8; ++j) y[j] *= s;
            }
            if (p.bias) {
                float b[8];
                load8<BF>(p.bias + n, cnt, b);
#pragma unroll
                for (int j = 0; j < 8; ++j) y[j] += b[j];
            }
            if (p.relu) {
#pragma unroll
                for (int j = 0; j < 8; ++j) y[j] = fmaxf(y[j], 0.0f);
            }
            if (p.R) {
                float r[8];
                load8<BF>(p.R + (long long)m * p.ldr + n, cnt, r);
#pragma unroll
                for (int j = 0; j < 8; ++j) y[j] += r[j];
            }
            store8<BF>(p.C + (long long)m * p.ldc + n, cnt, y);
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_pointwise(const PwParams& p, bool transposed, bool bf16, int sms,
                             cudaStream_t stream) {
    const long long cap = (long long)sms * 8;  // 8 blocks of 256 threads per SM
    long long blocks;
    if (transposed) {
        blocks = (long long)((p.M + 63) / 64) * ((p.N + 63) / 64);
    } else {
        blocks = ((long long)p.M * ((p.N + 7) / 8) + 255) / 256;
    }
    const unsigned grid = (unsigned)(blocks < cap ? blocks : cap);
    auto rows16 = [](const void* base, long long ld) {
        return base == nullptr ||
               ((reinterpret_cast<uintptr_t>(base) & 15u) == 0 && (ld * 2) % 16 == 0);
    };
    const bool vec = rows16(p.X, p.ldx) && rows16(p.C, p.ldc) && rows16(p.R, p.ldr) &&
                     rows16(p.bias, 8);
    if (transposed && vec) {
        if (bf16)
            pointwise_transposed_vec_kernel<true><<<grid, 256, 0, stream>>>(p);
        else
            pointwise_transposed_vec_kernel<false><<<grid, 256, 0, stream>>>(p);
    } else if (transposed) {
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

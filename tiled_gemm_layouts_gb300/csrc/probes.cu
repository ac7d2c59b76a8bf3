// probes.cu -- hardware probes that pin the layout module to what the GPU
// actually does:
//   * tg_probe_swizzle128: a TMA load with the 128-byte swizzle into shared
//     memory, dumped byte for byte, so the element found at every shared
//     offset can be compared with the (offset) -> (row, col) swizzle layout;
//   * tg_probe_tmem_32x32b: one tcgen05.mma whose accumulator encodes its own
//     coordinates (D[m][n] = 256 m + n), read back through tcgen05.ld 32x32b,
//     so the (register, lane, warp) -> (m, n) readout layout can be checked;
//   * tg_probe_folded_layout: a folded layout (tilegemm_layout_device.h)
//     evaluated by device code for every value of its variable inputs, so the
//     kernel-side evaluation can be checked against the host module.
// Every wait is bounded; a probe that gives up writes a status code.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/tilegemm.h"
#include "../../include/tilegemm_probes.h"
#include "ptx.cuh"

namespace tg {
namespace {

constexpr long long kProbeTimeout = 2000000000LL;

__device__ bool probe_wait(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kProbeTimeout) return false;
    return true;
}

// rows x 128 bytes through TMA (box {64 elements, rows}) -> raw dump.
__global__ void __launch_bounds__(128) swizzle_probe_kernel(const __grid_constant__ CUtensorMap map,
                                                            int rows, uint4* dst, int* status) {
    extern __shared__ uint8_t raw[];
    uint8_t* tile = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar;
    __shared__ int ok;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(b, rows * 128);
        tma_load_2d(smem_addr(tile), &map, b, 0, 0);
        ok = probe_wait(b, 0);
        if (!ok) atomicExch(status, 1);
    }
    __syncthreads();
    if (!ok) return;
    const uint4* s = reinterpret_cast<const uint4*>(tile);
    for (int i = threadIdx.x; i < rows * 8; i += blockDim.x) dst[i] = s[i];
}

// Byte offset of element (row, col) of a K-major tile with 128-byte rows in
// the 128-byte swizzle (chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t sw128(int row, int col) {
    const int byte = col * 2;
    return row * 128 + ((((byte >> 4) ^ (row & 7)) << 4) | (byte & 15));
}

template <int BN>
__global__ void __launch_bounds__(128) tmem_probe_kernel(uint32_t* dst, int* status) {
    extern __shared__ uint8_t raw[];
    uint8_t* sa = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sb = sa + 128 * 128;
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int ok;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t b = smem_addr(&bar);
    constexpr uint32_t kCols = BN < 32 ? 32 : BN;

    // A: 128 x 64 (K-major), A(m,0) = m, A(m,1) = 1.  B^T: BN x 64 (K-major),
    // B(0,n) = 256, B(1,n) = n.  Only the first 16 K columns are multiplied.
    uint16_t* a16 = reinterpret_cast<uint16_t*>(sa);
    uint16_t* b16 = reinterpret_cast<uint16_t*>(sb);
    for (int i = threadIdx.x; i < 128 * 64; i += blockDim.x) a16[i] = 0;
    for (int i = threadIdx.x; i < BN * 64; i += blockDim.x) b16[i] = 0;
    __syncthreads();
    for (int r = threadIdx.x; r < 128; r += blockDim.x) {
        a16[sw128(r, 0) / 2] = __half_as_ushort(__float2half_rn((float)r));
        a16[sw128(r, 1) / 2] = __half_as_ushort(__float2half_rn(1.0f));
    }
    for (int r = threadIdx.x; r < BN; r += blockDim.x) {
        b16[sw128(r, 0) / 2] = __half_as_ushort(__float2half_rn(256.0f));
        b16[sw128(r, 1) / 2] = __half_as_ushort(__float2half_rn((float)r));
    }
    fence_proxy_async_shared();  // generic writes -> visible to the tensor core
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc<1>(smem_addr(&tmem_slot), kCols);
        tmem_relinquish<1>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    if (threadIdx.x == 0) {
        const uint32_t idesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
        mma_f16<1>(tmem, smem_desc_sw128(smem_addr(sa), 16, 1024),
                   smem_desc_sw128(smem_addr(sb), 16, 1024), idesc, 0);
        mma_commit(b);
        ok = probe_wait(b, 0);
        if (!ok) atomicExch(status, 2);
    }
    __syncthreads();
    tc_fence_after();
    if (ok) {
        for (int c = 0; c < BN / 32; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tmem + ((uint32_t)(warp * 32) << 16) + c * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) dst[(warp * 32 + lane) * BN + c * 32 + j] = v[j];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<1>(tmem, kCols);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Thread c evaluates the folded layout at variable inputs split from c
// (first variable dim in the lowest bits) and writes its n_outs outputs.
__global__ void __launch_bounds__(256) folded_probe_kernel(const tg_folded_layout f, int32_t* dst) {
    const uint32_t c = blockIdx.x * 256u + threadIdx.x;
    if (c >= (1u << f.n_bits)) return;
    uint32_t vars[TG_FOLD_MAX_VARS];
    int shift = 0;
#pragma unroll
    for (int v = 0; v < TG_FOLD_MAX_VARS; ++v) {
        const int b = v < f.n_vars ? f.var_bits[v] : 0;
        vars[v] = b > 0 ? (c >> shift) & ((1u << b) - 1u) : 0u;
        shift += b;
    }
    const uint32_t packed = tg_folded_apply_packed(&f, vars);
    for (int o = 0; o < f.n_outs; ++o) dst[(size_t)c * f.n_outs + o] = tg_folded_output(&f, packed, o);
}

}  // namespace
}  // namespace tg

using namespace tg;


using namespace tg;

extern "C" int tg_probe_swizzle128(const void* src, int rows, int64_t ld, void* dst,
                                   int* status_dev, cudaStream_t stream) {
    if (!src || !dst || !status_dev || rows < 8 || rows > 256 || (rows & (rows - 1)) || ld < 64 ||
        (ld * 2) % 16 || (reinterpret_cast<uintptr_t>(src) & 15) ||
        (reinterpret_cast<uintptr_t>(dst) & 15))
        return TG_ERR_INVALID_ARG;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return TG_ERR_CUDA;
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)ld, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)rows};
    const cuuint32_t estr[2] = {1, 1};
    if (reinterpret_cast<EncodeTiledFn>(fn)(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                                            const_cast<void*>(src), dims, strides, box, estr,
                                            CU_TENSOR_MAP_INTERLEAVE_NONE,
                                            CU_TENSOR_MAP_SWIZZLE_128B,
                                            CU_TENSOR_MAP_L2_PROMOTION_NONE,
                                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return TG_ERR_CUDA;
    const int smem = 1024 + rows * 128;
    if (cudaFuncSetAttribute(swizzle_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
        return TG_ERR_CUDA;
    swizzle_probe_kernel<<<1, 128, smem, stream>>>(map, rows, static_cast<uint4*>(dst), status_dev);
    return cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

extern "C" int tg_probe_tmem_32x32b(int bn, void* dst, int* status_dev, cudaStream_t stream) {
    if (!dst || !status_dev) return TG_ERR_INVALID_ARG;
    const int smem = 1024 + 128 * 128 + bn * 128;
    cudaError_t e;
    switch (bn) {
        case 64:
            cudaFuncSetAttribute(tmem_probe_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            tmem_probe_kernel<64><<<1, 128, smem, stream>>>(static_cast<uint32_t*>(dst), status_dev);
            break;
        case 128:
            cudaFuncSetAttribute(tmem_probe_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            tmem_probe_kernel<128><<<1, 128, smem, stream>>>(static_cast<uint32_t*>(dst), status_dev);
            break;
        case 256:
            cudaFuncSetAttribute(tmem_probe_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            tmem_probe_kernel<256><<<1, 128, smem, stream>>>(static_cast<uint32_t*>(dst), status_dev);
            break;
        default:
            return TG_ERR_INVALID_ARG;
    }
    e = cudaGetLastError();
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

extern "C" int tg_probe_folded_layout(const tg_folded_layout* f, void* dst, size_t dst_bytes,
                                      cudaStream_t stream) {
    if (!f || !dst || f->n_vars < 0 || f->n_vars > TG_FOLD_MAX_VARS || f->n_bits < 0 ||
        f->n_bits > 20 || f->n_outs < 1 || f->n_outs > TG_FOLD_MAX_OUTS)
        return TG_ERR_INVALID_ARG;
    int bits = 0;
    for (int v = 0; v < f->n_vars; ++v) {
        if (f->var_bits[v] < 0 || f->var_bits[v] > 20) return TG_ERR_INVALID_ARG;
        bits += f->var_bits[v];
    }
    if (bits != f->n_bits) return TG_ERR_INVALID_ARG;
    for (int o = 0; o < f->n_outs; ++o)
        if (f->out_bits[o] < 0 || f->out_bits[o] > 30 || f->out_shift[o] < 0 ||
            f->out_shift[o] + f->out_bits[o] > 32)
            return TG_ERR_INVALID_ARG;
    const size_t n = (size_t)1 << f->n_bits;
    if (dst_bytes < n * f->n_outs * sizeof(int32_t)) return TG_ERR_BUFFER;
    int dev = -1;
    cudaPointerAttributes at;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaPointerGetAttributes(&at, dst) != cudaSuccess) {
        cudaGetLastError();
        return TG_ERR_POINTER;
    }
    if (at.type != cudaMemoryTypeDevice || at.device != dev) return TG_ERR_POINTER;
    folded_probe_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(*f, static_cast<int32_t*>(dst));
    return cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

// noalloc.cu -- tg_gemm_static_ws: the stream-K GEMM with its scratch in a
// fixed, statically allocated device array, for callers that cannot allocate
// device memory themselves.
//
// Who needs it: code for which cudaMalloc is not an option -- code under an
// outside allocator that owns all of the device's memory (a framework's
// memory pool), plugins whose host framework forbids device allocations, and
// latency-bound host paths that cannot afford the implicit device
// synchronisation a cudaMalloc or cudaFree may cause.  Such callers can still
// pass their inputs and outputs, but not the workspace tg_gemm_ws asks for.
//
// The scratch lives in one file-scope __device__ array of kScratchBytes that
// every GPU loading this library keeps until the process exits.  In host code
// the array's name is only a stand-in symbol, never a device address: the
// address is looked up once per device with cudaGetSymbolAddress (with that
// device current) and cached.  The library does not support cudaDeviceReset:
// after one, the cached address may be stale.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/tilegemm.h"
#include "select.h"

namespace {

// 40 MiB: enough for every stream-K split the default selection makes on a
// 152-SM GPU -- the tail after whole waves, two partial slots per worker of at
// most 256 x 256 fp32 per cluster (76 x 2 x 256 KB plus counters, 39.8 MB) --
// and for the staging copies of unaligned operands of smaller problems.
constexpr size_t kScratchBytes = size_t(40) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
bool g_scratch_ready[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (set up on the
// first call per device).
int scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return TG_ERR_UNSUPPORTED_DEVICE;
    }
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ready[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return TG_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
        g_scratch_ready[dev] = true;
    }
    *out = g_scratch_addr[dev];
    return TG_OK;
}

}  // namespace

extern "C" int tg_gemm_static_ws(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                                 tg_perm permA, const void* B, int64_t ldb, tg_perm permB,
                                 void* C, int64_t ldc, tg_dtype dtype, const tg_epilogue* epi,
                                 cudaStream_t stream) {
    // The whole scratch this call needs: the split's counters and partial
    // sums, then staging copies of operands a tensor map cannot describe.
    size_t need = 0;
    int rc = tg_gemm_workspace_size_ex(M, N, K, A, lda, permA, B, ldb, permB, C, ldc, dtype, epi,
                                       &need);
    if (rc != TG_OK) return rc;
    if (need > kScratchBytes) return TG_ERR_BUFFER;  // more scratch than the static array holds
    size_t counters = 0;
    const bool has_epi = epi && (epi->bias_n || epi->scale_m || epi->residual || epi->relu);
    if ((rc = tg::split_counter_bytes(M, N, K, (int)dtype, (int)permA, (int)permB, has_epi,
                                      &counters)) != TG_OK)
        return rc;
    if (counters > need) return TG_ERR_CUDA;  // inconsistent sizes: never launch on them
    void* scratch = nullptr;
    if ((rc = scratch_address(&scratch)) != TG_OK) return rc;
    if (counters > 0) {
        // The array keeps whatever the previous call left: zero the split's
        // arrival counters (in stream order, before this call's kernel reads
        // them).  The partial-sum slots and staging copies are always written
        // before they are read.
        if (cudaMemsetAsync(scratch, 0, counters, stream) != cudaSuccess) {
            cudaGetLastError();
            return TG_ERR_CUDA;
        }
    }
    return tg_gemm_ws(M, N, K, A, lda, permA, B, ldb, permB, C, ldc, dtype, epi,
                      need > 0 ? scratch : nullptr, need, stream);
}

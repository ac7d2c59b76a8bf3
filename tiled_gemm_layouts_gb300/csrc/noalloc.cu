// noalloc.cu -- tg_gemm_static_ws: the stream-K GEMM with its scratch in a
// fixed, statically allocated device array, for callers that cannot allocate
// device memory themselves.
//
// Who needs it: code that runs where cudaMalloc is not an option -- inside a
// CUDA stream capture (a cudaMalloc there breaks the capture), under an
// external allocator that owns all device memory, or in a plugin whose host
// framework forbids device allocations.  Such callers can still pass their
// inputs and outputs, but not the workspace tg_gemm_ws asks for.
//
// The scratch lives in one file-scope __device__ array of kScratchBytes that
// every GPU loading this library keeps until the process exits.  In host code
// the array's name is only a stand-in symbol, never a device address: the
// address is looked up once per device with cudaGetSymbolAddress (with that
// device current) and cached.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/tilegemm.h"

namespace {

// 40 MiB: enough for the stream-K split of every 256 x 256 CTA-pair tiling on
// a 152-SM GPU with two contributors per split tile (76 clusters x 2 slots x
// 256 KB plus counters, 39.8 MB).
constexpr size_t kScratchBytes = size_t(40) << 20;
// The arrival counters sit at the start of the workspace; they must be zero
// when a launch starts.  They occupy at most this many bytes for any split.
constexpr size_t kCounterBytes = 4096;

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
    size_t need = 0;
    int rc = tg_gemm_workspace_size_ex(M, N, K, A, lda, permA, B, ldb, permB, C, ldc, dtype, epi,
                                       &need);
    if (rc != TG_OK) return rc;
    if (need > kScratchBytes) return TG_ERR_BUFFER;  // more scratch than the static array holds
    void* scratch = nullptr;
    if ((rc = scratch_address(&scratch)) != TG_OK) return rc;
    if (need > 0) {
        // The array keeps whatever the previous call left: zero the counters
        // (in stream order, before this call's kernel reads them).
        if (cudaMemsetAsync(scratch, 0, need < kCounterBytes ? need : kCounterBytes, stream) !=
            cudaSuccess) {
            cudaGetLastError();
            return TG_ERR_CUDA;
        }
    }
    return tg_gemm_ws(M, N, K, A, lda, permA, B, ldb, permB, C, ldc, dtype, epi,
                      need > 0 ? scratch : nullptr, need, stream);
}

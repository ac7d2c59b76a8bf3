// api.cu -- host side of tg_gemm: argument checks, device and pointer
// checks, tile selection, tensor-map encoding and the single launch.
//
// Checks follow ninetoothed.org "Named layouts", section "Runtime and
// compilation": logical sizes and input strides positive, non-contiguous
// inputs allowed, output writes provably non-overlapping, output storage
// disjoint from every input, all checks before any kernel work, and an
// unprovable case is an error.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/tilegemm.h"
#include "gemm_params.h"
#include "pointwise.h"
#include "select.h"

namespace tg {

// Device status word: kernels record the first watchdog expiry here.
__device__ int g_device_status;

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxDim = 2147483647LL;
constexpr long long kDefaultTimeout = 4000000000LL;

std::atomic<long long> g_timeout{kDefaultTimeout};
std::atomic<long long> g_skip_kblock{-1};

struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int sms = 0;
    int* status = nullptr;  // device address of g_device_status
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*AddressRangeFn)(CUdeviceptr*, size_t*, CUdeviceptr);
EncodeTiledFn g_encode = nullptr;
AddressRangeFn g_range = nullptr;
std::once_flag g_driver_once;

void load_driver_entry_points() {
    std::call_once(g_driver_once, [] {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_range = reinterpret_cast<AddressRangeFn>(fn);
    });
}

// Current device, checked for tcgen05 (compute capability 10.x) once.
int current_device(int* dev_out, DeviceInfo** info_out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return TG_ERR_UNSUPPORTED_DEVICE;
    }
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return TG_ERR_UNSUPPORTED_DEVICE;
        }
        d.supported = (major == 10 && minor == 3);  // the library is built for sm_103a only
        d.sms = sms;
        if (d.supported) {
            void* addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) {
                cudaGetLastError();
                return TG_ERR_CUDA;
            }
            d.status = static_cast<int*>(addr);
        }
        d.ready = true;
    }
    if (!d.supported) return TG_ERR_UNSUPPORTED_DEVICE;
    *dev_out = dev;
    *info_out = &d;
    return TG_OK;
}

typedef unsigned __int128 u128;

struct Span {
    uintptr_t lo = 0;
    u128 hi = 0;  // exclusive
    bool present = false;
};

// Bytes [p, p + ((rows-1)*ld + width) * 2) of a row-strided 16-bit matrix.
Span span_of(const void* p, int64_t rows, int64_t width, int64_t ld) {
    Span s;
    if (!p) return s;
    s.present = true;
    s.lo = reinterpret_cast<uintptr_t>(p);
    s.hi = (u128)s.lo + ((u128)(rows - 1) * (u128)ld + (u128)width) * 2u;
    return s;
}

bool intersects(const Span& a, const Span& b) {
    if (!a.present || !b.present) return false;
    return (u128)a.lo < b.hi && (u128)b.lo < a.hi;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Args {
    int64_t M, N, K;
    const void* A;
    int64_t lda;
    int permA;
    const void* B;
    int64_t ldb;
    int permB;
    void* C;
    int64_t ldc;
    int dtype;
    const void *bias, *scale, *resid;
    int64_t ldr;
    int relu;
};

// Checks that need no device: sizes, enums, strides, alignment, overlap.
int check_shape(int64_t M, int64_t N, int64_t K, int dtype, int permA, int permB,
                const tg_epilogue* epi) {
    if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return TG_ERR_INVALID_ARG;
    if ((permA != TG_OP_N && permA != TG_OP_T) || (permB != TG_OP_N && permB != TG_OP_T))
        return TG_ERR_INVALID_ARG;
    if (epi && epi->relu != 0 && epi->relu != 1) return TG_ERR_INVALID_ARG;
    if (dtype != TG_F16 && dtype != TG_BF16) return TG_ERR_DTYPE;
    return TG_OK;
}

int check_args(const Args& a) {
    if (!a.A || !a.B || !a.C) return TG_ERR_INVALID_ARG;
    const int64_t a_rows = a.permA == TG_OP_N ? a.M : a.K, a_w = a.permA == TG_OP_N ? a.K : a.M;
    const int64_t b_rows = a.permB == TG_OP_N ? a.K : a.N, b_w = a.permB == TG_OP_N ? a.N : a.K;
    // Leading dimensions: >= row width (so rows never overlap), and below the
    // tensor-map stride limit of 2^40 bytes.
    constexpr int64_t kMaxLd = (1LL << 39) - 8;
    if (a.lda < a_w || a.ldb < b_w || a.ldc < a.N || a.lda > kMaxLd || a.ldb > kMaxLd ||
        a.ldc > kMaxLd)
        return TG_ERR_STRIDE;
    if (a.resid && (a.ldr < a.N || a.ldr > kMaxLd)) return TG_ERR_STRIDE;
    // every pointer addresses whole 16-bit elements
    auto odd = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) != 0; };
    if (odd(a.A) || odd(a.B) || odd(a.C) || odd(a.bias) || odd(a.scale) || odd(a.resid))
        return TG_ERR_ALIGN;
    const Span c = span_of(a.C, a.M, a.N, a.ldc);
    const Span ins[5] = {span_of(a.A, a_rows, a_w, a.lda), span_of(a.B, b_rows, b_w, a.ldb),
                         span_of(a.bias, 1, a.N, a.N), span_of(a.scale, 1, a.M, a.M),
                         span_of(a.resid, a.M, a.N, a.ldr)};
    for (const Span& s : ins)
        if (intersects(c, s)) return TG_ERR_OVERLAP;
    return TG_OK;
}

// The touched bytes of every operand must lie inside one allocation of the
// current device (proves the kernel cannot read or write outside caller memory).
int check_pointer(const void* p, const Span& s, int dev) {
    if (!p) return TG_OK;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return TG_ERR_POINTER;
    }
    if ((at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) || at.device != dev)
        return TG_ERR_POINTER;
    if (!g_range) return TG_ERR_POINTER;
    CUdeviceptr base = 0;
    size_t size = 0;
    if (g_range(&base, &size, reinterpret_cast<CUdeviceptr>(p)) != CUDA_SUCCESS)
        return TG_ERR_POINTER;
    if ((u128)s.lo < (u128)base || s.hi > (u128)base + size) return TG_ERR_POINTER;
    return TG_OK;
}

int check_pointers(const Args& a, int dev) {
    const int64_t a_rows = a.permA == TG_OP_N ? a.M : a.K, a_w = a.permA == TG_OP_N ? a.K : a.M;
    const int64_t b_rows = a.permB == TG_OP_N ? a.K : a.N, b_w = a.permB == TG_OP_N ? a.N : a.K;
    int rc;
    if ((rc = check_pointer(a.A, span_of(a.A, a_rows, a_w, a.lda), dev))) return rc;
    if ((rc = check_pointer(a.B, span_of(a.B, b_rows, b_w, a.ldb), dev))) return rc;
    if ((rc = check_pointer(a.C, span_of(a.C, a.M, a.N, a.ldc), dev))) return rc;
    if ((rc = check_pointer(a.bias, span_of(a.bias, 1, a.N, a.N), dev))) return rc;
    if ((rc = check_pointer(a.scale, span_of(a.scale, 1, a.M, a.M), dev))) return rc;
    if ((rc = check_pointer(a.resid, span_of(a.resid, a.M, a.N, a.ldr), dev))) return rc;
    return TG_OK;
}

bool encode_2d(CUtensorMap* map, int dtype, const void* base, uint64_t inner, uint64_t outer,
               int64_t ld, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt =
        dtype == TG_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Operand tensor map.  `rows` x `k` operand; if mn_major the storage has the
// rows dimension contiguous (dims {rows, K}), else K contiguous (dims {K, rows}).
bool encode_operand(CUtensorMap* map, int dtype, const void* base, int64_t rows, int64_t k,
                    int64_t ld, bool mn_major, int box_rows) {
    if (mn_major) return encode_2d(map, dtype, base, rows, k, ld, 64, 64);
    return encode_2d(map, dtype, base, k, rows, ld, 64, box_rows);
}

// An MN-major operand whose per-CTA stage is `atoms` 64-wide swizzle atoms,
// as one 3-D box: dims {64 contiguous elements, K, rows / 64} with strides
// {ld, 64} elements, box {64, 64, atoms}.  The atoms land 8 KB apart, which
// is the stage layout the MMA descriptors expect, and a stage takes one TMA
// instruction instead of `atoms` (each instruction costs TMA throughput).
// Only for `rows` a multiple of 64: dimension 0 always spans 64 elements, so
// a partial last atom would read past the end of its row.
bool encode_mn_atoms(CUtensorMap* map, int dtype, const void* base, int64_t rows, int64_t k,
                     int64_t ld, uint32_t atoms) {
    if (rows % 64 != 0 || atoms < 2 || atoms > 4) return false;
    const cuuint64_t dims[3] = {64, (cuuint64_t)k, (cuuint64_t)(rows / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)ld * 2, 128};
    const cuuint32_t box[3] = {64, 64, atoms};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt =
        dtype == TG_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return g_encode(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Two consecutive K-blocks of an operand as one box, for kernels that fill
// two ring slots per barrier transaction: the box lands as the two slots'
// stages back to back, so the pair takes one TMA instruction per operand
// instead of two (each instruction costs TMA throughput).  Only for K a
// multiple of 64: the K-block dimension spans whole blocks.
// K-major operand (`rows` x K, K contiguous): dims {64, rows, K / 64},
// strides {ld, 64} elements, box {64, box_rows, 2}.
bool encode_k_pairs(CUtensorMap* map, int dtype, const void* base, int64_t rows, int64_t k,
                    int64_t ld, uint32_t box_rows) {
    if (k % 64 != 0 || k < 128) return false;
    const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(k / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)ld * 2, 128};
    const cuuint32_t box[3] = {64, box_rows, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt =
        dtype == TG_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return g_encode(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MN-major operand whose stage is `atoms` 64-wide atoms (as encode_mn_atoms),
// two K-blocks per box: dims {64, 64, rows / 64, K / 64}, strides
// {ld, 64, 64 * ld} elements, box {64, 64, atoms, 2}.
bool encode_mn_atom_pairs(CUtensorMap* map, int dtype, const void* base, int64_t rows, int64_t k,
                          int64_t ld, uint32_t atoms) {
    if (rows % 64 != 0 || atoms < 2 || atoms > 4 || k % 64 != 0 || k < 128) return false;
    const cuuint64_t dims[4] = {64, 64, (cuuint64_t)(rows / 64), (cuuint64_t)(k / 64)};
    const cuuint64_t strides[3] = {(cuuint64_t)ld * 2, 128, (cuuint64_t)ld * 2 * 64};
    const cuuint32_t box[4] = {64, 64, atoms, 2};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt =
        dtype == TG_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return g_encode(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

uint32_t make_idesc(int dtype, bool p_mn, bool q_mn, int n, int m) {
    const uint32_t fmt = dtype == TG_BF16 ? 1u : 0u;
    return (1u << 4)                   // accumulator format: fp32
           | (fmt << 7) | (fmt << 10)  // A and B: fp16 or bf16 (always the same type)
           | ((p_mn ? 1u : 0u) << 15) | ((q_mn ? 1u : 0u) << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

}  // namespace

cudaError_t launch_copy_rows(const void* src, long long lds, void* dst, long long ldd,
                             long long rows, long long cols, cudaStream_t stream);

// Operands a tensor map cannot describe (base not 16-byte aligned, or a row
// stride that is not a whole number of 16-byte units) are staged through the
// caller's workspace: copied into aligned dense buffers (A, B, R, bias,
// scale), or, for C, written to one and copied out after the GEMM.
struct Staging {
    bool A = false, B = false, C = false, R = false, bias = false, scale = false;
    size_t bytes = 0;  // staging buffers, each rounded to 256 bytes
    bool any() const { return A || B || C || R || bias || scale; }
};

int64_t up8(int64_t x) { return (x + 7) / 8 * 8; }
size_t dense_bytes(int64_t rows, int64_t width) {
    return ((size_t)rows * (size_t)up8(width) * 2 + 255) / 256 * 256;
}

Staging staging_of(const Args& a) {
    Staging s;
    const int64_t a_rows = a.permA == TG_OP_N ? a.M : a.K, a_w = a.permA == TG_OP_N ? a.K : a.M;
    const int64_t b_rows = a.permB == TG_OP_N ? a.K : a.N, b_w = a.permB == TG_OP_N ? a.N : a.K;
    s.A = !aligned16(a.A) || (a.lda * 2) % 16;
    s.B = !aligned16(a.B) || (a.ldb * 2) % 16;
    s.C = !aligned16(a.C) || (a.ldc * 2) % 16;
    s.R = a.resid && (!aligned16(a.resid) || (a.ldr * 2) % 16);
    s.bias = a.bias && !aligned16(a.bias);
    s.scale = a.scale && !aligned16(a.scale);
    if (s.A) s.bytes += dense_bytes(a_rows, a_w);
    if (s.B) s.bytes += dense_bytes(b_rows, b_w);
    if (s.C) s.bytes += dense_bytes(a.M, a.N);
    if (s.R) s.bytes += dense_bytes(a.M, a.N);
    if (s.bias) s.bytes += dense_bytes(1, a.N);
    if (s.scale) s.bytes += dense_bytes(1, a.M);
    return s;
}

size_t split_bytes(const KernelConfig& cfg) {
    return cfg.sk_tiles > 0 ? ((size_t)cfg.ws_bytes + 255) / 256 * 256 : 0;
}

int gemm_impl(const Args& user, void* workspace, size_t ws_bytes, cudaStream_t stream) {
    int rc = check_shape(user.M, user.N, user.K, user.dtype, user.permA, user.permB, nullptr);
    if (rc) return rc;
    if (user.relu != 0 && user.relu != 1) return TG_ERR_INVALID_ARG;
    if ((rc = check_args(user))) return rc;
    const Staging st = staging_of(user);
    if (st.any() && !workspace) return TG_ERR_ALIGN;  // staging needs the caller's workspace
    int dev;
    DeviceInfo* info;
    if ((rc = current_device(&dev, &info))) return rc;
    load_driver_entry_points();
    if (!g_encode) return TG_ERR_CUDA;
    if ((rc = check_pointers(user, dev))) return rc;

    const KernelConfig cfg = select_config(user.M, user.N, user.K, user.dtype, user.permA,
                                           user.permB,
                                           user.bias != nullptr || user.scale != nullptr ||
                                               user.resid != nullptr || user.relu,
                                           info->sms, workspace != nullptr);
    const size_t sk_bytes = split_bytes(cfg), need = sk_bytes + st.bytes;
    if (need > 0) {
        // The workspace is written: it must be device memory of this device,
        // large enough, and disjoint from every operand.
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return TG_ERR_ALIGN;
        if (ws_bytes < need) return TG_ERR_BUFFER;
        Span ws;
        ws.present = true;
        ws.lo = reinterpret_cast<uintptr_t>(workspace);
        ws.hi = (u128)ws.lo + (u128)need;
        const int64_t a_rows = user.permA == TG_OP_N ? user.M : user.K;
        const int64_t a_w = user.permA == TG_OP_N ? user.K : user.M;
        const int64_t b_rows = user.permB == TG_OP_N ? user.K : user.N;
        const int64_t b_w = user.permB == TG_OP_N ? user.N : user.K;
        const Span others[6] = {span_of(user.C, user.M, user.N, user.ldc),
                                span_of(user.A, a_rows, a_w, user.lda),
                                span_of(user.B, b_rows, b_w, user.ldb),
                                span_of(user.bias, 1, user.N, user.N),
                                span_of(user.scale, 1, user.M, user.M),
                                span_of(user.resid, user.M, user.N, user.ldr)};
        for (const Span& o : others)
            if (intersects(ws, o)) return TG_ERR_OVERLAP;
        if ((rc = check_pointer(workspace, ws, dev))) return rc;
    }
    // Stage what the tensor maps cannot describe (after the split's region).
    Args staged = user;
    if (st.any()) {
        char* cursor = static_cast<char*>(workspace) + sk_bytes;
        auto take = [&](int64_t rows, int64_t width, int64_t* ld) {
            void* d = cursor;
            *ld = up8(width);
            cursor += dense_bytes(rows, width);
            return d;
        };
        auto copy_in = [&](const void* src, int64_t lds, int64_t rows, int64_t width,
                           const void** dst, int64_t* ldd) {
            void* d = take(rows, width, ldd);
            *dst = d;
            return launch_copy_rows(src, lds, d, *ldd, rows, width, stream) == cudaSuccess;
        };
        const int64_t a_rows = user.permA == TG_OP_N ? user.M : user.K;
        const int64_t a_w = user.permA == TG_OP_N ? user.K : user.M;
        const int64_t b_rows = user.permB == TG_OP_N ? user.K : user.N;
        const int64_t b_w = user.permB == TG_OP_N ? user.N : user.K;
        int64_t unused = 0;
        bool ok = true;
        if (st.A) ok = ok && copy_in(user.A, user.lda, a_rows, a_w, &staged.A, &staged.lda);
        if (st.B) ok = ok && copy_in(user.B, user.ldb, b_rows, b_w, &staged.B, &staged.ldb);
        if (st.R) ok = ok && copy_in(user.resid, user.ldr, user.M, user.N, &staged.resid, &staged.ldr);
        if (st.bias) ok = ok && copy_in(user.bias, user.N, 1, user.N, &staged.bias, &unused);
        if (st.scale) ok = ok && copy_in(user.scale, user.M, 1, user.M, &staged.scale, &unused);
        if (st.C) staged.C = take(user.M, user.N, &staged.ldc);
        if (!ok) {
            cudaGetLastError();
            return TG_ERR_CUDA;
        }
    }
    const Args& a = staged;
    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    const bool swap = cfg.swap != 0;
    p.Mk = (int)(swap ? a.N : a.M);
    p.Nk = (int)(swap ? a.M : a.N);
    p.K = (int)a.K;
    p.num_kb = (int)((a.K + 63) / 64);
    p.tiles_m = (p.Mk + cfg.bm - 1) / cfg.bm;
    p.tiles_n = (p.Nk + cfg.bn - 1) / cfg.bn;
    p.num_tiles = p.tiles_m * p.tiles_n;
    p.group_m = cfg.group_m;
    // Which operand storage has the kernel's row (P) / column (Q) index contiguous.
    bool p_mn, q_mn;
    bool ok;
    // Each CTA stages 128 rows of P and q_box columns of Q (half the tile's
    // columns when a CTA pair shares the tile).
    const int q_box = cfg.pair ? cfg.bn / 2 : cfg.bn;
    const void* p_base = swap ? a.B : a.A;
    const void* q_base = swap ? a.A : a.B;
    const int64_t p_ld = swap ? a.ldb : a.lda, q_ld = swap ? a.lda : a.ldb;
    if (!swap) {
        p_mn = a.permA == TG_OP_T;  // A stored K x M
        q_mn = a.permB == TG_OP_N;  // B stored K x N
    } else {
        p_mn = a.permB == TG_OP_N;  // P = B^T: rows n contiguous when B is K x N
        q_mn = a.permA == TG_OP_T;  // Q = A^T: columns m contiguous when A is K x M
    }
    // MN-major stages as one 3-D box where the tile's CTA offsets are whole
    // atoms (P: 128 rows per CTA; Q: q_box columns per CTA), else 2-D boxes.
    p.p_3d = p_mn && encode_mn_atoms(&p.map_p, a.dtype, p_base, p.Mk, a.K, p_ld, 2);
    p.q_3d = q_mn && q_box % 64 == 0 &&
             encode_mn_atoms(&p.map_q, a.dtype, q_base, p.Nk, a.K, q_ld, (uint32_t)(q_box / 64));
    ok = (p.p_3d || encode_operand(&p.map_p, a.dtype, p_base, p.Mk, a.K, p_ld, p_mn, 128)) &&
         (p.q_3d || encode_operand(&p.map_q, a.dtype, q_base, p.Nk, a.K, q_ld, q_mn, q_box));
    // two-K-block boxes for kernels that pair ring slots (whole-tile kernels)
    const bool pairs_slots = cfg.sk_tiles == 0;
    p.p_2k = pairs_slots && !p_mn && encode_k_pairs(&p.map_p2, a.dtype, p_base, p.Mk, a.K, p_ld, 128);
    p.q_2k = p.p_2k && p.q_3d &&
             encode_mn_atom_pairs(&p.map_q2, a.dtype, q_base, p.Nk, a.K, q_ld, (uint32_t)(q_box / 64));
    // C for the epilogue's tensor stores: 32 x 32 chunks, rows of 64 bytes.
    // A tensor store bounds the innermost dimension in 16-byte units, so the
    // map stops at N rounded down to 8 columns; the kernel stores the rest
    // of each row directly (a map of at least 8 columns stays encodable).
    p.n_tma = (int)(a.N & ~int64_t(7));
    ok = ok && encode_2d(&p.map_c, a.dtype, a.C, p.n_tma > 0 ? (uint64_t)p.n_tma : 8u, a.M,
                         a.ldc, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    if (!ok) return TG_ERR_CUDA;
    p.p_mn_major = p_mn;
    p.q_mn_major = q_mn;
    p.idesc = make_idesc(a.dtype, p_mn, q_mn, cfg.bn, cfg.bm);
    p.swap = swap;
    p.bf16 = a.dtype == TG_BF16;
    p.M = (int)a.M;
    p.N = (int)a.N;
    p.C = a.C;
    p.ldc = a.ldc;
    p.bias_n = a.bias;
    p.scale_m = a.scale;
    p.resid = a.resid;
    p.ldr = a.ldr;
    p.relu = a.relu;
    p.workers = cfg.pair ? cfg.grid / 2 : cfg.grid;
    p.sk_tiles = cfg.sk_tiles;
    p.dp_tiles = p.num_tiles - cfg.sk_tiles;
    p.sk_cmax = cfg.sk_cmax;
    p.sk_iters = (long long)cfg.sk_tiles * p.num_kb;
    if (cfg.sk_tiles > 0) {
        const long long counters = sk_counter_bytes(p.workers);
        p.ws_count = static_cast<int*>(workspace);
        p.ws_partial = reinterpret_cast<float*>(static_cast<char*>(workspace) + counters);
    }
    p.timeout_cycles = g_timeout.load();
    p.status = info->status;
    p.inject_skip_load = (int)g_skip_kblock.load();
    cudaError_t e = launch_gemm(p, cfg, info->sms, stream);
    if (e == cudaSuccess && st.C)  // the staged C out to the caller's
        e = launch_copy_rows(staged.C, staged.ldc, user.C, user.ldc, user.M, user.N, stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return TG_ERR_CUDA;
    }
    return TG_OK;
}

}  // namespace tg

using namespace tg;

extern "C" int tg_gemm(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                       tg_perm permA, const void* B, int64_t ldb, tg_perm permB, void* C,
                       int64_t ldc, tg_dtype dtype, const tg_epilogue* epi,
                       cudaStream_t stream) {
    Args a;
    a.M = M;
    a.N = N;
    a.K = K;
    a.A = A;
    a.lda = lda;
    a.permA = (int)permA;
    a.B = B;
    a.ldb = ldb;
    a.permB = (int)permB;
    a.C = C;
    a.ldc = ldc;
    a.dtype = (int)dtype;
    a.bias = epi ? epi->bias_n : nullptr;
    a.scale = epi ? epi->scale_m : nullptr;
    a.resid = epi ? epi->residual : nullptr;
    a.ldr = (epi && epi->residual) ? (epi->ldr ? epi->ldr : ldc) : 0;
    a.relu = epi ? epi->relu : 0;
    return gemm_impl(a, nullptr, 0, stream);
}

extern "C" int tg_gemm_ws(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                          tg_perm permA, const void* B, int64_t ldb, tg_perm permB, void* C,
                          int64_t ldc, tg_dtype dtype, const tg_epilogue* epi, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
    Args a;
    a.M = M;
    a.N = N;
    a.K = K;
    a.A = A;
    a.lda = lda;
    a.permA = (int)permA;
    a.B = B;
    a.ldb = ldb;
    a.permB = (int)permB;
    a.C = C;
    a.ldc = ldc;
    a.dtype = (int)dtype;
    a.bias = epi ? epi->bias_n : nullptr;
    a.scale = epi ? epi->scale_m : nullptr;
    a.resid = epi ? epi->residual : nullptr;
    a.ldr = (epi && epi->residual) ? (epi->ldr ? epi->ldr : ldc) : 0;
    a.relu = epi ? epi->relu : 0;
    return gemm_impl(a, workspace, workspace_bytes, stream);
}

extern "C" int tg_pointwise(int64_t M, int64_t N, const void* X, int64_t ldx, tg_perm permX,
                            void* C, int64_t ldc, tg_dtype dtype, const tg_epilogue* epi,
                            cudaStream_t stream) {
    if (M <= 0 || N <= 0 || M > kMaxDim || N > kMaxDim) return TG_ERR_INVALID_ARG;
    if (permX != TG_OP_N && permX != TG_OP_T) return TG_ERR_INVALID_ARG;
    if (epi && epi->relu != 0 && epi->relu != 1) return TG_ERR_INVALID_ARG;
    if (dtype != TG_F16 && dtype != TG_BF16) return TG_ERR_DTYPE;
    if (!X || !C) return TG_ERR_INVALID_ARG;
    const void* bias = epi ? epi->bias_n : nullptr;
    const void* scale = epi ? epi->scale_m : nullptr;
    const void* resid = epi ? epi->residual : nullptr;
    const int64_t ldr = resid ? (epi->ldr ? epi->ldr : ldc) : 0;
    const int64_t x_rows = permX == TG_OP_N ? M : N, x_w = permX == TG_OP_N ? N : M;
    constexpr int64_t kMaxLd = (1LL << 39) - 8;
    if (ldx < x_w || ldc < N || ldx > kMaxLd || ldc > kMaxLd) return TG_ERR_STRIDE;
    if (resid && (ldr < N || ldr > kMaxLd)) return TG_ERR_STRIDE;
    auto odd = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) != 0; };
    if (odd(X) || odd(C) || odd(bias) || odd(scale) || odd(resid)) return TG_ERR_ALIGN;
    // output storage disjoint from every input (rows of C never overlap: ldc >= N)
    const Span c = span_of(C, M, N, ldc);
    if (intersects(c, span_of(X, x_rows, x_w, ldx)) || intersects(c, span_of(bias, 1, N, N)) ||
        intersects(c, span_of(scale, 1, M, M)) || intersects(c, span_of(resid, M, N, ldr)))
        return TG_ERR_OVERLAP;
    int rc, dev;
    DeviceInfo* info;
    if ((rc = current_device(&dev, &info))) return rc;
    load_driver_entry_points();  // the allocation-range query of check_pointer
    if ((rc = check_pointer(X, span_of(X, x_rows, x_w, ldx), dev)) ||
        (rc = check_pointer(C, c, dev)) || (rc = check_pointer(bias, span_of(bias, 1, N, N), dev)) ||
        (rc = check_pointer(scale, span_of(scale, 1, M, M), dev)) ||
        (rc = check_pointer(resid, span_of(resid, M, N, ldr), dev)))
        return rc;
    PwParams p;
    p.M = (int)M;
    p.N = (int)N;
    p.X = static_cast<const uint16_t*>(X);
    p.ldx = ldx;
    p.C = static_cast<uint16_t*>(C);
    p.ldc = ldc;
    p.scale = static_cast<const uint16_t*>(scale);
    p.bias = static_cast<const uint16_t*>(bias);
    p.R = static_cast<const uint16_t*>(resid);
    p.ldr = ldr;
    p.relu = epi ? epi->relu : 0;
    if (launch_pointwise(p, permX == TG_OP_T, dtype == TG_BF16, info->sms, stream) != cudaSuccess) {
        cudaGetLastError();
        return TG_ERR_CUDA;
    }
    return TG_OK;
}

extern "C" int tg_gemm_workspace_size_ex(int64_t M, int64_t N, int64_t K, const void* A,
                                         int64_t lda, tg_perm permA, const void* B, int64_t ldb,
                                         tg_perm permB, const void* C, int64_t ldc,
                                         tg_dtype dtype, const tg_epilogue* epi, size_t* bytes) {
    int rc = check_shape(M, N, K, (int)dtype, (int)permA, (int)permB, epi);
    if (rc) return rc;
    if (!bytes) return TG_ERR_INVALID_ARG;
    Args a;
    a.M = M;
    a.N = N;
    a.K = K;
    a.A = A;
    a.lda = lda;
    a.permA = (int)permA;
    a.B = B;
    a.ldb = ldb;
    a.permB = (int)permB;
    a.C = const_cast<void*>(C);
    a.ldc = ldc;
    a.dtype = (int)dtype;
    a.bias = epi ? epi->bias_n : nullptr;
    a.scale = epi ? epi->scale_m : nullptr;
    a.resid = epi ? epi->residual : nullptr;
    a.ldr = (epi && epi->residual) ? (epi->ldr ? epi->ldr : ldc) : 0;
    a.relu = epi ? epi->relu : 0;
    if ((rc = check_args(a))) return rc;
    int dev;
    DeviceInfo* info;
    if ((rc = current_device(&dev, &info))) return rc;
    const KernelConfig c = select_config(M, N, K, (int)dtype, (int)permA, (int)permB,
                                         a.bias || a.scale || a.resid || a.relu, info->sms, true);
    *bytes = split_bytes(c) + staging_of(a).bytes;
    return TG_OK;
}

extern "C" int tg_gemm_workspace_size(int64_t M, int64_t N, int64_t K, tg_dtype dtype,
                                      tg_perm permA, tg_perm permB, const tg_epilogue* epi,
                                      size_t* bytes) {
    int rc = check_shape(M, N, K, (int)dtype, (int)permA, (int)permB, epi);
    if (rc) return rc;
    if (!bytes) return TG_ERR_INVALID_ARG;
    int dev;
    DeviceInfo* info;
    if ((rc = current_device(&dev, &info))) return rc;
    const bool has_epi = epi && (epi->bias_n || epi->scale_m || epi->residual || epi->relu);
    const KernelConfig c = select_config(M, N, K, (int)dtype, (int)permA, (int)permB, has_epi,
                                         info->sms, true);
    *bytes = (size_t)c.ws_bytes;
    return TG_OK;
}

namespace tg {
int split_counter_bytes(int64_t M, int64_t N, int64_t K, int dtype, int permA, int permB,
                        bool has_epilogue, size_t* bytes) {
    int rc = check_shape(M, N, K, dtype, permA, permB, nullptr);
    if (rc) return rc;
    int dev;
    DeviceInfo* info;
    if ((rc = current_device(&dev, &info))) return rc;
    const KernelConfig c = select_config(M, N, K, dtype, permA, permB, has_epilogue, info->sms, true);
    *bytes = c.sk_tiles > 0 ? (size_t)sk_counter_bytes(c.pair ? c.grid / 2 : c.grid) : 0;
    return TG_OK;
}
}  // namespace tg

extern "C" const char* tg_status_string(int status) {
    switch (status) {
        case TG_OK: return "TG_OK";
        case TG_ERR_INVALID_ARG: return "TG_ERR_INVALID_ARG";
        case TG_ERR_STRIDE: return "TG_ERR_STRIDE";
        case TG_ERR_ALIGN: return "TG_ERR_ALIGN";
        case TG_ERR_OVERLAP: return "TG_ERR_OVERLAP";
        case TG_ERR_DTYPE: return "TG_ERR_DTYPE";
        case TG_ERR_UNSUPPORTED_DEVICE: return "TG_ERR_UNSUPPORTED_DEVICE";
        case TG_ERR_CUDA: return "TG_ERR_CUDA";
        case TG_ERR_TIMEOUT: return "TG_ERR_TIMEOUT";
        case TG_ERR_POINTER: return "TG_ERR_POINTER";
        case TG_ERR_LAYOUT: return "TG_ERR_LAYOUT";
        case TG_ERR_BUFFER: return "TG_ERR_BUFFER";
        default: return "TG_ERR_UNKNOWN";
    }
}

static int query_config(int stream_k, int64_t M, int64_t N, int64_t K, tg_dtype dtype,
                        tg_perm permA, tg_perm permB, const tg_epilogue* epi, char* buf,
                        size_t len) {
    int rc = check_shape(M, N, K, (int)dtype, (int)permA, (int)permB, epi);
    if (rc) return rc;
    if (!buf) return TG_ERR_INVALID_ARG;
    int dev;
    DeviceInfo* info;
    if ((rc = current_device(&dev, &info))) return rc;
    const bool has_epi = epi && (epi->bias_n || epi->scale_m || epi->residual || epi->relu);
    const KernelConfig c = select_config(M, N, K, (int)dtype, (int)permA, (int)permB, has_epi,
                                         info->sms, stream_k != 0);
    const std::string s = describe_config(c);
    if (s.size() + 1 > len) return TG_ERR_BUFFER;
    std::memcpy(buf, s.c_str(), s.size() + 1);
    return TG_OK;
}

extern "C" int tg_query_config(int64_t M, int64_t N, int64_t K, tg_dtype dtype, tg_perm permA,
                               tg_perm permB, const tg_epilogue* epi, char* buf, size_t len) {
    return query_config(0, M, N, K, dtype, permA, permB, epi, buf, len);
}

extern "C" int tg_query_config_ws(int64_t M, int64_t N, int64_t K, tg_dtype dtype, tg_perm permA,
                                  tg_perm permB, const tg_epilogue* epi, char* buf, size_t len) {
    return query_config(1, M, N, K, dtype, permA, permB, epi, buf, len);
}

extern "C" int tg_query_config_for_sms(int sms, int stream_k, int64_t M, int64_t N, int64_t K,
                                       tg_dtype dtype, tg_perm permA, tg_perm permB,
                                       const tg_epilogue* epi, char* buf, size_t len) {
    int rc = check_shape(M, N, K, (int)dtype, (int)permA, (int)permB, epi);
    if (rc) return rc;
    if (!buf || sms < 2 || sms > 4096) return TG_ERR_INVALID_ARG;
    const bool has_epi = epi && (epi->bias_n || epi->scale_m || epi->residual || epi->relu);
    const KernelConfig c = select_config(M, N, K, (int)dtype, (int)permA, (int)permB, has_epi, sms,
                                         stream_k != 0);
    const std::string s = describe_config(c);
    if (s.size() + 1 > len) return TG_ERR_BUFFER;
    std::memcpy(buf, s.c_str(), s.size() + 1);
    return TG_OK;
}

extern "C" int tg_debug_status(int* detail) {
    int dev;
    DeviceInfo* info;
    int rc = current_device(&dev, &info);
    if (rc) return rc;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return TG_ERR_CUDA;
    }
    int v = 0;
    const int zero = 0;
    if (cudaMemcpy(&v, info->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(info->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return TG_ERR_CUDA;
    }
    if (detail) *detail = v;
    return v == 0 ? TG_OK : TG_ERR_TIMEOUT;
}

extern "C" int tg_debug_configure(int64_t timeout_cycles, int64_t skip_kblock) {
    if (timeout_cycles < 0 || skip_kblock < -1) return TG_ERR_INVALID_ARG;
    g_timeout.store(timeout_cycles == 0 ? kDefaultTimeout : (long long)timeout_cycles);
    g_skip_kblock.store((long long)skip_kblock);
    return TG_OK;
}

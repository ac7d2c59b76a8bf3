// host_pipeline.cpp -- tg_gemm_host: the GEMM with every operand in
// page-locked host memory, the copies overlapped with the arithmetic.
//
// C is cut into blocks of whole output-tile rows.  One copy stream brings B
// (and the broadcast bias), then each block's rows of A, scale and R, into a
// dense device image held in the caller's workspace; the caller's stream runs
// each block's GEMM (tg_gemm_ws) as soon as its rows have arrived; a second
// copy stream returns each block of C while the next blocks are still on
// their way in.  Every block is an ordinary output-tile-aligned sub-GEMM of
// the named-layout computation (ninetoothed.org "Named layouts", section
// "Contract": each output block is owned by one program instance, and the
// blocks are independent), so the pipeline changes when C's rows are
// computed, not what they are.
#include <cuda.h>
#include <cuda_runtime_api.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "../../include/tilegemm.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxBlocks = 64;
constexpr int64_t kMaxDim = 2147483647LL;

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t up8(int64_t x) { return (x + 7) / 8 * 8; }
size_t region(int64_t rows, int64_t width) {  // dense rows x up8(width) 16-bit elements
    return ((size_t)rows * (size_t)up8(width) * 2 + 255) / 256 * 256;
}

// Rows of C per pipelined block: whole 256-row tile pairs, about four blocks.
// Measured at 4096^3 on GB300 (host link about 208 GB/s in, 192 GB/s out,
// about 340 GB/s both ways at once): 1024-row blocks 0.46 ms, 512: 0.47,
// 256: 0.54, one block (no overlap): 0.60.  No C leaves before all of B and
// the first block of A have arrived, and the last block's GEMM and copy-out
// stay exposed: fewer, larger blocks lose overlap; more, smaller ones run
// GEMMs that fill the GPU poorly.  TG_HOST_BLOCK_ROWS (a positive multiple
// of 256) overrides the choice.
int64_t block_rows(int64_t M) {
    if (const char* env = std::getenv("TG_HOST_BLOCK_ROWS")) {
        const long long v = std::atoll(env);
        if (v > 0 && v % 256 == 0) return v;
    }
    int64_t r = cdiv(cdiv(M, 4), 256) * 256;
    if (cdiv(M, r) > kMaxBlocks) r = cdiv(cdiv(M, kMaxBlocks), 256) * 256;
    return r;
}

// Placement of every device image inside the workspace.
struct Plan {
    int64_t rows = 0;       // rows of C per block
    int blocks = 0;
    size_t split = 0;       // stream-K scratch of one compute lane (blocks alternate lanes)
    size_t off_b = 0, off_bias = 0, off_scale = 0, off_a = 0, off_r = 0, off_c = 0;
    size_t bytes = 0;
    int64_t lda = 0, ldb = 0, ldc = 0;  // device image strides (elements)
};

int make_plan(int64_t M, int64_t N, int64_t K, int permA, int permB, int dtype,
              const tg_epilogue* epi, Plan* p) {
    if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return TG_ERR_INVALID_ARG;
    p->rows = block_rows(M);
    p->blocks = (int)cdiv(M, p->rows);
    const int64_t tail = M - (int64_t)(p->blocks - 1) * p->rows;
    size_t full = 0, last = 0;
    int rc = tg_gemm_workspace_size(p->rows < M ? p->rows : M, N, K, (tg_dtype)dtype,
                                    (tg_perm)permA, (tg_perm)permB, epi, &full);
    if (rc) return rc;
    if ((rc = tg_gemm_workspace_size(tail, N, K, (tg_dtype)dtype, (tg_perm)permA, (tg_perm)permB,
                                     epi, &last)))
        return rc;
    p->split = ((full > last ? full : last) + 255) / 256 * 256;
    const int64_t a_rows = permA == TG_OP_N ? M : K, a_w = permA == TG_OP_N ? K : M;
    const int64_t b_rows = permB == TG_OP_N ? K : N, b_w = permB == TG_OP_N ? N : K;
    p->lda = up8(a_w);
    p->ldb = up8(b_w);
    p->ldc = up8(N);
    size_t at = 2 * p->split;
    p->off_b = at;
    at += region(b_rows, b_w);
    p->off_bias = at;
    if (epi && epi->bias_n) at += region(1, N);
    p->off_scale = at;
    if (epi && epi->scale_m) at += region(1, M);
    p->off_a = at;
    at += region(a_rows, a_w);
    p->off_r = at;
    if (epi && epi->residual) at += region(M, N);
    p->off_c = at;
    at += region(M, N);
    p->bytes = at;
    return TG_OK;
}

// Copy stream pair and event pool of one device, made on first use.
struct Pipes {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr, side = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t arrived[kMaxBlocks] = {}, computed[kMaxBlocks] = {};
    std::mutex mu;  // one call enqueues at a time (the events are reused)
};
Pipes g_pipes[kMaxDevices];
std::mutex g_init_mu;

int pipes_of(int dev, Pipes** out) {
    std::lock_guard<std::mutex> lk(g_init_mu);
    Pipes& p = g_pipes[dev];
    if (!p.ready) {
        bool ok = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&p.side, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming) == cudaSuccess &&
                  cudaEventCreateWithFlags(&p.done, cudaEventDisableTiming) == cudaSuccess;
        for (int i = 0; ok && i < kMaxBlocks; ++i)
            ok = cudaEventCreateWithFlags(&p.arrived[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&p.computed[i], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            cudaGetLastError();
            return TG_ERR_CUDA;
        }
        p.ready = true;
    }
    *out = &p;
    return TG_OK;
}

typedef unsigned __int128 u128;

struct Span {  // bytes [lo, hi) of a row-strided 16-bit matrix; empty if absent
    u128 lo = 0, hi = 0;
    bool present = false;
};

Span span_of(const void* p, int64_t rows, int64_t width, int64_t ld) {
    Span s;
    if (!p) return s;
    s.present = true;
    s.lo = (u128)reinterpret_cast<uintptr_t>(p);
    s.hi = s.lo + ((u128)(rows - 1) * (u128)ld + (u128)width) * 2u;
    return s;
}

bool intersects(const Span& a, const Span& b) {
    return a.present && b.present && a.lo < b.hi && b.lo < a.hi;
}

// Page-locked host memory at both ends of the span: the copy engines read
// and write it directly, so the copies stay asynchronous.
bool pinned(const Span& s) {
    if (!s.present) return true;
    for (u128 addr : {s.lo, s.hi - 1}) {
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, reinterpret_cast<const void*>((uintptr_t)addr)) !=
            cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        if (a.type != cudaMemoryTypeHost) return false;
    }
    return true;
}

typedef CUresult (*AddressRangeFn)(CUdeviceptr*, size_t*, CUdeviceptr);
AddressRangeFn g_range = nullptr;
std::once_flag g_range_once;

// [p, p + bytes) inside one device allocation of device `dev`.
bool device_span(const void* p, size_t bytes, int dev) {
    std::call_once(g_range_once, [] {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_range = reinterpret_cast<AddressRangeFn>(fn);
    });
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if ((a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) || a.device != dev)
        return false;
    CUdeviceptr base = 0;
    size_t size = 0;
    if (!g_range || g_range(&base, &size, reinterpret_cast<CUdeviceptr>(p)) != CUDA_SUCCESS)
        return false;
    const u128 lo = (u128)reinterpret_cast<uintptr_t>(p);
    return lo >= (u128)base && lo + bytes <= (u128)base + size;
}

// One strided copy of `rows` rows of `width` 16-bit elements.
bool copy_rows(void* dst, int64_t ldd, const void* src, int64_t lds, int64_t rows,
               int64_t width, cudaMemcpyKind kind, cudaStream_t s) {
    if (rows == 1 || (ldd == width && lds == width))
        return cudaMemcpyAsync(dst, src, (size_t)((rows - 1) * width + width) * 2, kind, s) ==
               cudaSuccess;
    return cudaMemcpy2DAsync(dst, (size_t)ldd * 2, src, (size_t)lds * 2, (size_t)width * 2,
                             (size_t)rows, kind, s) == cudaSuccess;
}

template <typename T>
T* at(void* base, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

}  // namespace

extern "C" int tg_gemm_host_workspace_size(int64_t M, int64_t N, int64_t K, tg_dtype dtype,
                                           tg_perm permA, tg_perm permB, const tg_epilogue* epi,
                                           size_t* bytes) {
    if (!bytes) return TG_ERR_INVALID_ARG;
    Plan p;
    const int rc = make_plan(M, N, K, (int)permA, (int)permB, (int)dtype, epi, &p);
    if (rc) return rc;
    *bytes = p.bytes;
    return TG_OK;
}

extern "C" int tg_gemm_host(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                            tg_perm permA, const void* B, int64_t ldb, tg_perm permB, void* C,
                            int64_t ldc, tg_dtype dtype, const tg_epilogue* epi, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream) {
    // ---- every check before any device work
    if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return TG_ERR_INVALID_ARG;
    if (!A || !B || !C || !workspace) return TG_ERR_INVALID_ARG;
    Plan p;
    int rc = make_plan(M, N, K, (int)permA, (int)permB, (int)dtype, epi, &p);
    if (rc) return rc;  // sizes, enums, dtype, relu, device
    const void* bias = epi ? epi->bias_n : nullptr;
    const void* scale = epi ? epi->scale_m : nullptr;
    const void* resid = epi ? epi->residual : nullptr;
    const int64_t ldr = resid ? (epi->ldr ? epi->ldr : ldc) : 0;
    const int64_t a_rows = permA == TG_OP_N ? M : K, a_w = permA == TG_OP_N ? K : M;
    const int64_t b_rows = permB == TG_OP_N ? K : N, b_w = permB == TG_OP_N ? N : K;
    if (lda < a_w || ldb < b_w || ldc < N || (resid && ldr < N)) return TG_ERR_STRIDE;
    auto odd = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 1u) != 0; };
    if (odd(A) || odd(B) || odd(C) || odd(bias) || odd(scale) || odd(resid) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return TG_ERR_ALIGN;
    const Span c = span_of(C, M, N, ldc);
    const Span ins[5] = {span_of(A, a_rows, a_w, lda), span_of(B, b_rows, b_w, ldb),
                         span_of(bias, 1, N, N), span_of(scale, 1, M, M),
                         span_of(resid, M, N, ldr)};
    Span ws;
    ws.present = true;
    ws.lo = (u128)reinterpret_cast<uintptr_t>(workspace);
    ws.hi = ws.lo + (u128)p.bytes;
    if (intersects(ws, c)) return TG_ERR_OVERLAP;
    for (const Span& s : ins)
        if (intersects(c, s) || intersects(ws, s)) return TG_ERR_OVERLAP;
    if (!pinned(c)) return TG_ERR_POINTER;
    for (const Span& s : ins)
        if (!pinned(s)) return TG_ERR_POINTER;
    if (workspace_bytes < p.bytes) return TG_ERR_BUFFER;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return TG_ERR_UNSUPPORTED_DEVICE;
    }
    if (!device_span(workspace, p.bytes, dev)) return TG_ERR_POINTER;
    Pipes* pp = nullptr;
    if ((rc = pipes_of(dev, &pp))) return rc;
    std::lock_guard<std::mutex> lk(pp->mu);

    // ---- device images inside the workspace
    uint16_t* dB = at<uint16_t>(workspace, p.off_b);
    uint16_t* dbias = bias ? at<uint16_t>(workspace, p.off_bias) : nullptr;
    uint16_t* dscale = scale ? at<uint16_t>(workspace, p.off_scale) : nullptr;
    uint16_t* dA = at<uint16_t>(workspace, p.off_a);
    uint16_t* dR = resid ? at<uint16_t>(workspace, p.off_r) : nullptr;
    uint16_t* dC = at<uint16_t>(workspace, p.off_c);
    const uint16_t* hA = static_cast<const uint16_t*>(A);
    const uint16_t* hR = static_cast<const uint16_t*>(resid);
    const uint16_t* hS = static_cast<const uint16_t*>(scale);
    uint16_t* hC = static_cast<uint16_t*>(C);
    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;

    // Fork: both copy streams start after the work already queued on `stream`.
    bool ok = cudaEventRecord(pp->start, stream) == cudaSuccess &&
              cudaStreamWaitEvent(pp->in, pp->start, 0) == cudaSuccess;
    // Inbound: what every block needs, then each block's rows in order.
    ok = ok && (!bias || copy_rows(dbias, N, bias, N, 1, N, h2d, pp->in));
    ok = ok && copy_rows(dB, p.ldb, B, ldb, b_rows, b_w, h2d, pp->in);
    for (int i = 0; ok && i < p.blocks; ++i) {
        const int64_t r0 = (int64_t)i * p.rows, rows = (M - r0 < p.rows) ? M - r0 : p.rows;
        ok = permA == TG_OP_N
                 ? copy_rows(dA + r0 * p.lda, p.lda, hA + r0 * lda, lda, rows, K, h2d, pp->in)
                 : copy_rows(dA + r0, p.lda, hA + r0, lda, K, rows, h2d, pp->in);
        ok = ok && (!scale || copy_rows(dscale + r0, rows, hS + r0, rows, 1, rows, h2d, pp->in));
        ok = ok && (!resid ||
                    copy_rows(dR + r0 * p.ldc, p.ldc, hR + r0 * ldr, ldr, rows, N, h2d, pp->in));
        ok = ok && cudaEventRecord(pp->arrived[i], pp->in) == cudaSuccess;
    }
    // Each block's GEMM once its rows are in, on two compute lanes in turn
    // (`stream` and a side stream, each with its own stream-K scratch): a
    // block of a few hundred rows fills well under half the SMs, so two run
    // side by side.  Its C goes back on the outbound stream while later
    // blocks compute.
    for (int i = 0; ok && i < p.blocks; ++i) {
        const int64_t r0 = (int64_t)i * p.rows, rows = (M - r0 < p.rows) ? M - r0 : p.rows;
        cudaStream_t lane = (i & 1) ? pp->side : stream;
        tg_epilogue e{};
        e.bias_n = dbias;
        e.scale_m = dscale ? dscale + r0 : nullptr;
        e.relu = epi ? epi->relu : 0;
        e.residual = dR ? dR + r0 * p.ldc : nullptr;
        e.ldr = dR ? p.ldc : 0;
        ok = cudaStreamWaitEvent(lane, pp->arrived[i], 0) == cudaSuccess;
        if (ok) {
            rc = tg_gemm_ws(rows, N, K, permA == TG_OP_N ? dA + r0 * p.lda : dA + r0, p.lda, permA,
                            dB, p.ldb, permB, dC + r0 * p.ldc, p.ldc, dtype, epi ? &e : nullptr,
                            at<void>(workspace, (i & 1) * p.split), p.split, lane);
            ok = rc == TG_OK;
        }
        ok = ok && cudaEventRecord(pp->computed[i], lane) == cudaSuccess &&
             cudaStreamWaitEvent(pp->out, pp->computed[i], 0) == cudaSuccess &&
             copy_rows(hC + r0 * ldc, ldc, dC + r0 * p.ldc, p.ldc, rows, N, d2h, pp->out);
    }
    // Join: `stream` continues after the copy streams and the side lane.
    bool joined = true;
    for (cudaStream_t t : {pp->in, pp->side, pp->out})
        joined = joined && cudaEventRecord(pp->done, t) == cudaSuccess &&
                 cudaStreamWaitEvent(stream, pp->done, 0) == cudaSuccess;
    if (!ok || !joined) {
        cudaGetLastError();
        return rc != TG_OK ? rc : TG_ERR_CUDA;
    }
    return TG_OK;
}

// gemm_kernel.cuh -- persistent, warp-specialised tiled GEMM for sm_103a.
//
// The computation is the tiled matrix multiply of the named-layout GEMM
// (ninetoothed.org "Named layouts"): every output block C[BM, BN] starts from
// a zero fp32 accumulator, adds dot(A_k[BM, 64], B_k[64, BN]) for each of the
// ceil(K / 64) K-blocks, then applies the same-output-domain epilogue
// (row scale, column bias, ReLU, residual) and is stored in the input dtype.
//
// GB300 mapping (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer of A: fills an S-slot ring of 128B-swizzled
//               shared tiles and arms each barrier transaction (one mbarrier
//               "full"/"empty" pair per group of slots).  Tails of M, N and K
//               are zero-filled by the tensor map, so they add 0.
//   warp 6      TMA producer of B into the same transactions.
//   warp 1      owns TMEM; one thread issues tcgen05.mma (K=16 per
//               instruction) into a double-buffered fp32 accumulator.
//   warps 2..5  epilogue: tcgen05.ld 32x32b (thread t of warp w holds TMEM
//               lane 32*(w%4)+t = tile row, register j = tile column), applies
//               the epilogue in fp32, stages each 32 x 32 output chunk in
//               swizzled shared memory and writes it with a TMA tensor store
//               (rows past M and columns past N clipped by the tensor map; a
//               ragged last few columns stored directly), while the next
//               tile's main loop already runs in the other accumulator buffer.
//   warps 0, 1, 6 (once their roles end) and 7 take half of the chunks of a
//               worker's last tile, whose epilogue nothing else overlaps.
// SK = true adds the stream-K tail: tiles of the last, part-empty wave are
// cut into K-ranges dealt out to every worker; contributors publish fp32
// partial sums to a caller workspace and the last to arrive adds them and
// runs the epilogue.
// PAIR = true runs each 256 x BN tile on a cluster of two CTAs with
// tcgen05.mma.cta_group::2: CTA r holds rows 128r..128r+127 of the A block and
// columns r*BN/2 .. (r+1)*BN/2-1 of the B block, so each SM stages half the
// operand bytes of a single-CTA 128 x BN tile per flop.  The leader (rank 0)
// issues the MMAs; both producers signal the leader's "full" barrier, the
// MMA completion is multicast to both CTAs' "empty"/"tmem full" barriers, and
// both epilogues release the accumulator on the leader's "tmem empty".
// Every wait is bounded: after p.timeout_cycles the waiting thread records a
// status code, raises the abort flag of its CTA (and of the peer), every role
// drains what it has in flight (TMA loads, MMAs), TMEM is freed and the
// kernel returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_params.h"
#include "ptx.cuh"

namespace tg {

constexpr int kBK = 64;        // K elements per ring slot: one 128-byte swizzle row of fp16/bf16
// K-blocks per barrier transaction: in whole-tile kernels with tiles wider
// than 64 columns two consecutive ring slots fill and drain together under
// one full/empty barrier pair.  Each transaction has a fixed cost beside its
// bytes (a bare TMA stream of 64 KB transactions measured 64.8 B/clk per SM
// where 32 KB ones reached 39.6): pairs measured +2.5 % at 8192 x 8192 x 4096
// with one producer thread, and still +0.7 % on the fused GEMM with two.
// Stream-K kernels keep one K-block per transaction (pairs measured 2.5-4 %
// slower there with two producer threads), and so do tiles of 32 or 64
// columns, whose stages are small: the bandwidth-bound 32 x 16384 x 16384
// measured 1.5 % faster with one.
template <bool SK, int BN>
struct KBlocksPerStage {
    static constexpr int value = (SK || BN <= 64) ? 1 : 2;
};
constexpr int kUmmaK = 16;     // K per tcgen05.mma of kind::f16
constexpr int kEpiWarps = 4;   // one epilogue warp per TMEM lane quadrant (8 measured no faster overall)
constexpr int kHelper0 = 2 + kEpiWarps;       // second producer (B loads), then a helper with a last item
constexpr int kThreads = 64 + 32 * kEpiWarps + 64;  // producer, MMA, epilogue and helper warps
constexpr int kStageBufs = 4;  // output staging buffers per epilogue warp

template <int BN, bool PAIR>
struct TileShape {
    static constexpr int kBM = PAIR ? 256 : 128;              // rows per tile (whole cluster)
    static constexpr int kBNC = PAIR ? BN / 2 : BN;           // B columns staged per CTA
    static constexpr int kBBoxes = (kBNC + 63) / 64;          // 64-column swizzle atoms
    static constexpr int kAStage = 128 * kBK * 2;             // 16 KB
    static constexpr int kBStage = kBBoxes * 64 * kBK * 2;    // whole atoms
    static constexpr int kStage = kAStage + kBStage;
    // epilogue staging: per epilogue warp kStageBufs 32 x 32 output chunks (2 KB each)
    static constexpr int kStaging = kEpiWarps * kStageBufs * 2048;
    static constexpr int kSmemLimit = 232448;  // opt-in dynamic shared memory per block
    static constexpr int kStagesFit = (kSmemLimit - 1024 - 256 - kStaging) / kStage;
    static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
    static constexpr int kTmemCols = 2 * BN <= 32 ? 32 : 2 * BN <= 64 ? 64 : 2 * BN <= 128 ? 128
                                   : 2 * BN <= 256 ? 256 : 512;
    static constexpr int kSmemBytes = 1024 + kStages * kStage + kStaging + (2 * kStages + 7) * 8 + 16;
    static_assert(kStages >= 4, "too few pipeline stages");
    static_assert(kStages % 2 == 0, "ring slots come in whole barrier groups");
    static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN: multiple of 32 in 32..256");
    static_assert(!PAIR || BN % 32 == 0, "pair tiles split BN in halves of 16-multiples");
};

struct Watch {
    volatile int* abort;
    uint32_t peer_abort;  // shared::cluster address of the peer's flag (PAIR only)
    bool pair;
    int* status;
    long long timeout;
};

__device__ __forceinline__ void raise_abort(const Watch& w, int code) {
    *w.abort = 1;
    if (w.pair) st_shared_cluster_u32(w.peer_abort, 1);
    atomicCAS(w.status, 0, code);
}

// Longest a waiting thread stays suspended inside one try_wait before it
// checks the abort flag and its time limit again.
constexpr uint32_t kSuspendNs = 200000;

// Bounded wait on an mbarrier phase.  Returns false if the CTA is aborting or
// this wait ran out of time (then it raises the abort flags and records `code`).
// The thread sleeps in the try_wait until the phase completes (or for at most
// kSuspendNs), so it takes no issue slots or shared-memory bandwidth while it
// waits.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Watch& w, int code) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_suspend(bar, parity, kSuspendNs)) return true;
        if (*w.abort) return false;
        if (clock64() - t0 > w.timeout) {
            raise_abort(w, code);
            return false;
        }
    }
}

// Bounded wait used while draining after an abort: ignores the abort flag.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, const Watch& w) {
    const long long t0 = clock64();
    while (!mbar_try_wait_suspend(bar, parity, kSuspendNs)) {
        if (clock64() - t0 > w.timeout) return;
    }
}

__device__ __forceinline__ void tile_coords(const GemmParams& p, int t, int& tm, int& tn) {
    const int group_size = p.group_m * p.tiles_n;
    const int g = t / group_size;
    const int first = g * p.group_m;
    const int gm = min(p.tiles_m - first, p.group_m);
    const int r = t - g * group_size;
    tm = first + r % gm;
    tn = r / gm;
}

__device__ __forceinline__ float to_f32(uint16_t h, int bf16) {
    return bf16 ? __bfloat162float(__ushort_as_bfloat16(h)) : __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ uint16_t from_f32(float x, int bf16) {
    return bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(x)) : __half_as_ushort(__float2half_rn(x));
}

// Two floats -> one word of two 16-bit values with round-to-nearest-even, for
// a dtype fixed at compile time.
template <bool BF>
__device__ __forceinline__ uint32_t pack2t(float a, float b) {
    uint32_t w;
    if constexpr (BF) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        w = *reinterpret_cast<uint32_t*>(&h);
    } else {
        __half2 h = __floats2half2_rn(a, b);
        w = *reinterpret_cast<uint32_t*>(&h);
    }
    return w;
}

// y[0], y[1] += the two 16-bit values of w (low half first).  Each is added
// by one mixed-precision add: the 16-bit operand is widened exactly and the
// fp32 sum rounded once to nearest, the same result as converting first,
// without the conversion instructions.
template <bool BF>
__device__ __forceinline__ void add2_wide(float* y, uint32_t w) {
    if constexpr (BF)
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
            : "+f"(y[0]), "+f"(y[1])
            : "r"(w));
    else
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
            : "+f"(y[0]), "+f"(y[1])
            : "r"(w));
}

// y[0], y[1] *= s as one packed fp32x2 multiply (round to nearest): half the
// multiply instructions of the epilogue warps.
__device__ __forceinline__ void mul2(float* y, float s) {
    unsigned long long a, b;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(y[0]), "f"(y[1]));
    asm("mov.b64 %0, {%1, %1};" : "=l"(b) : "f"(s));
    asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(a) : "l"(b));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(y[0]), "=f"(y[1]) : "l"(a));
}

// y[0], y[1] += x0, x1 as one packed fp32x2 add (round to nearest).
__device__ __forceinline__ void add2(float* y, float x0, float x1) {
    unsigned long long a, b;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(y[0]), "f"(y[1]));
    asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(x0), "f"(x1));
    asm("add.rn.f32x2 %0, %0, %1;" : "+l"(a) : "l"(b));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(y[0]), "=f"(y[1]) : "l"(a));
}

// v[i] for a run-time i without indexing the array (which would put it in
// local memory): N selects, N <= 8.
template <int N>
__device__ __forceinline__ float pick(const float (&v)[N], int i) {
    float r = 0.0f;
#pragma unroll
    for (int k = 0; k < N; ++k) r = k == i ? v[k] : r;
    return r;
}

template <bool BF>
__device__ __forceinline__ void add8(const uint4& u, float* y) {
    add2_wide<BF>(y, u.x);
    add2_wide<BF>(y + 2, u.y);
    add2_wide<BF>(y + 4, u.z);
    add2_wide<BF>(y + 6, u.w);
}

// Residual values of one full 32-column run of row m, loaded one run ahead
// (and before the accumulator is ready) so that their latency overlaps the
// work on the run before.
struct Aux {
    uint4 r[4];
};

// Issues the residual loads for the run C(m, c0 .. c0+31) if it is full and
// inside C; returns whether it is (otherwise the chunk takes the masked
// scalar path).
// Residual lines are read exactly once: `pol` marks them first to leave L2,
// so they do not push operand panels out (measured +0.3 % on the fused GEMM).
__device__ __forceinline__ bool prefetch_aux(const GemmParams& p, int m, int c0, Aux& a,
                                             uint64_t pol) {
    if (p.swap || m >= p.M || c0 + 32 > p.N) return false;
    if (p.resid) {
        const uint4* r = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.resid) +
                                                        (long long)m * p.ldr + c0);
#pragma unroll
        for (int v = 0; v < 4; ++v) a.r[v] = ld_nc_hint(r + v, pol);
    }
    return true;
}

// Epilogue arithmetic for the run C(m, c0 .. c0+31) held in y[], in fp32:
// scale, bias, ReLU, residual.  Called by all 32 lanes of a warp together
// (lane = row): lane j holds in `bias_lane` the bias of column c0 + j (0
// outside C), which shuffles hand to every row; `add_bias` is false where
// the caller holds no bias (the plain epilogue: no bias step compiled in).
// `a` holds the prefetched residual of a full in-bounds run; otherwise (edge
// runs) it is loaded here with per-element masks.  Values outside C are
// computed but never stored.
template <bool BF>
__device__ __forceinline__ void epilogue_math(const GemmParams& p, int m, int c0, float (&y)[32],
                                              float row_scale, float bias_lane, bool add_bias,
                                              const Aux* a) {
    const bool inside = m < p.M && c0 < p.N;
    const bool full = inside && c0 + 32 <= p.N;
    if (p.scale_m) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) mul2(y + j, row_scale);
    }
    if (p.bias_n && add_bias) {
#pragma unroll
        for (int j = 0; j < 32; j += 2)
            add2(y + j, __shfl_sync(0xffffffffu, bias_lane, j), __shfl_sync(0xffffffffu, bias_lane, j + 1));
    }
    if (p.relu) {
#pragma unroll
        for (int j = 0; j < 32; ++j) y[j] = fmaxf(y[j], 0.0f);
    }
    if (p.resid && inside) {
        const uint16_t* r = static_cast<const uint16_t*>(p.resid) + (long long)m * p.ldr + c0;
        if (full) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
                add8<BF>(a ? a->r[v] : __ldg(reinterpret_cast<const uint4*>(r) + v), y + 8 * v);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (c0 + j < p.N) y[j] += to_f32(r[j], BF);
        }
    }
}

// Writes row `r` (0..31) of a 32 x 32 output chunk into its staging buffer:
// 64-byte rows in the 64-byte XOR swizzle the C tensor map uses (16-byte
// chunk index XOR (r / 2) mod 4), so the 32 lanes of a warp spread every
// store over all banks.
template <bool BF>
__device__ __forceinline__ void stage_row(uint8_t* buf, int r, const float (&y)[32]) {
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        uint4 u;
        u.x = pack2t<BF>(y[8 * v + 0], y[8 * v + 1]);
        u.y = pack2t<BF>(y[8 * v + 2], y[8 * v + 3]);
        u.z = pack2t<BF>(y[8 * v + 4], y[8 * v + 5]);
        u.w = pack2t<BF>(y[8 * v + 6], y[8 * v + 7]);
        *reinterpret_cast<uint4*>(buf + r * 64 + ((v ^ ((r >> 1) & 3)) << 4)) = u;
    }
}

// One warp stores its 32 x 32 chunk C(row0.., c0..) through shared memory
// with a TMA tensor store.  The tensor store clips rows at M and columns at
// n_tma = N rounded down to 8 (it bounds the innermost dimension in whole
// 16-byte units); the few columns [n_tma, N) of a row are stored directly.
// kStageBufs staging buffers per warp rotate; `count` is the warp's running
// chunk number.
template <bool BF>
__device__ __forceinline__ void store_chunk(const GemmParams& p, uint8_t* stage, uint32_t& count,
                                            int lane, int row0, int c0, const float (&y)[32]) {
    uint8_t* buf = stage + (count % kStageBufs) * 2048;
    if (count >= kStageBufs && lane == 0)
        bulk_wait_group_read<kStageBufs - 1>();  // its previous store has read it
    __syncwarp();
    stage_row<BF>(buf, lane, y);
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
        // output lines are written once: first to leave L2, ahead of operand panels
        if (row0 < p.M && c0 < p.n_tma)
            tma_store_2d_hint(&p.map_c, smem_addr(buf), c0, row0, l2_policy_evict_first());
        bulk_commit_group();
    }
    if (c0 + 32 > p.n_tma && c0 < p.N && row0 + lane < p.M) {
        uint16_t* c = static_cast<uint16_t*>(p.C) + (long long)(row0 + lane) * p.ldc;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (c0 + j >= p.n_tma && c0 + j < p.N) c[c0 + j] = from_f32(y[j], BF);
    }
    ++count;
}

// Epilogue arithmetic and store of one 32-column chunk, with the element type
// resolved once per chunk (instead of per element).
__device__ __forceinline__ void finish_chunk(const GemmParams& p, uint8_t* stage, uint32_t& count,
                                             int lane, int rk, int row0, int c0, float (&y)[32],
                                             float row_scale, float bias_lane, bool add_bias,
                                             const Aux* a) {
    if (p.bf16) {
        epilogue_math<true>(p, rk, c0, y, row_scale, bias_lane, add_bias, a);
        store_chunk<true>(p, stage, count, lane, row0, c0, y);
    } else {
        epilogue_math<false>(p, rk, c0, y, row_scale, bias_lane, add_bias, a);
        store_chunk<false>(p, stage, count, lane, row0, c0, y);
    }
}

// Epilogue of the swapped (transposed-output) layout for one 32-column chunk:
// kernel row rk is C's column n, kernel column c0+j is C's row m.  Lanes of a
// warp hold consecutive n, so every store instruction writes one contiguous
// run of a C row.
__device__ __forceinline__ void epilogue_swap(const GemmParams& p, int rk, int c0,
                                              const float (&y)[32], float row_bias) {
    const int bf = p.bf16;
    const int n = rk;
    if (n >= p.N) return;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const int m = c0 + j;
        if (m >= p.M) continue;
        float v = y[j];
        if (p.scale_m) v *= to_f32(static_cast<const uint16_t*>(p.scale_m)[m], bf);
        if (p.bias_n) v += row_bias;
        if (p.relu) v = fmaxf(v, 0.0f);
        if (p.resid) v += to_f32(static_cast<const uint16_t*>(p.resid)[(long long)m * p.ldr + n], bf);
        static_cast<uint16_t*>(p.C)[(long long)m * p.ldc + n] = from_f32(v, bf);
    }
}

// The work items of one persistent worker.  Its whole tiles are w, w +
// workers, ... below dp_tiles; its stream-K iterations are one contiguous
// range, cut at tile boundaries into (tile, k-block range) pieces.  Order: all
// whole tiles but the last, then the range, then the last whole tile.  So a
// worker ends on a whole tile, whose epilogue the helper warps halve, and the
// fix-ups of split tiles run beside that tile's main loop.  (With the range
// last, the worker finishing a split tile did so in its final item, queued
// behind the previous tile's epilogue: 4096^3 measured 1-2 % slower.)
struct WorkIter {
    int workers, dp_tiles, num_kb, dp_next, dp_left;
    long long it, it_end;

    __device__ __forceinline__ WorkIter(const GemmParams& p, int worker)
        : workers(p.workers), dp_tiles(p.dp_tiles), num_kb(p.num_kb), dp_next(worker),
          dp_left(worker < p.dp_tiles ? (p.dp_tiles - worker + p.workers - 1) / p.workers : 0),
          it(p.sk_iters * worker / p.workers), it_end(p.sk_iters * (worker + 1) / p.workers) {}

    __device__ __forceinline__ bool next(int& tile, int& kb0, int& kb1) {
        if (dp_left > 1 || (dp_left == 1 && it >= it_end)) {
            --dp_left;
            tile = dp_next;
            kb0 = 0;
            kb1 = num_kb;
            dp_next += workers;
            return true;
        }
        if (it < it_end) {
            const long long ts = it / num_kb;
            tile = dp_tiles + (int)ts;
            kb0 = (int)(it - ts * num_kb);
            const long long left = it_end - it;
            kb1 = (int)(left < (long long)(num_kb - kb0) ? kb0 + left : num_kb);
            it += kb1 - kb0;
            return true;
        }
        return false;
    }
};

// Compile-time role of a producer thread.
template <int V>
struct RoleTag {
    static constexpr int value = V;
};

// Worker whose stream-K range holds iteration `it`.
__device__ __forceinline__ int sk_owner(const GemmParams& p, long long it) {
    int w = (int)(it * p.workers / p.sk_iters);
    while (w + 1 < p.workers && p.sk_iters * (w + 1) / p.workers <= it) ++w;
    while (w > 0 && p.sk_iters * w / p.workers > it) --w;
    return w;
}

// Named barrier over the four epilogue warps that also ANDs a flag: every
// epilogue thread leaves with the same decision.
__device__ __forceinline__ int epilogue_sync_and(int v) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.and.pred po, 1, %2, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)v), "n"(32 * kEpiWarps)
        : "memory");
    return (int)out;
}

// AUX = true: the epilogue reads a bias and/or residual: the bias once per
// tile, the residual one 32-column run ahead (both issued before the
// accumulator is ready).
// AUX = false keeps the plain epilogue lean.
// SK = true: the launch deals tail tiles out in K-ranges (the stream-K code is
// compiled only into these instantiations; whole-tile kernels stay lean).
template <int BN, bool PAIR, bool AUX, bool SK>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
    using TS = TileShape<BN, PAIR>;
    constexpr int STAGES = TS::kStages;
    constexpr int kKPerStage = KBlocksPerStage<SK, BN>::value;
    constexpr int CG = PAIR ? 2 : 1;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128B-swizzle atoms (same offset in both CTAs of a pair)
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * TS::kAStage;
    uint8_t* staging = sB + STAGES * TS::kBStage;  // epilogue output chunks (1024-aligned)
    uint64_t* bars = reinterpret_cast<uint64_t*>(staging + TS::kStaging);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint64_t* hsync = drain + 1;     // a last split tile's fix-up decision, for the helper warps
    uint64_t* lastfull = hsync + 1;  // the worker's last accumulator is complete (one phase)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(lastfull + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* sk_last = reinterpret_cast<volatile int*>(tmem_slot + 2);
    volatile int* sk_help = reinterpret_cast<volatile int*>(tmem_slot + 3);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0;
    const bool leader = rank == 0;
    const int worker = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const Watch w{abort_flag,
                  PAIR ? mapa_shared(smem_addr((const void*)abort_flag), rank ^ 1u) : 0u, PAIR,
                  p.status, p.timeout_cycles};

    if (threadIdx.x == 0) {
        prefetch_tensormap(&p.map_p);
        prefetch_tensormap(&p.map_q);
        prefetch_tensormap(&p.map_c);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&tfull[b]), 1);
            mbar_init(smem_addr(&tempty[b]), (PAIR ? 2 : 1) * kEpiWarps);  // one per epilogue warp
        }
        mbar_init(smem_addr(drain), 1);
        mbar_init(smem_addr(hsync), 1);
        mbar_init(smem_addr(lastfull), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_addr(tmem_slot), TS::kTmemCols);
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    if constexpr (PAIR)
        cluster_sync();  // the peer's barriers exist before anyone signals them
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // ------------------------------------------------------ TMA producers
    // Two threads fill the ring: role 1 (warp 0) arms each barrier
    // transaction with both operands' bytes and loads P (A); role 2 (warp
    // kHelper0, idle until the last tile's epilogue) loads Q (B) into the same
    // transaction.  A Q load may complete before the transaction is armed: the
    // phase cannot complete while the arming arrival is pending.  The single
    // producer thread's loop was on the critical path of the main loop.
    auto run_producer = [&](auto role) {
        constexpr int ROLE = decltype(role)::value;
        // Slots are filled kKPerStage at a time: group q holds slots
        // q*kKPerStage.. and one full/empty barrier pair; a work item's last
        // group may hold fewer K-blocks.
        constexpr int GROUPS = STAGES / kKPerStage;
        int grp = 0;
        uint32_t phase = 0;
        uint32_t armed = 0, armed_parity = 0;
        long long g = 0;
        bool ok = true;
        // bytes this CTA lands per K-block (A half + its B columns)
        const uint32_t a_bytes = TS::kAStage;
        const uint32_t b_bytes = p.q_mn_major ? (uint32_t)TS::kBStage : (uint32_t)TS::kBNC * 128u;
        const uint32_t stage_tx = (a_bytes + b_bytes) * (PAIR ? 2u : 1u);
        const bool both_2k = p.p_2k && p.q_2k;  // both operands have two-K-block maps
        WorkIter items(p, worker);
        int t, kb0, kb1;
        while (ok && items.next(t, kb0, kb1)) {
            int tm, tn;
            tile_coords(p, t, tm, tn);
            const int m0 = tm * TS::kBM + (int)rank * 128;
            const int n0 = tn * BN + (int)rank * TS::kBNC;
            for (int kb = kb0; kb < kb1; kb += kKPerStage) {
                const int n = kb1 - kb < kKPerStage ? kb1 - kb : kKPerStage;
                if (!wait_bar(smem_addr(&empty[grp]), phase ^ 1, w, DEV_TIMEOUT_PRODUCER)) {
                    ok = false;
                    break;
                }
                if (p.inject_skip_load < g || p.inject_skip_load >= g + n) {
                    const uint32_t fb_local = smem_addr(&full[grp]);
                    if (ROLE == 1 && leader) {
                        mbar_arrive_expect_tx(fb_local, stage_tx * (uint32_t)n);
                        armed |= 1u << grp;
                        armed_parity = (armed_parity & ~(1u << grp)) | (phase << grp);
                    }
                    const uint32_t fb = PAIR ? mapa_shared(fb_local, 0) : fb_local;
                    if (kKPerStage == 2 && n == 2 && both_2k) {
                        // both K-blocks of each operand as one box
                        const uint32_t a_dst = smem_addr(sA + grp * kKPerStage * TS::kAStage);
                        const uint32_t b_dst = smem_addr(sB + grp * kKPerStage * TS::kBStage);
                        if constexpr (ROLE == 1) {
                            if constexpr (PAIR)
                                tma_load_3d_pair(a_dst, &p.map_p2, fb, 0, m0, kb);
                            else
                                tma_load_3d(a_dst, &p.map_p2, fb, 0, m0, kb);
                        } else {
                            if constexpr (PAIR)
                                tma_load_4d_pair(b_dst, &p.map_q2, fb, 0, 0, n0 >> 6, kb);
                            else
                                tma_load_4d(b_dst, &p.map_q2, fb, 0, 0, n0 >> 6, kb);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < kKPerStage; ++j) {
                            if (j >= n) break;
                            const int slot = grp * kKPerStage + j;
                            const uint32_t a_dst = smem_addr(sA + slot * TS::kAStage);
                            const uint32_t b_dst = smem_addr(sB + slot * TS::kBStage);
                            const int k0 = (kb + j) * kBK;
                            if constexpr (ROLE == 1) {
                            if (p.p_3d) {
                                if constexpr (PAIR)
                                    tma_load_3d_pair(a_dst, &p.map_p, fb, 0, k0, m0 >> 6);
                                else
                                    tma_load_3d(a_dst, &p.map_p, fb, 0, k0, m0 >> 6);
                            } else if (p.p_mn_major) {
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    if constexpr (PAIR)
                                        tma_load_2d_pair(a_dst + h * 8192, &p.map_p, fb, m0 + 64 * h, k0);
                                    else
                                        tma_load_2d(a_dst + h * 8192, &p.map_p, fb, m0 + 64 * h, k0);
                                }
                            } else {
                                if constexpr (PAIR)
                                    tma_load_2d_pair(a_dst, &p.map_p, fb, k0, m0);
                                else
                                    tma_load_2d(a_dst, &p.map_p, fb, k0, m0);
                            }
                            } else {
                            if (p.q_3d) {
                                if constexpr (PAIR)
                                    tma_load_3d_pair(b_dst, &p.map_q, fb, 0, k0, n0 >> 6);
                                else
                                    tma_load_3d(b_dst, &p.map_q, fb, 0, k0, n0 >> 6);
                            } else if (p.q_mn_major) {
#pragma unroll
                                for (int h = 0; h < TS::kBBoxes; ++h) {
                                    if constexpr (PAIR)
                                        tma_load_2d_pair(b_dst + h * 8192, &p.map_q, fb, n0 + 64 * h, k0);
                                    else
                                        tma_load_2d(b_dst + h * 8192, &p.map_q, fb, n0 + 64 * h, k0);
                                }
                            } else {
                                if constexpr (PAIR)
                                    tma_load_2d_pair(b_dst, &p.map_q, fb, k0, n0);
                                else
                                    tma_load_2d(b_dst, &p.map_q, fb, k0, n0);
                            }
                            }
                        }
                    }
                }
                g += n;
                if (++grp == GROUPS) {
                    grp = 0;
                    phase ^= 1;
                }
            }
        }
        if (*abort_flag) {
            // No TMA write may land after the CTA exits: wait for the last
            // armed phase of every group (the leader's barriers count the
            // bytes of both CTAs).
            for (int q = 0; q < GROUPS; ++q)
                if (armed & (1u << q)) drain_bar(smem_addr(&full[q]), (armed_parity >> q) & 1, w);
        }
    };
    if (warp == 0 && lane == 0) {
        run_producer(RoleTag<1>{});
    } else if (warp == kHelper0 && lane == 0) {
        run_producer(RoleTag<2>{});
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------ MMA issuer
            constexpr int GROUPS = STAGES / kKPerStage;
            int grp = 0;
            uint32_t phase = 0;
            bool ok = true;
            int i = 0;
            // One thread issues every MMA, so the instructions between two
            // MMAs are on the critical path of the tensor pipe: the operand
            // descriptors are built once here, and a K step or a stage step
            // is a 32-bit add on their low words.  K-major operands step 16
            // elements = 32 bytes inside the swizzle row (LBO unused);
            // MN-major ones step 16 K-rows of 128 bytes, with LBO = 8 KB to
            // the next 64-wide atom.
            const uint32_t idesc = p.idesc;
            const uint32_t d_hi = smem_desc_hi_sw128(1024);
            const uint32_t a_lo0 = smem_desc_lo(smem_addr(sA), p.p_mn_major ? 8192u : 16u);
            const uint32_t b_lo0 = smem_desc_lo(smem_addr(sB), p.q_mn_major ? 8192u : 16u);
            const uint32_t a_kstep = p.p_mn_major ? (2048u >> 4) : (32u >> 4);
            const uint32_t b_kstep = p.q_mn_major ? (2048u >> 4) : (32u >> 4);
            WorkIter items(p, worker);
            int t, kb0, kb1;
            for (; ok && items.next(t, kb0, kb1); ++i) {
                const int buf = i & 1;
                const uint32_t aph = (i >> 1) & 1;
                if (!wait_bar(smem_addr(&tempty[buf]), aph ^ 1, w, DEV_TIMEOUT_MMA + 1)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int kb = kb0; kb < kb1; kb += kKPerStage) {
                    const int n = kb1 - kb < kKPerStage ? kb1 - kb : kKPerStage;
                    if (!wait_bar(smem_addr(&full[grp]), phase, w, DEV_TIMEOUT_MMA + 2)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < kKPerStage; ++j) {
                        if (j >= n) break;
                        const uint32_t slot = (uint32_t)(grp * kKPerStage + j);
                        const uint32_t a_lo = a_lo0 + slot * (TS::kAStage >> 4);
                        const uint32_t b_lo = b_lo0 + slot * (TS::kBStage >> 4);
#pragma unroll
                        for (int kk = 0; kk < kBK / kUmmaK; ++kk)
                            mma_f16<CG>(d_tmem, smem_desc_join(a_lo + kk * a_kstep, d_hi),
                                        smem_desc_join(b_lo + kk * b_kstep, d_hi), idesc,
                                        (kb + j != kb0) || (kk != 0));
                    }
                    // frees the group's slots (in both CTAs) once the MMAs have read them
                    if constexpr (PAIR)
                        mma_commit_pair(smem_addr(&empty[grp]), 0x3);
                    else
                        mma_commit(smem_addr(&empty[grp]));
                    if (++grp == GROUPS) {
                        grp = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                // accumulator complete (in both CTAs' TMEM)
                if constexpr (PAIR)
                    mma_commit_pair(smem_addr(&tfull[buf]), 0x3);
                else
                    mma_commit(smem_addr(&tfull[buf]));
                // the last item's, again on a one-shot barrier for the helper
                // warps (a parity wait on tfull could alias an earlier phase)
                WorkIter peek = items;
                int t2, a2, b2;
                if (!peek.next(t2, a2, b2)) {
                    if constexpr (PAIR)
                        mma_commit_pair(smem_addr(lastfull), 0x3);
                    else
                        mma_commit(smem_addr(lastfull));
                }
            }
            // Nothing may still write TMEM when it is released.
            if constexpr (PAIR)
                mma_commit_pair_local(smem_addr(drain));
            else
                mma_commit(smem_addr(drain));
            drain_bar(smem_addr(drain), 0, w);
        }
    }

    // -------------------------------------------------------- epilogue
    // Warps 2 .. 1 + kEpiWarps finish every work item, one per TMEM lane
    // quadrant.  Nothing overlaps the epilogue of a worker's last item, so
    // that one is split with a second warp per quadrant (a "helper"): warps
    // 0, 1 and kHelper0 once their producer / MMA roles are done, and warp
    // kHelper0 + 1, which waits for it from the start.  A helper takes the
    // second half of its quadrant's chunks and stages them in the operand
    // ring, which no load or MMA touches once the last accumulator is
    // complete.  Helpers meet the main warps at no named barrier: they learn
    // a split tile's fix-up decision through the mbarrier `hsync`, with
    // bounded waits, so an aborting CTA cannot strand them.
    __syncwarp();  // the lanes of warps 0, 1 and kHelper0 wait for their role's lane 0
    {
        const bool helper = warp < 2 || warp >= kHelper0;
        const int q = warp & 3;  // TMEM lane quadrant this warp may read
        // the warps of a quadrant (kEpiWarps / 4 of them) split the tile's
        // 32-column chunks
        constexpr int kChunks = BN / 32;
        constexpr int kPerQuadrant = kEpiWarps / 4;
        const int part = helper ? 0 : (warp - 2) / 4;
        const int c_begin = part * kChunks / kPerQuadrant;
        const int c_end = (part + 1) * kChunks / kPerQuadrant;
        // this warp's output buffers
        uint8_t* stage = helper ? sA + q * kStageBufs * 2048 : staging + (warp - 2) * kStageBufs * 2048;
        const uint64_t pol = AUX ? l2_policy_evict_first() : 0;     // residual lines are read once
        uint32_t chunks = 0;                           // output chunks stored so far
        int i = 0;
        WorkIter items(p, worker);
        int t, kb0, kb1;
        for (; items.next(t, kb0, kb1); ++i) {
            bool last_item;
            {
                WorkIter peek = items;
                int t2, a2, b2;
                last_item = !peek.next(t2, a2, b2);
            }
            if (helper && !last_item) continue;
            // this warp's chunks of a tile it finishes: all of its quadrant's,
            // or for a last item the main warp's first half, the helper's second
            const int mid = c_begin + (c_end - c_begin + 1) / 2;
            const int cb = last_item && helper ? mid : c_begin;
            const int ce = last_item && !helper ? mid : c_end;
            const int buf = i & 1;
            const uint32_t aph = (i >> 1) & 1;
            int tm, tn;
            tile_coords(p, t, tm, tn);
            const int rk = tm * TS::kBM + (int)rank * 128 + q * 32 + lane;
            const bool whole = !SK || (kb0 == 0 && kb1 == p.num_kb);
            // Lane j's bias of column j of each of this warp's chunks, loaded
            // once per tile before the accumulator wait; a chunk hands them
            // to its rows by shuffles.  (A broadcast load of each chunk's 32
            // values, one chunk ahead, sat in the epilogue's dependent chain:
            // 4096 x 3136 x 1024 with a bias ran 10 % slower than without.)
            float bcol[kChunks];
#pragma unroll
            for (int k = 0; k < kChunks; ++k) bcol[k] = 0.0f;
            if constexpr (AUX) {
                if (p.bias_n && !p.swap) {
                    const uint16_t* bv = static_cast<const uint16_t*>(p.bias_n);
#pragma unroll
                    for (int k = 0; k < kChunks; ++k) {
                        const int n = tn * BN + k * 32 + lane;
                        if (k >= cb && k < ce && n < p.N) bcol[k] = to_f32(bv[n], p.bf16);
                    }
                }
            }
            // the residual of the first run does not depend on the
            // accumulator: fetch it while the main loop still runs.  (Moving
            // the later runs' residual rows into L2 here as well measured
            // 1.2 % slower on the fused GEMM: they evict operand lines.)
            Aux cur, nxt;
            bool cur_full = (AUX && whole && cb < ce) ? prefetch_aux(p, rk, tn * BN + cb * 32, cur, pol) : false;
            int ok = 1;
            if (lane == 0) {
                if (!helper) {
                    ok = wait_bar(smem_addr(&tfull[buf]), aph, w, DEV_TIMEOUT_EPILOGUE);
                } else {
                    // A helper waits for the last item from the start, on a
                    // one-shot barrier; its time limit covers every item
                    // before it (each of which the main warps wait for within
                    // one limit).
                    Watch wt = w;
                    wt.timeout = w.timeout * (long long)(i + 1);
                    ok = wait_bar(smem_addr(lastfull), 0, wt, DEV_TIMEOUT_EPILOGUE + 3);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!helper) {
                ok = epilogue_sync_and(ok);  // all main warps continue, or all stop
            } else if (ok) {
                drain_bar(smem_addr(lastfull), 0, w);  // complete: every lane observes it
                fence_proxy_async_shared();  // the buffers last held TMA-written operands
            }
            if (!ok) break;
            tc_fence_after();
            float row_scale = 1.0f, row_bias = 0.0f;
            if (!p.swap) {
                if (p.scale_m && rk < p.M) row_scale = to_f32(static_cast<const uint16_t*>(p.scale_m)[rk], p.bf16);
            } else {
                if (p.bias_n && rk < p.N) row_bias = to_f32(static_cast<const uint16_t*>(p.bias_n)[rk], p.bf16);
            }
            const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN;
            const int row0 = tm * TS::kBM + (int)rank * 128 + q * 32;  // this warp's first row
            if (!helper && c_begin == c_end) {
                // no columns for this warp (narrow tile): release the buffer at once
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR)
                        mbar_arrive_cluster(smem_addr(&tempty[buf]), 0);
                    else
                        mbar_arrive(smem_addr(&tempty[buf]));
                }
            }
            if (SK && !whole) {
                // ---- stream-K part of tile t: publish this worker's partial sum
                const long long f = (long long)(t - p.dp_tiles) * p.num_kb;
                const int wf = sk_owner(p, f), wl = sk_owner(p, f + p.num_kb - 1);
                const int contributors = wl - wf + 1, mine = worker - wf;
                // slot k of this tile and CTA: 128 rows x BN fp32 stored as
                // [BN/4][128 rows][4], so that the 32 lanes of a warp (32
                // consecutive rows) move 512 contiguous bytes per access
                const size_t slot = (size_t)TS::kBM * BN;
                float* base = p.ws_partial + (size_t)wf * p.sk_cmax * slot +
                              (size_t)rank * 128 * BN + (size_t)(q * 32 + lane) * 4;
                int* counter = p.ws_count + wf * 2 + rank;
                bool last;
                if (helper) {
                    // the main warps' decision: finish the tile (1) or not (0)
                    int got = 1;
                    if (lane == 0) got = wait_bar(smem_addr(hsync), 0, w, DEV_TIMEOUT_EPILOGUE + 2);
                    if (!__shfl_sync(0xffffffffu, got, 0)) break;
                    drain_bar(smem_addr(hsync), 0, w);  // every lane observes it (acquire)
                    last = *sk_help != 0;
                    if (!last) continue;
                } else {
                    // If every other part is already published this worker finishes
                    // the tile at once and never writes its own partial.
                    if (warp == 2 && lane == 0) {
                        int seen;
                        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(seen) : "l"(counter) : "memory");
                        *sk_last = seen == contributors - 1;
                    }
                    const bool early_last = epilogue_sync_and(1) && *sk_last;
#pragma unroll 1
                    for (int c = c_begin; c < c_end && !early_last; ++c) {
                        uint32_t v[32];
                        __syncwarp();
                        tmem_ld_32x32b_x32(t_row + c * 32, v);
                        tmem_wait_ld();
                        float4* dst = reinterpret_cast<float4*>(base + (size_t)mine * slot) + c * 8 * 128;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            __stcg(dst + j * 128, make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                                        __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])));
                    }
                    last = early_last;
                    if (!early_last) {
                        // all four warps' partial stores happen-before the release below
                        epilogue_sync_and(1);
                        if (warp == 2 && lane == 0) {
                            const bool l = atomic_add_release_gpu(counter, 1) == contributors - 1;
                            if (l) fence_acquire_gpu();  // the other partials are visible to this CTA
                            *sk_last = l;
                        }
                        last = epilogue_sync_and(1) && *sk_last;
                    }
                    if (last_item && warp == 2 && lane == 0) {
                        // tell the helpers (release: with the acquire above, the
                        // other partials are visible to them too)
                        *sk_help = last ? 1 : 0;
                        mbar_arrive(smem_addr(hsync));
                    }
                    if (!last) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0 && c_begin != c_end) {
                            if constexpr (PAIR)
                                mbar_arrive_cluster(smem_addr(&tempty[buf]), 0);
                            else
                                mbar_arrive(smem_addr(&tempty[buf]));
                        }
                        continue;
                    }
                }
                // last to arrive: every other partial is published; add them
                // all in K order (own part from TMEM) and finish the tile.  The
                // other contributor's next chunk is loaded while this one is
                // finished (two contributors is the common case).
                const int other = contributors == 2 ? 1 - mine : -1;
                float4 pre[8];
                if (other >= 0 && cb < ce) {
                    const float4* src = reinterpret_cast<const float4*>(base + (size_t)other * slot) +
                                        cb * 8 * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j) pre[j] = __ldcg(src + j * 128);
                }
#pragma unroll 1
                for (int c = cb; c < ce; ++c) {
                    uint32_t v[32];
                    __syncwarp();
                    tmem_ld_32x32b_x32(t_row + c * 32, v);
                    float4 cur4[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) cur4[j] = pre[j];
                    if (other >= 0 && c + 1 < ce) {
                        const float4* src = reinterpret_cast<const float4*>(base + (size_t)other * slot) +
                                            (c + 1) * 8 * 128;
#pragma unroll
                        for (int j = 0; j < 8; ++j) pre[j] = __ldcg(src + j * 128);
                    }
                    tmem_wait_ld();
                    if (c == ce - 1 && !helper) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            if constexpr (PAIR)
                                mbar_arrive_cluster(smem_addr(&tempty[buf]), 0);
                            else
                                mbar_arrive(smem_addr(&tempty[buf]));
                        }
                    }
                    float y[32];
                    if (other >= 0) {
                        // two parts: p0 + p1 (fp32 addition of two terms is order-free)
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            y[4 * j] = __uint_as_float(v[4 * j]) + cur4[j].x;
                            y[4 * j + 1] = __uint_as_float(v[4 * j + 1]) + cur4[j].y;
                            y[4 * j + 2] = __uint_as_float(v[4 * j + 2]) + cur4[j].z;
                            y[4 * j + 3] = __uint_as_float(v[4 * j + 3]) + cur4[j].w;
                        }
                    } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) y[j] = 0.0f;
                    for (int k = 0; k < contributors; ++k) {
                        if (k == mine) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) y[j] += __uint_as_float(v[j]);
                        } else {
                            const float4* src =
                                reinterpret_cast<const float4*>(base + (size_t)k * slot) + c * 8 * 128;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const float4 u = __ldcg(src + j * 128);
                                y[4 * j] += u.x;
                                y[4 * j + 1] += u.y;
                                y[4 * j + 2] += u.z;
                                y[4 * j + 3] += u.w;
                            }
                        }
                    }
                    }
                    if (p.swap) {
                        epilogue_swap(p, rk, tn * BN + c * 32, y, row_bias);
                    } else {
                        finish_chunk(p, stage, chunks, lane, rk, row0, tn * BN + c * 32, y, row_scale,
                                     pick(bcol, c), true, nullptr);
                    }
                }
                if (warp == 2 && lane == 0) *counter = 0;  // ready for the next call
                continue;
            }
#pragma unroll 1
            for (int c = cb; c < ce; ++c) {
                uint32_t v[32];
                __syncwarp();
                tmem_ld_32x32b_x32(t_row + c * 32, v);
                tmem_wait_ld();
                if (c == ce - 1 && !helper) {
                    // every column of this buffer is in registers: release it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (PAIR)
                            mbar_arrive_cluster(smem_addr(&tempty[buf]), 0);  // leader's barrier
                        else
                            mbar_arrive(smem_addr(&tempty[buf]));
                    }
                }
                float y[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) y[j] = __uint_as_float(v[j]);
                if (p.swap) {
                    epilogue_swap(p, rk, tn * BN + c * 32, y, row_bias);
                    continue;
                }
                if constexpr (AUX) {
                    bool nxt_full = false;
                    if (c + 1 < ce)
                        nxt_full = prefetch_aux(p, rk, tn * BN + (c + 1) * 32, nxt, pol);
                    finish_chunk(p, stage, chunks, lane, rk, row0, tn * BN + c * 32, y, row_scale,
                                 pick(bcol, c), true, cur_full ? &cur : nullptr);
                    cur = nxt;
                    cur_full = nxt_full;
                } else {
                    finish_chunk(p, stage, chunks, lane, rk, row0, tn * BN + c * 32, y, row_scale,
                                 0.0f, false, nullptr);
                }
            }
        }
        if (lane == 0) bulk_wait_group<0>();  // every output chunk has reached global memory
    }

    tc_fence_before();
    __syncwarp();
    if (*abort_flag) {
        // loads for phases that were never armed (the peer's, or the second
        // producer's) cannot be observed here: give any such copy ample time
        // to land
        const long long t0 = clock64();
        while (clock64() - t0 < 2000000) {
        }
    }
    if constexpr (PAIR) {
        cluster_sync();  // no CTA leaves while its peer may still signal it
    } else {
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, TS::kTmemCols);
    }
}

}  // namespace tg

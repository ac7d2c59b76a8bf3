// gemm_kernel.cuh -- persistent, warp-specialised tiled GEMM for sm_103a.
//
// The computation is the tiled matrix multiply of the named-layout GEMM
// (ninetoothed.org "Named layouts"): every output block C[BM, BN] starts from
// a zero fp32 accumulator, adds dot(A_k[BM, 64], B_k[64, BN]) for each of the
// ceil(K / 64) K-blocks, then applies the same-output-domain epilogue
// (row scale, column bias, ReLU, residual) and is stored in the input dtype.
//
// GB300 mapping (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer: fills an S-stage ring of 128B-swizzled shared
//               tiles, one mbarrier "full"/"empty" pair per stage.  Tails of
//               M, N and K are zero-filled by the tensor map, so they add 0.
//   warp 1      owns TMEM; one thread issues tcgen05.mma (K=16 per
//               instruction) into a double-buffered fp32 accumulator.
//   warps 2..5  epilogue: tcgen05.ld 32x32b (thread t of warp w holds TMEM
//               lane 32*(w%4)+t = tile row, register j = tile column), applies
//               the epilogue in fp32 and stores with per-element edge masks,
//               while the next tile's main loop already runs in the other
//               accumulator buffer.
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

constexpr int kBK = 64;        // K elements per stage: one 128-byte swizzle row of fp16/bf16
constexpr int kUmmaK = 16;     // K per tcgen05.mma of kind::f16
constexpr int kThreads = 192;  // producer warp, MMA warp, four epilogue warps

template <int BN, bool PAIR>
struct TileShape {
    static constexpr int kBM = PAIR ? 256 : 128;              // rows per tile (whole cluster)
    static constexpr int kBNC = PAIR ? BN / 2 : BN;           // B columns staged per CTA
    static constexpr int kBBoxes = (kBNC + 63) / 64;          // 64-column swizzle atoms
    static constexpr int kAStage = 128 * kBK * 2;             // 16 KB
    static constexpr int kBStage = kBBoxes * 64 * kBK * 2;    // whole atoms
    static constexpr int kStage = kAStage + kBStage;
    static constexpr int kStages = (200 * 1024 / kStage) > 8 ? 8 : (200 * 1024 / kStage);
    static constexpr int kTmemCols = 2 * BN <= 32 ? 32 : 2 * BN <= 64 ? 64 : 2 * BN <= 128 ? 128
                                   : 2 * BN <= 256 ? 256 : 512;
    static constexpr int kSmemBytes = 1024 + kStages * kStage + (2 * kStages + 5) * 8 + 16;
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

// Bounded wait on an mbarrier phase.  Returns false if the CTA is aborting or
// this wait ran out of time (then it raises the abort flags and records `code`).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Watch& w, int code) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
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
    while (!mbar_try_wait(bar, parity)) {
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

__device__ __forceinline__ uint32_t pack2(float a, float b, int bf16) {
    return (uint32_t)from_f32(a, bf16) | ((uint32_t)from_f32(b, bf16) << 16);
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8], int bf16) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = to_f32((uint16_t)(w[i] & 0xFFFFu), bf16);
        f[2 * i + 1] = to_f32((uint16_t)(w[i] >> 16), bf16);
    }
}

// Residual and bias values of one full 32-column run of row m, loaded ahead
// of the accumulator so that their latency overlaps the TMEM read.
struct Aux {
    uint4 r[4];
    uint4 b[4];
};

// Issues the loads for the run C(m, c0 .. c0+31) if it is full and inside C;
// returns whether it is (otherwise the chunk takes the masked scalar path).
__device__ __forceinline__ bool prefetch_aux(const GemmParams& p, int m, int c0, Aux& a) {
    if (p.swap || m >= p.M || c0 + 32 > p.N) return false;
    if (p.resid) {
        const uint4* r = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.resid) +
                                                        (long long)m * p.ldr + c0);
#pragma unroll
        for (int v = 0; v < 4; ++v) a.r[v] = __ldg(r + v);
    }
    if (p.bias_n) {
        const uint4* b = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.bias_n) + c0);
#pragma unroll
        for (int v = 0; v < 4; ++v) a.b[v] = __ldg(b + v);
    }
    return true;
}

// Epilogue of a full run C(m, c0 .. c0+31) with its operands already loaded.
__device__ __forceinline__ void epilogue_run(const GemmParams& p, int m, int c0, float (&y)[32],
                                             float row_scale, const Aux& a) {
    const int bf = p.bf16;
    if (p.scale_m) {
#pragma unroll
        for (int j = 0; j < 32; ++j) y[j] *= row_scale;
    }
    if (p.bias_n) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            float f[8];
            unpack8(a.b[v], f, bf);
#pragma unroll
            for (int i = 0; i < 8; ++i) y[8 * v + i] += f[i];
        }
    }
    if (p.relu) {
#pragma unroll
        for (int j = 0; j < 32; ++j) y[j] = fmaxf(y[j], 0.0f);
    }
    if (p.resid) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            float f[8];
            unpack8(a.r[v], f, bf);
#pragma unroll
            for (int i = 0; i < 8; ++i) y[8 * v + i] += f[i];
        }
    }
    uint4* c = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.C) + (long long)m * p.ldc + c0);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        uint4 u;
        u.x = pack2(y[8 * v + 0], y[8 * v + 1], bf);
        u.y = pack2(y[8 * v + 2], y[8 * v + 3], bf);
        u.z = pack2(y[8 * v + 4], y[8 * v + 5], bf);
        u.w = pack2(y[8 * v + 6], y[8 * v + 7], bf);
        c[v] = u;
    }
}

// Epilogue for one 32-column chunk held by this thread: kernel row `rk`
// (one TMEM lane), kernel columns c0 .. c0+31 in y[].  General path: edge
// runs of C, and the swapped (transposed-output) layout.
__device__ __forceinline__ void epilogue_chunk(const GemmParams& p, int rk, int c0,
                                               float (&y)[32], float row_scale, float row_bias) {
    const int bf = p.bf16;
    if (!p.swap) {
        // C(m = rk, n = c0 + j): a contiguous run of 32 outputs in one row.
        const int m = rk;
        if (m >= p.M || c0 >= p.N) return;
        const bool full = c0 + 32 <= p.N;
        if (p.scale_m) {
#pragma unroll
            for (int j = 0; j < 32; ++j) y[j] *= row_scale;
        }
        if (p.bias_n) {
            const uint16_t* b = static_cast<const uint16_t*>(p.bias_n) + c0;
            if (full) {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    float f[8];
                    unpack8(__ldg(reinterpret_cast<const uint4*>(b) + v), f, bf);
#pragma unroll
                    for (int i = 0; i < 8; ++i) y[8 * v + i] += f[i];
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (c0 + j < p.N) y[j] += to_f32(b[j], bf);
            }
        }
        if (p.relu) {
#pragma unroll
            for (int j = 0; j < 32; ++j) y[j] = fmaxf(y[j], 0.0f);
        }
        if (p.resid) {
            const uint16_t* r = static_cast<const uint16_t*>(p.resid) + (long long)m * p.ldr + c0;
            if (full) {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    float f[8];
                    unpack8(__ldg(reinterpret_cast<const uint4*>(r) + v), f, bf);
#pragma unroll
                    for (int i = 0; i < 8; ++i) y[8 * v + i] += f[i];
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (c0 + j < p.N) y[j] += to_f32(r[j], bf);
            }
        }
        uint16_t* c = static_cast<uint16_t*>(p.C) + (long long)m * p.ldc + c0;
        if (full) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                uint4 u;
                u.x = pack2(y[8 * v + 0], y[8 * v + 1], bf);
                u.y = pack2(y[8 * v + 2], y[8 * v + 3], bf);
                u.z = pack2(y[8 * v + 4], y[8 * v + 5], bf);
                u.w = pack2(y[8 * v + 6], y[8 * v + 7], bf);
                reinterpret_cast<uint4*>(c)[v] = u;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (c0 + j < p.N) c[j] = from_f32(y[j], bf);
        }
    } else {
        // Swapped operands: kernel row rk is C's column n, kernel column c0+j is
        // C's row m.  Lanes of a warp hold consecutive n, so every store
        // instruction writes one contiguous run of a C row.
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
}

// AUX = true: the epilogue reads a bias and/or residual; their loads are
// issued one 32-column run ahead (and before the accumulator is ready).
// AUX = false keeps the plain epilogue lean.
template <int BN, bool PAIR, bool AUX>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
    using TS = TileShape<BN, PAIR>;
    constexpr int STAGES = TS::kStages;
    constexpr int CG = PAIR ? 2 : 1;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128B-swizzle atoms (same offset in both CTAs of a pair)
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * TS::kAStage;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * TS::kBStage);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0;
    const bool leader = rank == 0;
    const int cta_tile0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;  // first tile
    const int tile_step = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    const Watch w{abort_flag,
                  PAIR ? mapa_shared(smem_addr((const void*)abort_flag), rank ^ 1u) : 0u, PAIR,
                  p.status, p.timeout_cycles};

    if (threadIdx.x == 0) {
        prefetch_tensormap(&p.map_p);
        prefetch_tensormap(&p.map_q);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&tfull[b]), 1);
            mbar_init(smem_addr(&tempty[b]), PAIR ? 8 : 4);  // one arrival per epilogue warp
        }
        mbar_init(smem_addr(drain), 1);
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

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_parity = 0;
            long long g = 0;
            bool ok = true;
            // bytes this CTA lands per stage (A half + its B columns)
            const uint32_t a_bytes = TS::kAStage;
            const uint32_t b_bytes = p.q_mn_major ? (uint32_t)TS::kBStage : (uint32_t)TS::kBNC * 128u;
            const uint32_t stage_tx = (a_bytes + b_bytes) * (PAIR ? 2u : 1u);
            for (int t = cta_tile0; ok && t < p.num_tiles; t += tile_step) {
                int tm, tn;
                tile_coords(p, t, tm, tn);
                const int m0 = tm * TS::kBM + (int)rank * 128;
                const int n0 = tn * BN + (int)rank * TS::kBNC;
                for (int kb = 0; kb < p.num_kb; ++kb, ++g) {
                    if (!wait_bar(smem_addr(&empty[stage]), phase ^ 1, w, DEV_TIMEOUT_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    if (g != p.inject_skip_load) {
                        const uint32_t fb_local = smem_addr(&full[stage]);
                        if (leader) {
                            mbar_arrive_expect_tx(fb_local, stage_tx);
                            armed |= 1u << stage;
                            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                        }
                        const uint32_t fb = PAIR ? mapa_shared(fb_local, 0) : fb_local;
                        const uint32_t a_dst = smem_addr(sA + stage * TS::kAStage);
                        const uint32_t b_dst = smem_addr(sB + stage * TS::kBStage);
                        const int k0 = kb * kBK;
                        if (p.p_mn_major) {
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                if constexpr (PAIR)
                                    tma_load_2d_pair(a_dst + j * 8192, &p.map_p, fb, m0 + 64 * j, k0);
                                else
                                    tma_load_2d(a_dst + j * 8192, &p.map_p, fb, m0 + 64 * j, k0);
                            }
                        } else {
                            if constexpr (PAIR)
                                tma_load_2d_pair(a_dst, &p.map_p, fb, k0, m0);
                            else
                                tma_load_2d(a_dst, &p.map_p, fb, k0, m0);
                        }
                        if (p.q_mn_major) {
#pragma unroll
                            for (int j = 0; j < TS::kBBoxes; ++j) {
                                if constexpr (PAIR)
                                    tma_load_2d_pair(b_dst + j * 8192, &p.map_q, fb, n0 + 64 * j, k0);
                                else
                                    tma_load_2d(b_dst + j * 8192, &p.map_q, fb, n0 + 64 * j, k0);
                            }
                        } else {
                            if constexpr (PAIR)
                                tma_load_2d_pair(b_dst, &p.map_q, fb, k0, n0);
                            else
                                tma_load_2d(b_dst, &p.map_q, fb, k0, n0);
                        }
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (*abort_flag) {
                // No TMA write may land after the CTA exits: wait for the last
                // armed phase of every stage (the leader's barriers count the
                // bytes of both CTAs).
                for (int s = 0; s < STAGES; ++s)
                    if (armed & (1u << s)) drain_bar(smem_addr(&full[s]), (armed_parity >> s) & 1, w);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------ MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int i = 0;
            for (int t = cta_tile0; ok && t < p.num_tiles; t += tile_step, ++i) {
                const int buf = i & 1;
                const uint32_t aph = (i >> 1) & 1;
                if (!wait_bar(smem_addr(&tempty[buf]), aph ^ 1, w, DEV_TIMEOUT_MMA + 1)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bar(smem_addr(&full[stage]), phase, w, DEV_TIMEOUT_MMA + 2)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_addr(sA + stage * TS::kAStage);
                    const uint32_t b_addr = smem_addr(sB + stage * TS::kBStage);
#pragma unroll
                    for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                        // K-major: step 16 elements = 32 bytes inside the swizzle row.
                        // MN-major: step 16 K-rows of 128 bytes.
                        const uint64_t ad = p.p_mn_major
                                                ? smem_desc_sw128(a_addr + kk * 2048, 8192, 1024)
                                                : smem_desc_sw128(a_addr + kk * 32, 16, 1024);
                        const uint64_t bd = p.q_mn_major
                                                ? smem_desc_sw128(b_addr + kk * 2048, 8192, 1024)
                                                : smem_desc_sw128(b_addr + kk * 32, 16, 1024);
                        mma_f16<CG>(d_tmem, ad, bd, p.idesc, (kb | kk) != 0);
                    }
                    // frees the stage (in both CTAs) once the MMAs have read it
                    if constexpr (PAIR)
                        mma_commit_pair(smem_addr(&empty[stage]), 0x3);
                    else
                        mma_commit(smem_addr(&empty[stage]));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                // accumulator complete (in both CTAs' TMEM)
                if constexpr (PAIR)
                    mma_commit_pair(smem_addr(&tfull[buf]), 0x3);
                else
                    mma_commit(smem_addr(&tfull[buf]));
            }
            // Nothing may still write TMEM when it is released.
            if constexpr (PAIR)
                mma_commit_pair_local(smem_addr(drain));
            else
                mma_commit(smem_addr(drain));
            drain_bar(smem_addr(drain), 0, w);
        }
    } else {
        // ---------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quadrant this warp may read
        int i = 0;
        for (int t = cta_tile0; t < p.num_tiles; t += tile_step, ++i) {
            const int buf = i & 1;
            const uint32_t aph = (i >> 1) & 1;
            int tm, tn;
            tile_coords(p, t, tm, tn);
            const int rk = tm * TS::kBM + (int)rank * 128 + q * 32 + lane;
            // operands of the first run do not depend on the accumulator:
            // fetch them while the main loop still runs
            Aux cur, nxt;
            bool cur_full = AUX ? prefetch_aux(p, rk, tn * BN, cur) : false;
            int ok = 1;
            if (lane == 0) ok = wait_bar(smem_addr(&tfull[buf]), aph, w, DEV_TIMEOUT_EPILOGUE);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            float row_scale = 1.0f, row_bias = 0.0f;
            if (!p.swap) {
                if (p.scale_m && rk < p.M) row_scale = to_f32(static_cast<const uint16_t*>(p.scale_m)[rk], p.bf16);
            } else {
                if (p.bias_n && rk < p.N) row_bias = to_f32(static_cast<const uint16_t*>(p.bias_n)[rk], p.bf16);
            }
            const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t v[32];
                __syncwarp();
                tmem_ld_32x32b_x32(t_row + c * 32, v);
                tmem_wait_ld();
                if (c == BN / 32 - 1) {
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
                if constexpr (AUX) {
                    bool nxt_full = false;
                    if (c + 1 < BN / 32)
                        nxt_full = prefetch_aux(p, rk, tn * BN + (c + 1) * 32, nxt);
                    if (cur_full)
                        epilogue_run(p, rk, tn * BN + c * 32, y, row_scale, cur);
                    else
                        epilogue_chunk(p, rk, tn * BN + c * 32, y, row_scale, row_bias);
                    cur = nxt;
                    cur_full = nxt_full;
                } else {
                    epilogue_chunk(p, rk, tn * BN + c * 32, y, row_scale, row_bias);
                }
            }
        }
    }

    tc_fence_before();
    __syncwarp();
    if constexpr (PAIR) {
        if (*abort_flag) {
            // the peer's loads for phases the leader never armed cannot be
            // observed here: give any such copy ample time to land
            const long long t0 = clock64();
            while (clock64() - t0 < 2000000) {
            }
        }
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

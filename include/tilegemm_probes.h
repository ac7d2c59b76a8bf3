/*
 * tilegemm_probes.h -- hardware probes of libtilegemm (test hooks).
 *
 * They pin the host layout module to what the GPU does: the shared-memory
 * XOR swizzle that a TMA copy writes and the tensor cores read (retepy.com
 * "Triton LinearLayout": an XOR shared-memory swizzle is a linear layout), and
 * which thread and register receive which accumulator element when TMEM is
 * read back (the register/lane/warp ownership that section models;
 * pbelevich.github.io "My Triton From Scratch Part 16: Register Tiles":
 * several accumulators per thread with an exact logical coordinate each).
 *
 * All pointers are device pointers of the current device; each call makes one
 * launch on `stream` and returns without synchronising.  A probe whose
 * bounded wait gives up writes a nonzero code to *status_dev (one int, set
 * to 0 by the caller beforehand).  Return values are TG_* codes (tilegemm.h).
 */
#ifndef TILEGEMM_PROBES_H
#define TILEGEMM_PROBES_H

#include <stdint.h>

#include <cuda_runtime_api.h>

#include "tilegemm_layout_device.h" /* tg_folded_layout */

#ifdef __cplusplus
extern "C" {
#endif

/* TMA-loads columns 0..63 of rows 0..rows-1 of the 16-bit matrix src
 * (row stride ld elements, ld >= 64, ld*2 a multiple of 16, src 16-byte
 * aligned) into shared memory with the 128-byte swizzle and copies the
 * rows*128 shared bytes unchanged to dst.  rows: power of two in 8..256. */
int tg_probe_swizzle128(const void* src, int rows, int64_t ld, void* dst, int* status_dev,
                        cudaStream_t stream);

/* One tcgen05.mma (M=128, N=bn, K=16, fp16 in, fp32 accumulate) with
 * D[m][n] = 256*m + n, read back by four warps with tcgen05.ld 32x32b:
 * dst[(warp*32 + lane)*bn + register] = raw fp32 bits that thread `lane` of
 * warp `warp` received in that register.  bn: 64, 128 or 256; dst holds
 * 128*bn uint32. */
int tg_probe_tmem_32x32b(int bn, void* dst, int* status_dev, cudaStream_t stream);

/* Device evaluation of a folded layout (tg_layout_fold): thread c splits c
 * into the variable inputs (first variable dim in the lowest bits), applies
 * the layout with tg_folded_apply_packed and writes output o to
 * dst[c*n_outs + o] (int32).  f->n_bits <= 20; dst: device memory of the
 * current device, at least 2^n_bits * n_outs * 4 bytes (TG_ERR_BUFFER
 * otherwise, TG_ERR_POINTER if dst is not device memory). */
int tg_probe_folded_layout(const tg_folded_layout* f, void* dst, size_t dst_bytes,
                           cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TILEGEMM_PROBES_H */

/*
 * tilegemm_layout_device.h -- evaluating a linear layout inside a kernel,
 * with every input whose value is known ahead of time folded away.
 *
 * The scheme follows the lowering of a layout to index arithmetic in
 * retepy.com "Triton LinearLayout", section "applyLinearLayout": inputs with
 * known values are applied once to give a constant part of every output;
 * the remaining inputs are concatenated into one bit vector x, and each
 * output is the constant part XOR the GF(2) product of the remaining inputs'
 * sublayout matrix with x.  Here the folding happens on the host
 * (tg_layout_fold in tilegemm.h), and every output coordinate is packed as a
 * bit field of one 32-bit word, so the product is one XOR of a packed column
 * per set bit of x -- a few integer instructions per call, no table lookups
 * per output dim.
 *
 * The struct is plain data: pass it to a kernel by value, or keep it in
 * constant or global memory.  The functions compile for host and device.
 */
#ifndef TILEGEMM_LAYOUT_DEVICE_H
#define TILEGEMM_LAYOUT_DEVICE_H

#include <stdint.h>

#if defined(__CUDACC__)
#define TG_LAYOUT_FN __host__ __device__ __forceinline__
#else
#define TG_LAYOUT_FN static inline
#endif

#define TG_FOLD_MAX_VARS 8
#define TG_FOLD_MAX_OUTS 8
#define TG_FOLD_MAX_BITS 32

typedef struct {
    int n_vars;                              /* input dims left variable, in the layout's order */
    int var_bits[TG_FOLD_MAX_VARS];          /* log2 size of each of them */
    int n_bits;                              /* their total, at most 32 */
    uint32_t cols[TG_FOLD_MAX_BITS];         /* packed outputs of each variable input bit */
    uint32_t constant;                       /* packed outputs of the folded (fixed) inputs */
    int n_outs;                              /* output dims, in the layout's order */
    int out_shift[TG_FOLD_MAX_OUTS];         /* bit offset of each output in a packed word */
    int out_bits[TG_FOLD_MAX_OUTS];          /* log2 size of each output; total at most 32 */
} tg_folded_layout;

/* All outputs, packed, for the variable inputs vars[0 .. n_vars) (each
 * below 2^var_bits of its dim; higher bits are ignored). */
TG_LAYOUT_FN uint32_t tg_folded_apply_packed(const tg_folded_layout* f, const uint32_t* vars) {
    uint32_t x = 0;
    int shift = 0;
    for (int v = 0; v < f->n_vars; ++v) {
        const int b = f->var_bits[v];
        if (b > 0) x |= (vars[v] & ((b >= 32) ? 0xffffffffu : ((1u << b) - 1u))) << shift;
        shift += b;
    }
    uint32_t y = f->constant;
    for (int i = 0; i < f->n_bits; ++i) y ^= f->cols[i] & (0u - ((x >> i) & 1u));
    return y;
}

/* Output dim o of a packed word. */
TG_LAYOUT_FN int32_t tg_folded_output(const tg_folded_layout* f, uint32_t packed, int o) {
    const int b = f->out_bits[o];
    return b == 0 ? 0 : (int32_t)((packed >> f->out_shift[o]) & ((1u << b) - 1u));
}

#undef TG_LAYOUT_FN

#endif /* TILEGEMM_LAYOUT_DEVICE_H */

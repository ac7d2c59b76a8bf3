/*
 * tilegemm.h -- C ABI of libtilegemm, a tiled GEMM with a fused output-domain
 * epilogue for GB300 (sm_103a), and its GF(2) layout module.
 *
 * Every call takes plain pointers and sizes.  GEMM operand pointers are DEVICE
 * pointers (memory of the current CUDA device); layout calls are host-only.
 *
 * Status codes: every call returns TG_OK (0) or one of the TG_ERR_* codes
 * below; tg_status_string() names them.  Argument checks run before any
 * device work, cannot be switched off, and "cannot prove it is safe" is an
 * error (ninetoothed.org "Named layouts", section "Runtime and compilation":
 * positive sizes and strides, non-contiguous inputs allowed, output storage
 * disjoint from every input, checks before kernel work).
 *
 * Per-device state (device attributes, the device address of the watchdog
 * word and of the static scratch array, copy streams) is looked up once per
 * device and cached for the life of the process; the library does not
 * support cudaDeviceReset.
 */
#ifndef TILEGEMM_H
#define TILEGEMM_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h> /* cudaStream_t */

#include "tilegemm_layout_device.h" /* tg_folded_layout */

#ifdef __cplusplus
extern "C" {
#endif

enum {
    TG_OK = 0,
    TG_ERR_INVALID_ARG = 1,        /* null pointer, size <= 0 or > 2^31-1, bad enum, relu not 0/1 */
    TG_ERR_STRIDE = 2,             /* leading dimension < row width (or <= 0) */
    TG_ERR_ALIGN = 3,              /* pointer not 16-byte aligned or ld*2 not a multiple of 16 (tg_gemm),
                                      or a pointer not 2-byte aligned (every call) */
    TG_ERR_OVERLAP = 4,            /* output bytes intersect an input's bytes */
    TG_ERR_DTYPE = 5,              /* dtype not TG_F16 / TG_BF16 */
    TG_ERR_UNSUPPORTED_DEVICE = 6, /* no CUDA device, or not compute capability 10.x with tcgen05 */
    TG_ERR_CUDA = 7,               /* a CUDA runtime/driver call or the launch failed */
    TG_ERR_TIMEOUT = 8,            /* a bounded device wait expired (reported by tg_debug_status) */
    TG_ERR_POINTER = 9,            /* a pointer is not device memory of the current device, or the
                                      bytes the call touches run past the end of its allocation */
    TG_ERR_LAYOUT = 10,            /* layout arguments violate a layout invariant */
    TG_ERR_BUFFER = 11             /* caller's output buffer too small */
};

typedef enum { TG_F16 = 0, TG_BF16 = 1 } tg_dtype;

/* Explicit permute of an operand's storage.  A transposed input must say so;
 * a matching size never stands in for a transpose (ninetoothed.org "Named
 * layouts", section "Contract"). */
typedef enum { TG_OP_N = 0, TG_OP_T = 1 } tg_perm;

/* Same-output-domain epilogue (ninetoothed.org "Named layouts": a column bias
 * has axes ("n"), a row scale axes ("m"); bias/ReLU/residual postprocessing):
 *
 *     y = acc;  y *= scale_m[m];  y += bias_n[n];  y = max(y, 0);  y += R[m*ldr + n]
 *
 * each step only when its operand is given, in that order.  All operands have
 * the GEMM's dtype and are device pointers; R must not overlap C. */
typedef struct {
    const void* bias_n;   /* [N] or NULL */
    const void* scale_m;  /* [M] or NULL */
    int relu;             /* 0 or 1 */
    const void* residual; /* M rows of ldr elements, or NULL */
    int64_t ldr;          /* residual row stride in elements; 0 means ldc */
} tg_epilogue;

/*
 * C = epilogue(A * B), accumulated in fp32, stored as dtype with
 * round-to-nearest-even.
 *
 * The computation is the named-layout GEMM (ninetoothed.org "Named layouts":
 * acc = zeros(f32); for each of ceil(K/BK) blocks acc += dot(lhs[k], rhs[k]);
 * output = acc.to(dtype)), tiled over output blocks
 * (pbelevich.github.io "My Triton From Scratch Part 16: Register Tiles":
 * several fp32 accumulators per thread, per-element masked stores on edges).
 *
 * Layout (strides in elements, inner stride 1, all ld > 0):
 *   permA = TG_OP_N: A(m,k) = A[m*lda + k], lda >= K   (M x K row-major)
 *   permA = TG_OP_T: A(m,k) = A[k*lda + m], lda >= M   (storage K x M)
 *   permB = TG_OP_N: B(k,n) = B[k*ldb + n], ldb >= N   (K x N row-major)
 *   permB = TG_OP_T: B(k,n) = B[n*ldb + k], ldb >= K   (storage N x K)
 *   C(m,n) = C[m*ldc + n], ldc >= N.
 * Requirements: 1 <= M, N, K <= 2^31-1; every pointer 16-byte aligned and
 * every ld*2 a multiple of 16 bytes (tensor-memory-access copies); C's bytes
 * disjoint from A, B, bias, scale and R; every pointer inside one device
 * allocation of the current device that covers all bytes the call touches.
 *
 * Ownership: the caller owns all buffers.  The call allocates nothing, makes
 * one kernel launch on `stream` (0 = legacy default stream) and returns
 * without synchronising.  `epi` may be NULL (plain GEMM).
 * Errors: any failed check returns its code before device work starts;
 * TG_ERR_CUDA if the launch fails.  Device-side watchdog expiries are
 * reported later by tg_debug_status().
 */
int tg_gemm(int64_t M, int64_t N, int64_t K,
            const void* A, int64_t lda, tg_perm permA,
            const void* B, int64_t ldb, tg_perm permB,
            void* C, int64_t ldc, tg_dtype dtype,
            const tg_epilogue* epi, cudaStream_t stream);

/*
 * tg_gemm with a caller-provided workspace that lets the kernel deal the
 * tiles of its last waves out as equal K-ranges over all SMs ("stream-K"):
 * when the tile count is not a multiple of the number of persistent workers,
 * the tail would otherwise leave SMs idle.  A tile whose K-range is split
 * is finished by the contributor that arrives last, which adds the fp32
 * partial sums in K order (results are reproducible call to call); no CTA
 * ever waits for another.
 *
 * workspace: device memory of the current device, 256-byte aligned, at least
 *   tg_gemm_workspace_size() bytes, disjoint from every operand, filled with
 *   zero bytes before its first use (e.g. cudaMemset once); every completed
 *   call leaves its counters at zero again.  After TG_ERR_TIMEOUT from
 *   tg_debug_status, zero it again.  Calls that share a workspace must not
 *   run concurrently on the GPU.
 * Unaligned operands: unlike tg_gemm, any pointer that is 2-byte aligned
 *   and any positive stride are accepted (ninetoothed.org "Named layouts",
 *   section "Runtime and compilation": positive, possibly non-contiguous
 *   strides).  An operand a tensor map cannot describe (base not 16-byte
 *   aligned, or ld*2 not a multiple of 16) is copied into an aligned dense
 *   buffer inside the workspace first (A, B, R, bias, scale), and an
 *   unaligned C is written to one and copied out afterwards: up to three
 *   more kernel launches on `stream`, and workspace for the copies, as
 *   tg_gemm_workspace_size_ex() reports.
 * workspace == NULL: exactly tg_gemm.  Other arguments, checks and errors as
 * tg_gemm; TG_ERR_BUFFER if workspace_bytes is too small, TG_ERR_ALIGN /
 * TG_ERR_OVERLAP / TG_ERR_POINTER for a misplaced workspace.
 */
int tg_gemm_ws(int64_t M, int64_t N, int64_t K,
               const void* A, int64_t lda, tg_perm permA,
               const void* B, int64_t ldb, tg_perm permB,
               void* C, int64_t ldc, tg_dtype dtype,
               const tg_epilogue* epi, void* workspace, size_t workspace_bytes,
               cudaStream_t stream);

/*
 * tg_gemm_ws without a caller workspace, for callers that cannot allocate
 * device memory: code under an outside allocator that owns all of the
 * device's memory, plugins whose host framework forbids device allocations,
 * and latency-bound host paths that cannot afford the implicit device
 * synchronisation of cudaMalloc / cudaFree.  The pages this library follows
 * have no counterpart of this call; it exists for these callers only.
 *
 * The scratch is one statically allocated device array of 40 MiB (41943040
 * bytes) that every GPU loading this library keeps until the process exits;
 * nothing is allocated per call (no cudaMalloc, no cudaFree, no allocating
 * library routine).  It holds what tg_gemm_workspace_size_ex() reports for
 * these arguments: the stream-K split's counters and partial sums, then the
 * staging copies of operands a tensor map cannot describe (unaligned base or
 * stride).  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and caches it: make that first call before any
 * stream capture on that device.  The library does not support
 * cudaDeviceReset (the cached address may go stale).  When the call splits
 * tiles, it zeroes the split's arrival counters on `stream`
 * (cudaMemsetAsync) before its kernel.  Every call shares the one array:
 * calls whose kernels overlap on the GPU (other streams, other host threads)
 * race and corrupt each other's results -- serialise them.
 *
 * Arguments, checks and errors as tg_gemm_ws; TG_ERR_BUFFER when the call
 * needs more scratch than the array holds (tg_gemm_workspace_size_ex()
 * above 41943040; every split the default selection makes on a 152-SM GPU
 * fits, staging copies come on top).  Shapes that need neither a split nor staging run whole
 * tiles and touch no scratch.
 */
int tg_gemm_static_ws(int64_t M, int64_t N, int64_t K,
                      const void* A, int64_t lda, tg_perm permA,
                      const void* B, int64_t ldb, tg_perm permB,
                      void* C, int64_t ldc, tg_dtype dtype,
                      const tg_epilogue* epi, cudaStream_t stream);

/* Workspace bytes tg_gemm_ws needs for these arguments on the current device
 * when every operand is aligned (0 when every tile is computed whole). */
int tg_gemm_workspace_size(int64_t M, int64_t N, int64_t K, tg_dtype dtype, tg_perm permA,
                           tg_perm permB, const tg_epilogue* epi, size_t* bytes);

/* Workspace bytes tg_gemm_ws needs for exactly these arguments: the split's
 * scratch plus a dense 16-byte-aligned copy (rows x round-up(width, 8)
 * elements, each rounded to 256 bytes) of every operand a tensor map cannot
 * describe.  The pointers are only inspected, never dereferenced.  Errors as
 * tg_gemm's argument checks. */
int tg_gemm_workspace_size_ex(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                              tg_perm permA, const void* B, int64_t ldb, tg_perm permB,
                              const void* C, int64_t ldc, tg_dtype dtype,
                              const tg_epilogue* epi, size_t* bytes);

/*
 * tg_gemm with A, B, C and the epilogue operands in page-locked HOST memory
 * (cudaHostAlloc / cudaHostRegister); the same computation, layouts, perms,
 * epilogue order and rounding as tg_gemm.  Host strides are any ld >= the
 * row width, pointers 2-byte aligned.
 *
 * The host<->device copies overlap the arithmetic: C is cut into blocks of
 * whole 256-row output-tile rows (about four blocks; TG_HOST_BLOCK_ROWS, a
 * multiple of 256, overrides).  An inbound copy stream brings B and bias,
 * then each block's rows of A, scale and R, into dense device images inside
 * `workspace`; each block's GEMM (tg_gemm_ws, one kernel) starts as soon as
 * its rows have arrived, the blocks alternating between `stream` and a side
 * stream so that two run side by side; an outbound copy stream returns each
 * block of C while later blocks are still arriving.  Each block is an independent
 * sub-GEMM over whole output tiles (ninetoothed.org "Named layouts",
 * section "Contract": one program instance per output block).
 *
 * workspace: device memory of the current device, 256-byte aligned, at
 *   least tg_gemm_host_workspace_size() bytes (two stream-K scratch areas,
 *   one per compute stream, zeroed before first use as for tg_gemm_ws, then
 *   dense images of B, bias, scale, A, R and C), inside one allocation;
 *   calls sharing a workspace must not overlap on the GPU.
 * Ordering: the copies start after the work already queued on `stream`, and
 *   work queued on `stream` after the call starts once C is back in host
 *   memory.  The call returns without synchronising; the two copy streams, the
 *   side stream and their events are made once per device and reused (calls
 *   from several host threads enqueue one at a time).
 * Errors (all before any device work): as tg_gemm's shape, enum and stride
 *   checks; TG_ERR_ALIGN for an odd host address or a workspace not 256-byte
 *   aligned; TG_ERR_OVERLAP if C's bytes meet an input's or the workspace's;
 *   TG_ERR_POINTER if a host span does not start and end in page-locked host
 *   memory, or the workspace is not device memory of the current device
 *   covering the bytes needed; TG_ERR_BUFFER if workspace_bytes is too small.
 *   TG_ERR_CUDA if a copy or launch fails while enqueuing (work already
 *   queued then still runs, and `stream` still waits for it).
 */
int tg_gemm_host(int64_t M, int64_t N, int64_t K,
                 const void* A, int64_t lda, tg_perm permA,
                 const void* B, int64_t ldb, tg_perm permB,
                 void* C, int64_t ldc, tg_dtype dtype,
                 const tg_epilogue* epi, void* workspace, size_t workspace_bytes,
                 cudaStream_t stream);

/* Workspace bytes tg_gemm_host needs for this shape on the current device
 * (independent of the host strides; `epi` only says which epilogue operands
 * are present).  Arguments in tg_gemm_workspace_size's order.  Errors as
 * tg_gemm's shape and enum checks. */
int tg_gemm_host_workspace_size(int64_t M, int64_t N, int64_t K, tg_dtype dtype, tg_perm permA,
                                tg_perm permB, const tg_epilogue* epi, size_t* bytes);

/*
 * Pointwise program of the named-layout pages (ninetoothed.org "Named
 * layouts": pointwise work, missing-axis broadcasting, reordering and
 * same-output-domain bias/ReLU/residual postprocessing):
 *
 *     C[m, n] = epilogue( X(m, n) )       (the tg_epilogue above, same order)
 *
 * scale_m has axes ("m") and bias_n axes ("n"): each broadcasts along the
 * axis it lacks.  X(m, n) = X[m*ldx + n] with ldx >= N (permX = TG_OP_N), or
 * X[n*ldx + m] with ldx >= M when the input is given permuted (TG_OP_T,
 * storage N x M): an explicit permute, never inferred from sizes.
 * C(m, n) = C[m*ldc + n], ldc >= N.  fp32 arithmetic, round to nearest even.
 *
 * Any positive strides and any 2-byte-aligned pointers (16-byte-aligned
 * rows use vector accesses).  C's bytes must be disjoint from X, bias,
 * scale and R; every pointer inside one device allocation of the current
 * device.  One kernel launch on `stream`; nothing allocated.  Errors as
 * tg_gemm's checks (TG_ERR_ALIGN only for an odd byte address).
 */
int tg_pointwise(int64_t M, int64_t N, const void* X, int64_t ldx, tg_perm permX,
                 void* C, int64_t ldc, tg_dtype dtype, const tg_epilogue* epi,
                 cudaStream_t stream);

/* Static name of a status code ("TG_OK", "TG_ERR_ALIGN", ...). */
const char* tg_status_string(int status);

/*
 * Writes the configuration tg_gemm would use for these arguments into buf
 * (NUL-terminated, e.g. "swap=0 bm=128 bn=256 pair=0 stages=4 group_m=8
 * grid=152 tiles=512"); the selector is deterministic (pbelevich.github.io
 * Part 16, "Choosing the physical thread shape": a deterministic policy, not
 * an autotuner; ninetoothed.org "Named layouts": tile sizes belong to the
 * layout).  Needs a device for the SM count; pointers are not inspected.
 * Environment TG_FORCE_CONFIG="bn=128,swap=0,pair=0,group_m=8" overrides it.
 * Returns TG_ERR_BUFFER if len is too small.
 */
int tg_query_config(int64_t M, int64_t N, int64_t K, tg_dtype dtype, tg_perm permA,
                    tg_perm permB, const tg_epilogue* epi, char* buf, size_t len);

/* The configuration tg_gemm_ws would use (adds sk_tiles, sk_cmax, ws_bytes). */
int tg_query_config_ws(int64_t M, int64_t N, int64_t K, tg_dtype dtype, tg_perm permA,
                       tg_perm permB, const tg_epilogue* epi, char* buf, size_t len);

/* tg_query_config (stream_k = 0) or tg_query_config_ws (stream_k = 1) for a
 * device with `sms` SMs (2..4096), without touching any device: the
 * selector's host logic alone. */
int tg_query_config_for_sms(int sms, int stream_k, int64_t M, int64_t N, int64_t K,
                            tg_dtype dtype, tg_perm permA, tg_perm permB, const tg_epilogue* epi,
                            char* buf, size_t len);

/*
 * Reads and clears the device status word of the current device: TG_OK, or
 * TG_ERR_TIMEOUT if some earlier kernel's bounded wait expired (the kernel
 * then stopped early and its output is incomplete).  Synchronises the device.
 * If detail != NULL it receives the raw device code (which wait gave up).
 */
int tg_debug_status(int* detail);

/*
 * Watchdog settings for later launches on this process: the wait limit in
 * SM clock cycles (0 restores the default of 4e9, about two seconds) and a
 * test hook: the producer skips arming k-block `skip_kblock` (counted across
 * the CTA's tiles; -1 = off) so a wait provably expires.
 */
int tg_debug_configure(int64_t timeout_cycles, int64_t skip_kblock);

/* ------------------------------------------------------------------------
 * GF(2) linear layouts (retepy.com "Triton LinearLayout").
 *
 * A layout maps named input dims (e.g. register, lane, warp) to named output
 * dims (e.g. tensor dims) and is linear over GF(2): L(x XOR y) = L(x) XOR
 * L(y), L(0) = 0, every dim size a power of two (section "Linear Layout").
 * It is stored as one basis vector per input bit with one coordinate per
 * output dim (section "Basis-vector representation").  Input tuples and
 * outputs are passed in the layout's dim order.  Handles are host objects,
 * owned by the caller, freed with tg_layout_destroy; the library never
 * retains caller pointers.  Dim names are at most 31 characters.
 * ---------------------------------------------------------------------- */
typedef struct tg_layout tg_layout;

/* bases: row-major [sum of in_bits][n_out]; basis i of input dim d lives at
 * row (in_bits[0] + ... + in_bits[d-1] + i).  Coordinates must fit out_bits.
 * TG_ERR_LAYOUT on duplicate names, bits outside 0..30 or a coordinate too
 * large (the invariant check of section "Surjectivity, injectivity, and
 * broadcasts"). */
int tg_layout_create(int n_in, const char* const* in_names, const int* in_bits,
                     int n_out, const char* const* out_names, const int* out_bits,
                     const int32_t* bases, tg_layout** out);
void tg_layout_destroy(tg_layout* l);

/* Dim counts, names (copied into name[len]) and log2 sizes. */
int tg_layout_num_dims(const tg_layout* l, int* n_in, int* n_out);
int tg_layout_in_dim(const tg_layout* l, int i, char* name, size_t len, int* bits);
int tg_layout_out_dim(const tg_layout* l, int i, char* name, size_t len, int* bits);
/* Copies the basis table in tg_layout_create's format. */
int tg_layout_get_bases(const tg_layout* l, int32_t* bases, size_t count);

/* outs[j] = XOR of the bases selected by the set bits of ins (section
 * "LinearLayout::apply").  Each ins[i] must be < 2^in_bits[i]. */
int tg_layout_apply(const tg_layout* l, const int32_t* ins, int32_t* outs);

/* outer o inner: outer applied to every basis of inner (section "Combining
 * layouts").  inner's out dims must equal outer's in dims (names and sizes,
 * same order). */
int tg_layout_compose(const tg_layout* inner, const tg_layout* outer, tg_layout** out);

/* Direct-sum-like product a * b (section "Combining layouts"): dims of b not
 * in a are appended; for a dim name both have, b's bits become the more
 * significant bits, i.e. (a*b)(x | y << bits_a) = a(x) | b(y) << outbits_a. */
int tg_layout_product(const tg_layout* a, const tg_layout* b, tg_layout** out);

/* Restriction to the named input and output dims (section "Combining layouts",
 * sublayout), in the order given. */
int tg_layout_sublayout(const tg_layout* l, int n_in, const char* const* in_names,
                        int n_out, const char* const* out_names, tg_layout** out);

/* Same map with the output dims reordered (transposeOuts). */
int tg_layout_transpose_outs(const tg_layout* l, int n_out, const char* const* out_names,
                             tg_layout** out);

/* Same map with the input dims reordered (transposeIns); in_names must name
 * every input dim once. */
int tg_layout_transpose_ins(const tg_layout* l, int n_in, const char* const* in_names,
                            tg_layout** out);

/* reshapeIns / reshapeOuts (section "Combining layouts": they "reorganize
 * named dimensions and their bits"; the page gives no further definition).
 * Reading taken: the input (output) bits are flattened with the first dim
 * least significant and regrouped, in order, into the new dims of the given
 * log2 sizes, whose total must equal the old total.  So the flattened input
 * index keeps its value and so does the flattened output coordinate.
 * TG_ERR_LAYOUT on a different total, a duplicate name or a size outside
 * 0..30. */
int tg_layout_reshape_ins(const tg_layout* l, int n_in, const char* const* in_names,
                          const int* in_bits, tg_layout** out);
int tg_layout_reshape_outs(const tg_layout* l, int n_out, const char* const* out_names,
                           const int* out_bits, tg_layout** out);

/* divideLeft / divideRight (section "Combining layouts": they "factor
 * compatible layouts"; no further definition on the page).  Reading taken:
 * the inverses of tg_layout_product.  divide_left returns C with
 * A = B * C and divide_right returns C with A = C * B, equal as maps once
 * dims are matched by name.  C has A's dims in A's order, each with A's bits
 * less B's.  TG_ERR_LAYOUT when B is not such a factor of A. */
int tg_layout_divide_left(const tg_layout* A, const tg_layout* B, tg_layout** out);
int tg_layout_divide_right(const tg_layout* A, const tg_layout* B, tg_layout** out);

/* Rank of the GF(2) matrix by row reduction; injective iff rank = total input
 * bits, surjective iff rank = total output bits (section "Surjectivity,
 * injectivity, and broadcasts").  Results in *value. */
int tg_layout_rank(const tg_layout* l, int* value);
int tg_layout_is_injective(const tg_layout* l, int* value);
int tg_layout_is_surjective(const tg_layout* l, int* value);

/* R.invertAndCompose(S) (section "invertAndCompose: derive data movement"):
 * a layout X from R's input dims to S's input dims with S(X(x)) = R(x) for
 * every x.  R and S must have the same output dims; S may broadcast (its
 * pseudoinverse sets free variables to zero).  TG_ERR_LAYOUT if some R(x) is
 * outside S's image. */
int tg_layout_invert_and_compose(const tg_layout* R, const tg_layout* S, tg_layout** out);

/* Rank-2 Triton blocked layout -> (register, lane, warp) -> (dim0, dim1)
 * (section "Blocked-layout example").  Per dim in `order` (minor first):
 * size_per_thread bits -> register, threads_per_warp -> lane, warps_per_cta
 * -> warp, then repetitions over the rest of `shape` -> more register bits;
 * a CTA tile larger than shape broadcasts.  All sizes powers of two. */
int tg_layout_blocked(const int size_per_thread[2], const int threads_per_warp[2],
                      const int warps_per_cta[2], const int order[2], const int shape[2],
                      tg_layout** out);

/* The same rule for a tensor of any rank 1..8: (register, lane, warp) ->
 * (dim0, ..., dim{rank-1}); each array has `rank` entries and `order` is a
 * permutation of 0..rank-1 (minor dim first).  Lane and warp ids split over
 * the dims in `order`; registers hold first the per-thread elements, then the
 * CTA tile's repetitions (section "Blocked-layout example", the encoding
 * the rank-2 example instantiates).  TG_ERR_INVALID_ARG for a null pointer or
 * rank outside 1..8, TG_ERR_LAYOUT for a size that is not a power of two, an
 * order that is not a permutation, or more bits than the module holds. */
int tg_layout_blocked_nd(int rank, const int* size_per_thread, const int* threads_per_warp,
                         const int* warps_per_cta, const int* order, const int* shape,
                         tg_layout** out);

/* Folds a layout for evaluation in a kernel (retepy.com "Triton
 * LinearLayout", section "applyLinearLayout"): the inputs named in
 * fixed_names take fixed_values and are applied once, giving the constant
 * part of every output; every other input dim stays variable, in the
 * layout's input order, and contributes one packed column per bit.  Evaluate
 * with tg_folded_apply_packed / tg_folded_output (tilegemm_layout_device.h,
 * host or device).  `out` is plain data owned by the caller.
 * TG_ERR_INVALID_ARG for null pointers or n_fixed < 0; TG_ERR_LAYOUT for an
 * unknown or repeated name, a value outside its dim, more than 8 variable
 * dims or 32 variable bits, or more than 8 output dims or 32 output bits. */
int tg_layout_fold(const tg_layout* l, int n_fixed, const char* const* fixed_names,
                   const int32_t* fixed_values, tg_folded_layout* out);

/* Host evaluation of a folded layout through the same inline functions a
 * kernel uses: outs[o] for variable inputs vars[0 .. n_vars).
 * TG_ERR_INVALID_ARG for a null pointer or a value outside its dim. */
int tg_layout_folded_apply(const tg_folded_layout* f, const int32_t* vars, int32_t* outs);

/* Cooperative traversal of a rank-2 tile by `threads` threads
 * (pbelevich.github.io Part 12, "Cooperative tile layouts": thread t at
 * iteration i visits linear index t + i*threads, peeled axis by axis in
 * `order`) -> (thread, iteration) -> (dim0, dim1).  Powers of two and
 * threads <= tile size (tail lanes are not linear). */
int tg_layout_cooperative(const int shape[2], int threads, const int order[2], tg_layout** out);

/* Register tile (pbelevich.github.io Part 16, "A strided ownership rule":
 * logical = thread + register * thread_shape) -> (register, thread) ->
 * (dim0, dim1); thread ids are row-major over thread_shape, register ids
 * row-major over logical/thread_shape.  Powers of two. */
int tg_layout_register_tile(const int logical[2], const int thread_shape[2], tg_layout** out);

/* Shared-memory 128-byte XOR swizzle of a tile with 128-byte rows of
 * elem_bytes-wide elements: (offset) -> (row, col), offset counted in
 * elements; the 16-byte chunk index of each row is XORed with row mod 8.
 * rows a power of two >= 8. */
int tg_layout_swizzle128(int rows, int elem_bytes, tg_layout** out);

/* Accumulator readout of a 128 x bn fp32 tile through tcgen05.ld 32x32b by
 * four warps: (register, lane, warp) -> (m, n) with m = 32*(warp%4) + lane,
 * n = register.  bn a power of two in 32..256. */
int tg_layout_tmem_32x32b(int bn, tg_layout** out);

#ifdef __cplusplus
}
#endif

#endif /* TILEGEMM_H */

/*
 * gemm.h -- C ABI of the GB300 (sm_103a) generalized GEMM library, libgemm.so.
 *
 *     D = epilogue( alpha * op(A) * op(B) + beta * C )
 *     epilogue(v)[i,j] = cast_out( act( v[i,j] + bias ) )
 *
 * The operation is the BLAS-style scaled product C := alpha*A*B + beta*C of
 * "CUTLASS: Fast Linear Algebra in CUDA C++" (section "Efficient Matrix
 * Multiplication on GPUs"), with the transposition of the inputs of the
 * BLAS-like interface in "Flexible Performant GEMM Kernels on GPUs" (section
 * 4.3, Listings 10-11), the N (column-major) / T (row-major) operand layouts of
 * that paper's section 5.1, and the fused epilogue of both pages: the
 * fused_bias_relu_epilogue functor of the CUTLASS page ("Fusing Element-wise
 * Operations: An Example with SGEMM": alpha*acc + bias + beta*c, then a ReLU
 * clamp) and the bias vector added to every row in section 5.3 of the paper
 * (Table 2).
 *
 * Conventions shared by every entry point:
 *   - A is logically M x K, B is K x N, C and D are M x N.
 *   - Layout N: column-major storage; element (r, c) at ptr[r + c*ld].
 *     Layout T: row-major storage;    element (r, c) at ptr[r*ld + c].
 *     (The paper's linearisation n*M + m of a column-major tile, section 3.2,
 *     Figure 4, with the leading dimension in place of M.)
 *   - C and D are always row-major: element (i, j) at ptr[i*ld + j], ld >= N.
 *     A column-major D is obtained from the identity D^T = op(B)^T op(A)^T:
 *     swap the operands, flip both layout letters and use GEMM_BIAS_ROW.
 *   - All sizes and leading dimensions are in elements, not bytes.
 *   - Device pointers (gemm_run) and the stream are owned by the caller; the
 *     library never frees them.  A plan owns only its own device scratch
 *     (an error word, and the staging and partial-sum buffers described at
 *     gemm_run).
 *   - gemm_run is asynchronous on `stream`: its return value reports argument
 *     and launch errors only.  Device-side failures surface at the caller's
 *     stream synchronisation or through gemm_plan_device_status.
 *   - No entry point falls back to the CPU.  Unsupported requests return
 *     GEMM_ERR_UNSUPPORTED.
 */
#ifndef DENSE_GEMM_EPILOGUES_GB300_GEMM_H
#define DENSE_GEMM_EPILOGUES_GB300_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t is a pointer to this opaque driver type; 0 is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st* gemm_stream_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,  /* a size, leading dimension, pointer or enum is invalid */
    GEMM_ERR_UNSUPPORTED = 2,  /* valid request the library does not implement */
    GEMM_ERR_ALIGNMENT = 3,    /* a forced kernel needs alignment the buffers lack */
    GEMM_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed (no device, launch error) */
    GEMM_ERR_TIMEOUT = 5       /* a bounded in-kernel wait expired (read via gemm_plan_device_status) */
} gemm_status_t;

typedef enum { GEMM_OP_N = 0 /* column-major */, GEMM_OP_T = 1 /* row-major */ } gemm_layout_t;

typedef enum {
    GEMM_F32 = 0,
    GEMM_F16 = 1,
    GEMM_BF16 = 2,
    GEMM_S8 = 3,
    GEMM_S32 = 4
} gemm_dtype_t;

typedef enum { GEMM_ACT_NONE = 0, GEMM_ACT_RELU = 1 } gemm_act_t;

typedef enum {
    GEMM_BIAS_NONE = 0,
    GEMM_BIAS_COL = 1, /* bias has N entries; bias[j] is added to column j of every row */
    GEMM_BIAS_ROW = 2  /* bias has M entries; bias[i] is added to row i (transposed use) */
} gemm_bias_mode_t;

/* Fused epilogue.  Order: v = alpha*acc + beta*c_act(C[i,j]) + bias; v = act(v);
 * D[i,j] = cast to out_dtype (round to nearest even).  NULL epilogue pointer
 * means: no bias, no activations, out_dtype equal to the plan's c_dtype.
 * S8 plans may write int8 D (out_dtype GEMM_S8): the int32 result v is
 * requantised as D = saturate_int8(round_half_even(fp32(v) * out_scale)), the
 * product taken in fp32 (the pages define no requantisation; this is the
 * library's reading).  out_scale is read for that cast only.
 * c_act is the elementwise transform applied to C as it is read ("ReLU on C",
 * "Flexible Performant GEMM Kernels on GPUs", section 5.3, Table 2); it only
 * matters when beta != 0.
 *
 * Operand transforms (load_xf != 0): the elementwise transforms that section
 * 4.2 of the same paper ("Transforms", Figure 10) applies to the A and B tiles
 * right after they are loaded and before the multiply-accumulate, e.g. a
 * scaling and an activation.  With bit GEMM_XF_A of load_xf set, every element
 * a of op(A) enters the product as
 *     t_A(a) = a_act(a_scale * a)
 * (the same for B with bit GEMM_XF_B, b_act and b_scale): the product is taken
 * in fp32 and rounded to nearest even, then the activation (GEMM_ACT_NONE, or
 * GEMM_ACT_RELU with threshold 0); for F16/BF16 plans the result is rounded to
 * nearest even back to the operand's own type, since the tensor cores multiply
 * 16-bit operands; F32 plans keep the fp32 value.  S8 plans accept the
 * activation only (scale exactly 1; anything else is GEMM_ERR_UNSUPPORTED).
 * Scales must be finite (else GEMM_ERR_INVALID_ARG).  load_xf == 0 (a
 * zero-initialised struct) applies no transform and ignores the four fields.
 * Where they run: the CUDA-core kernels transform each element as they load it;
 * S8 plans in the int8 -> fp16 staging pass.  The tensor-core kernels either
 * transform the staged shared-memory tiles in place, in extra warps, or -- for
 * an operand that several output tiles re-read and that is at least 4 MiB --
 * run a transform pass over the operand into plan-owned device scratch first
 * (one read and one write of the operand at memory bandwidth, cheaper than
 * transforming it once per re-reading tile inside the kernel);
 * gemm_config_t.xf_staged reports which.  Environment GEMM_XF_STAGE=0 keeps
 * every transform inside the kernel, =1 stages every transformed 16-bit
 * operand.  The operands in memory are never modified.
 * gemm_run_diag and gemm_run_complex return GEMM_ERR_UNSUPPORTED when
 * load_xf != 0. */
#define GEMM_XF_A 1u
#define GEMM_XF_B 2u
typedef struct {
    const void* bias;             /* device pointer, or NULL when bias_mode == GEMM_BIAS_NONE */
    gemm_dtype_t bias_dtype;      /* F32/F16/BF16 for floating plans, S32 for int8 plans */
    gemm_bias_mode_t bias_mode;
    gemm_act_t act;               /* activation of the result (before the cast) */
    gemm_dtype_t out_dtype;       /* dtype of D */
    gemm_act_t c_act;             /* transform of C as it is read (GEMM_ACT_NONE / GEMM_ACT_RELU) */
    float out_scale;              /* S8 plans with out_dtype GEMM_S8: the requantisation scale (finite) */
    uint32_t load_xf;             /* GEMM_XF_A | GEMM_XF_B: which operands are transformed after load */
    gemm_act_t a_act;             /* t_A(a) = a_act(a_scale * a) */
    float a_scale;
    gemm_act_t b_act;             /* t_B(b) = b_act(b_scale * b) */
    float b_scale;
} gemm_epilogue_t;

typedef struct gemm_plan* gemm_plan_t;

/* Kernels the selector chooses between (gemm_config_t.kernel). */
typedef enum {
    GEMM_KERNEL_AUTO = 0,   /* let the selector decide (default) */
    GEMM_KERNEL_NONE = 1,   /* nothing to launch (M == 0 or N == 0) */
    GEMM_KERNEL_TC = 2,     /* tcgen05 + TMA persistent warp-specialised kernel, fp16/bf16 */
    GEMM_KERNEL_TC_INT8 = 3,/* int8 exact: int8->fp16 staging, tcgen05 in 1024-deep K-chunks, int32 accumulation */
    GEMM_KERNEL_FFMA = 4,   /* fp32 SGEMM on CUDA cores, register-blocked FFMA */
    GEMM_KERNEL_SIMT = 5,   /* generic CUDA-core kernel: any alignment, K == 0, every dtype */
    GEMM_KERNEL_TC_PAIR = 6,/* tcgen05 on CTA pairs (cta_group::2), 256x256 tiles, fp16/bf16 */
    GEMM_KERNEL_DIAG = 7    /* gemm_run_diag: one product per output (reported, never forced) */
} gemm_kernel_t;

/* A launch configuration (what the selector returns; what a run used). */
typedef struct {
    int32_t kernel;       /* gemm_kernel_t */
    int32_t bm, bn, bk;   /* CTA tile (rows of D, columns of D, K per pipeline stage) */
    int32_t stages;       /* shared-memory pipeline depth */
    int32_t cta_group;    /* CTAs cooperating on one MMA tile (1 or 2) */
    int32_t split_k;      /* most K segments any tile is split into (1 = no split); FFMA kernel:
                             the parts of each split tail tile (see sk_tiles) */
    int32_t raster;       /* tile rows per raster group (L2 reuse) */
    int32_t grid;         /* CTAs launched */
    int32_t k_chunk;      /* int8 path: K elements per exact fp32 chunk; 0 otherwise */
    int32_t tiles;        /* output tiles */
    int32_t sk_tiles;     /* stream-K tiles: their K blocks are shared out over all CTAs
                             (single-CTA kernel) or CTA pairs of the launch; FFMA kernel: the
                             tiles of a last wave at most half full, each split over K into
                             split_k parts that a reduction pass adds in K order; 0 = every
                             tile runs whole on one CTA or CTA pair */
    int32_t cluster;      /* CTAs per thread-block cluster: 1, or 2 (one CTA pair) */
    int32_t half_tiles;   /* CTA-pair kernel: the last half_tiles tiles (a partial last wave
                             of at most half the CTA pairs) each run as two units of 256 x 128,
                             on two CTA pairs, so that the last wave takes half a tile's time */
    int32_t xf_staged;    /* operand transforms (gemm_epilogue_t.load_xf) applied by a staging
                             pass into plan scratch before the GEMM rather than inside it:
                             GEMM_XF_A and/or GEMM_XF_B; 0 = every requested transform runs
                             inside the GEMM kernel (or none was requested) */
} gemm_config_t;

/* ---------------------------------------------------------------------------
 * gemm_plan_create -- make a plan for one device and one operand type.
 *   plan      out: the new plan (owned by the caller, release with gemm_plan_destroy).
 *   ab_dtype  type of A and B: GEMM_F16, GEMM_BF16 (tensor cores, fp32 accumulate),
 *             GEMM_S8 (exact int32 accumulate), GEMM_F32 (CUDA-core FFMA, no TF32).
 *   c_dtype   type of C: F32/F16/BF16 for 16-bit inputs, F32 for F32, S32 for S8.
 *   device    CUDA device ordinal.
 * Allocates a 4-byte device error word on `device`.  Returns GEMM_ERR_INVALID_ARG
 * for a bad type pair, GEMM_ERR_CUDA when the device cannot be used.
 * Paper counterpart: the get_config step of "Flexible Performant GEMM Kernels on
 * GPUs" (section 4.3, Listing 9) and the plan-then-launch split of cuBLASLt
 * discussed in its section 6.
 * ------------------------------------------------------------------------- */
gemm_status_t gemm_plan_create(gemm_plan_t* plan, gemm_dtype_t ab_dtype, gemm_dtype_t c_dtype,
                               int device);

/* Release a plan and its device scratch.  Synchronises the plan's device.  NULL is a no-op. */
gemm_status_t gemm_plan_destroy(gemm_plan_t plan);

/* ---------------------------------------------------------------------------
 * gemm_run -- D = epilogue(alpha * op(A) * op(B) + beta * C) on `stream`.
 *   layoutA/B   GEMM_OP_N (column-major) or GEMM_OP_T (row-major).
 *   M, N, K     sizes (>= 0).  M == 0 or N == 0 returns GEMM_OK and launches
 *               nothing; K == 0 gives D = epilogue(beta*C).
 *   alpha,beta  scalars.  Floating plans apply them in fp32.  S8 plans require
 *               integral values within int32 and apply them in int32.
 *               beta == 0: C is not read (may be NULL; NaNs in C are ignored).
 *   A, lda      device pointer, leading dimension: lda >= M for N, >= K for T.
 *   B, ldb      device pointer, leading dimension: ldb >= K for N, >= N for T.
 *   C, ldc      device pointer (row-major), ldc >= N when beta != 0.
 *   D, ldd      device pointer (row-major), ldd >= N.  D may equal C only when
 *               ldc == ldd and the types match (in-place C := ...).
 *   epi         fused epilogue (NULL: none, out_dtype = c_dtype).
 *   stream      CUDA stream (cudaStream_t) the kernels are enqueued on.
 * Kernel choice: 16-byte aligned A/B with 16-byte multiple strides use the
 * tcgen05 tensor-core kernel (S8: an int8->fp16 staging pass into plan-owned
 * device scratch, grown on demand with stream-ordered allocation, then the
 * tensor-core kernel in exact K-chunks); F32 uses the FFMA kernel (a last
 * wave at most half full is split over K, its partial sums in plan scratch);
 * anything else uses the generic CUDA-core kernel.  Staged operand transforms
 * (see gemm_epilogue_t) also write plan scratch.  All paths run on the GPU.
 * Errors: GEMM_ERR_INVALID_ARG / GEMM_ERR_UNSUPPORTED before any launch;
 * GEMM_ERR_CUDA when a launch or scratch allocation fails.
 * A plan's device scratch (int8 and operand-transform staging, stream-K and
 * split-tail partials, host staging) is
 * reused by every call: calls that use one plan from several streams or host
 * threads at once race on it; use one plan per concurrent stream.
 * Stream-K (environment GEMM_STREAM_K=1, off by default) lets CTA pairs of one
 * launch wait for each other's partial results; it assumes the launch's CTA
 * pairs are all resident, so kernels running concurrently on other streams can
 * delay it (every such wait is bounded and reports GEMM_ERR_TIMEOUT).
 * ------------------------------------------------------------------------- */
gemm_status_t gemm_run(gemm_plan_t plan, gemm_layout_t layoutA, gemm_layout_t layoutB,
                       int64_t M, int64_t N, int64_t K, double alpha,
                       const void* A, int64_t lda, const void* B, int64_t ldb, double beta,
                       const void* C, int64_t ldc, void* D, int64_t ldd,
                       const gemm_epilogue_t* epi, gemm_stream_t stream);

/* ---------------------------------------------------------------------------
 * gemm_run_strided_batched -- `batch` independent problems in one call:
 *     D_z = epilogue(alpha * op(A_z) * op(B_z) + beta * C_z),  z = 0 .. batch-1,
 * with X_z = X + z * stride_x (element strides) for A, B, C, D and the bias.
 * The batched GEMMs named among the motivations of "Flexible Performant GEMM
 * Kernels on GPUs" (section 3: requirements of the tiling API; section 4.1:
 * GEMM-based tensor contractions), run by the same kernels with the problem
 * index as an outer tile coordinate (TMA tensor maps with a third dimension).
 *   Arguments of one problem mean what they mean for gemm_run.
 *   stride_a, stride_b, stride_c, stride_bias  >= 0; 0 shares one operand
 *               (or bias vector) among all problems.
 *   stride_d    >= (M-1)*ldd + N when batch > 1 (outputs must not overlap);
 *               C == D requires stride_c == stride_d.
 *   batch       >= 0 (0: nothing is launched).
 * Strides whose byte size is not a multiple of 16, or more than 65535
 * problems, are served by one launch per problem.  Errors as for gemm_run.
 * ------------------------------------------------------------------------- */
gemm_status_t gemm_run_strided_batched(gemm_plan_t plan, gemm_layout_t layoutA, gemm_layout_t layoutB,
                                       int64_t M, int64_t N, int64_t K, double alpha,
                                       const void* A, int64_t lda, int64_t stride_a,
                                       const void* B, int64_t ldb, int64_t stride_b, double beta,
                                       const void* C, int64_t ldc, int64_t stride_c,
                                       void* D, int64_t ldd, int64_t stride_d, int64_t batch,
                                       const gemm_epilogue_t* epi, int64_t stride_bias,
                                       gemm_stream_t stream);

/* ---------------------------------------------------------------------------
 * gemm_run_diag -- GEMM with one diagonal operand, stored as its diagonal only:
 *     side GEMM_SIDE_LEFT:   D = epilogue(alpha * diag(d) * op(X) + beta * C)
 *                            (A = diag(d) is M x M, K = M, X plays B: M x N)
 *     side GEMM_SIDE_RIGHT:  D = epilogue(alpha * op(X) * diag(d) + beta * C)
 *                            (B = diag(d) is N x N, K = N, X plays A: M x N)
 * The diagonal-matrix GEMM of "Flexible Performant GEMM Kernels on GPUs",
 * section 5.2 (Table 1): a layout that yields zero off the diagonal without a
 * memory access, and a predicate that skips the inner-loop steps on those
 * zeros.  Together they leave one product per output, d[i]*x(i,j) (left) or
 * x(i,j)*d[j] (right), which the library computes directly (no tensor cores);
 * the result equals gemm_run on the materialised diagonal matrix.
 *   plan      any plan; its ab_dtype is the type of d and X, its c_dtype that of C.
 *   side      gemm_side_t.
 *   layoutX   GEMM_OP_N: X column-major, x(i,j) at X[i + j*ldx], ldx >= M;
 *             GEMM_OP_T: X row-major,    x(i,j) at X[i*ldx + j], ldx >= N.
 *   diag      device pointer to M (left) or N (right) contiguous entries.
 *   Other arguments mean what they mean for gemm_run (alpha, beta, C, D, the
 *   epilogue; S8 plans: integral alpha/beta, int32 arithmetic, exact).
 * Device pointers stay owned by the caller; nothing is allocated.
 * Errors: those of gemm_run for the equivalent dense call, plus
 * GEMM_ERR_INVALID_ARG for an unknown side.  gemm_plan_last_config reports
 * kernel GEMM_KERNEL_DIAG, the 64 x 64 output tile and the grid.
 * ------------------------------------------------------------------------- */
typedef enum { GEMM_SIDE_LEFT = 0 /* A = diag(d) */, GEMM_SIDE_RIGHT = 1 /* B = diag(d) */ } gemm_side_t;

gemm_status_t gemm_run_diag(gemm_plan_t plan, gemm_side_t side, gemm_layout_t layoutX,
                            int64_t M, int64_t N, double alpha, const void* diag,
                            const void* X, int64_t ldx, double beta,
                            const void* C, int64_t ldc, void* D, int64_t ldd,
                            const gemm_epilogue_t* epi, gemm_stream_t stream);

/* ---------------------------------------------------------------------------
 * gemm_run_complex -- the GEMM over complex or dual numbers:
 *     D = epilogue(alpha * op(A) * op(B) + beta * C),
 * every element a pair x + y*u, u the imaginary unit (GEMM_UNIT_IMAGINARY:
 * i*i = -1) or the dual unit (GEMM_UNIT_DUAL: eps*eps = 0), so that
 *     (a + b u)(c + d u) = (a c + b d u*u) + (a d + b c) u.
 * The complex and dual-number GEMMs of "Flexible Performant GEMM Kernels on
 * GPUs", section 5.4 (Figure 12), with its interleaved storage in global
 * memory: the pair of the element at storage offset e (layout and leading
 * dimension as for gemm_run, counted in pairs) occupies scalars 2e (real
 * part) and 2e + 1 (u part).  A, B, C, D and the bias are all interleaved.
 *   plan        ab_dtype F16, BF16 (tensor cores, fp32 accumulation) or F32
 *               (CUDA cores); c_dtype and the epilogue's out_dtype as for gemm_run.
 *   unit        gemm_unit_t.
 *   M, N, K, lda, ldb, ldc, ldd   in pairs; 2N and 2K must fit the kernels' 32-bit range.
 *   alpha, beta real scalars (beta == 0: C is not read).
 *   epi         bias: N pairs (GEMM_BIAS_COL; GEMM_BIAS_ROW returns
 *               GEMM_ERR_UNSUPPORTED); act and c_act act on each part alone.
 * Method: one real GEMM of size M x 2N x 2K on the same kernels as gemm_run.
 * A row-major (T) A is read in place as an M x 2K real matrix; B, and a
 * column-major (N) A, are first rearranged by a staging pass into plan-owned
 * device scratch (grown on demand, stream-ordered): 4 x B's bytes of scratch
 * for B, 2 x A's bytes for A (plus alignment padding).  Complex products cost
 * exactly their 4 real multiplies; dual products multiply one zero in four.
 * gemm_plan_last_config reports the real GEMM's launch (N' = 2N, K' = 2K).
 * Errors: those of gemm_run; GEMM_ERR_UNSUPPORTED for S8 plans.  Calls that
 * share a plan from several streams race on its scratch, as for gemm_run.
 * ------------------------------------------------------------------------- */
typedef enum { GEMM_UNIT_IMAGINARY = 0 /* complex */, GEMM_UNIT_DUAL = 1 /* dual */ } gemm_unit_t;

gemm_status_t gemm_run_complex(gemm_plan_t plan, gemm_unit_t unit, gemm_layout_t layoutA,
                               gemm_layout_t layoutB, int64_t M, int64_t N, int64_t K, double alpha,
                               const void* A, int64_t lda, const void* B, int64_t ldb, double beta,
                               const void* C, int64_t ldc, void* D, int64_t ldd,
                               const gemm_epilogue_t* epi, gemm_stream_t stream);

/* ---------------------------------------------------------------------------
 * gemm_run_host -- the same operation on HOST buffers (pinned or pageable).
 * Copies A, B, C (when beta != 0) and the bias into plan-owned device staging
 * (grown on demand), runs gemm_run, copies D back to the host and synchronises
 * `stream` before returning.  Arguments mean what they mean for gemm_run, with
 * host pointers; the bias pointer in `epi` is a host pointer too.  Host buffers
 * stay owned by the caller; only the N columns of each row of D are written.
 * Large problems (M >= 2048, 64 MB or more to move) run as a pipeline of row
 * panels over two plan-owned copy streams: B first, then each panel's rows of A
 * and C are copied in while the previous panel's GEMM runs on `stream` and the
 * one before it is copied out, so both directions of the host link stay busy.
 * Pinned host memory lets the copies overlap; pageable memory stays correct.
 * ------------------------------------------------------------------------- */
gemm_status_t gemm_run_host(gemm_plan_t plan, gemm_layout_t layoutA, gemm_layout_t layoutB,
                            int64_t M, int64_t N, int64_t K, double alpha,
                            const void* A, int64_t lda, const void* B, int64_t ldb, double beta,
                            const void* C, int64_t ldc, void* D, int64_t ldd,
                            const gemm_epilogue_t* epi, gemm_stream_t stream);

/* ---------------------------------------------------------------------------
 * gemm_validate -- the argument checks gemm_run performs, on the host only
 * (no device access; pointers are checked for NULL-ness, never dereferenced).
 * Returns GEMM_OK when gemm_run would accept the arguments for a plan of
 * (ab_dtype, c_dtype).
 * ------------------------------------------------------------------------- */
gemm_status_t gemm_validate(gemm_dtype_t ab_dtype, gemm_dtype_t c_dtype,
                            gemm_layout_t layoutA, gemm_layout_t layoutB,
                            int64_t M, int64_t N, int64_t K, double alpha,
                            const void* A, int64_t lda, const void* B, int64_t ldb, double beta,
                            const void* C, int64_t ldc, const void* D, int64_t ldd,
                            const gemm_epilogue_t* epi);

/* ---------------------------------------------------------------------------
 * gemm_select -- the tile-shape selector, on the host only.
 *   Inputs are those of gemm_run (pointers are used for their alignment only,
 *   never dereferenced) plus the SM count of the target device.
 *   out   the kernel, tile, pipeline depth, raster group and grid gemm_run
 *         would launch.
 * Paper counterpart: the defaulting heuristics of the params abstraction in
 * "Flexible Performant GEMM Kernels on GPUs" (section 4.2: the largest square
 * or nearly-square tile that fits in shared memory) and the shape-keyed
 * policies (a tall/skinny policy) of the CUTLASS page.
 * ------------------------------------------------------------------------- */
gemm_status_t gemm_select(gemm_dtype_t ab_dtype, gemm_dtype_t c_dtype,
                          gemm_layout_t layoutA, gemm_layout_t layoutB,
                          int64_t M, int64_t N, int64_t K,
                          const void* A, int64_t lda, const void* B, int64_t ldb,
                          const void* C, int64_t ldc, const void* D, int64_t ldd,
                          double beta, const gemm_epilogue_t* epi, int sm_count,
                          gemm_config_t* out);

/* Force a kernel for subsequent runs of `plan` (GEMM_KERNEL_AUTO restores the
 * selector).  A forced kernel that cannot serve a request makes gemm_run return
 * GEMM_ERR_ALIGNMENT or GEMM_ERR_UNSUPPORTED instead of running another one. */
gemm_status_t gemm_plan_set_kernel(gemm_plan_t plan, gemm_kernel_t kernel);

/* The configuration the most recent successful gemm_run of `plan` launched. */
gemm_status_t gemm_plan_last_config(gemm_plan_t plan, gemm_config_t* out);

/* Synchronise `stream`, then read and clear the plan's device error word.
 * *code is 0 when no kernel reported a failure; otherwise the status
 * (GEMM_ERR_TIMEOUT) of the first failure since the last read. */
gemm_status_t gemm_plan_device_status(gemm_plan_t plan, gemm_stream_t stream, int32_t* code);

/* Set the bound of every in-kernel wait, in nanoseconds (default 4e9).  A wait
 * that runs past it records GEMM_ERR_TIMEOUT in the error word and its CTA
 * winds down (waiting, again bounded, for its own copies in flight and
 * releasing its tensor memory) instead of spinning for ever. */
gemm_status_t gemm_plan_set_timeout(gemm_plan_t plan, uint64_t timeout_ns);

/* Human-readable name of a status code (static storage; never NULL). */
const char* gemm_status_string(gemm_status_t status);

/* ABI version of this header (major * 100 + minor): 109 (gemm_epilogue_t.c_act,
 * gemm_run_strided_batched, gemm_run_diag, gemm_run_complex, gemm_config_t.cluster,
 * gemm_epilogue_t.out_scale and int8 D, gemm_config_t.half_tiles,
 * gemm_noalloc_device_status and gemm_noalloc_set_timeout, the operand
 * transforms gemm_epilogue_t.load_xf / a_act / a_scale / b_act / b_scale). */
int gemm_abi_version(void);

/* ---------------------------------------------------------------------------
 * gemm_run_s8_noalloc -- the exact int8 GEMM (int32 accumulation) without
 * allocating any device memory.  It runs the int8 -> fp16 staging pass and the
 * single-CTA tensor-core int8 kernel (gemm_run on an S8 plan may take the
 * CTA-pair int8 kernel for large shapes instead; both give the same exact
 * result); with K == 0 it runs the generic CUDA-core kernel on beta*C alone.
 * The paper has no counterpart: this is a service of the library.
 *
 * Why: some callers cannot allocate device memory when they call the GEMM --
 * a process whose device memory was reserved up front by a framework's memory
 * pool (a cudaMalloc would fail or fragment the pool), a latency-bound loop
 * that must not pay for cudaMalloc/cudaFree and the synchronisation they
 * imply, or a program held to a memory budget fixed in advance.  gemm_run on
 * an S8 plan allocates its fp16 staging of A and B on demand and the plan
 * allocates an error word; this entry point needs neither a plan nor an
 * allocation: the staging lives in a fixed array inside the library,
 * GEMM_NOALLOC_SCRATCH_BYTES per device, which every GPU that loads the
 * library holds until the process exits.
 *
 *   Arguments mean what they mean for gemm_run with an (S8, S32) plan, on the
 *   current CUDA device; inputs and outputs are caller-owned device buffers.
 *   status  optional caller-owned device word (4 bytes) that receives
 *           GEMM_ERR_TIMEOUT if an in-kernel wait expires; NULL selects a word
 *           inside the library, which each call first clears to zero.
 * Limits: the staging needs 2 bytes per element of A's storage (rounded up to
 * 256 bytes) plus 2 bytes per element of B's storage; a problem needing more
 * than GEMM_NOALLOC_SCRATCH_BYTES returns GEMM_ERR_UNSUPPORTED before anything
 * is launched.  With K > 0, lda and ldb must be multiples of 8, else
 * GEMM_ERR_ALIGNMENT.
 * The first call on a device looks up the device address of the array
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture.
 * Every call shares the array, which keeps the last call's contents; calls
 * that overlap on the GPU (other streams, other host threads) race on it, so
 * the caller must serialise them.
 * No cudaMalloc, cudaFree or allocating library routine is called.
 * ------------------------------------------------------------------------- */
#define GEMM_NOALLOC_SCRATCH_BYTES (32u << 20)

gemm_status_t gemm_run_s8_noalloc(gemm_layout_t layoutA, gemm_layout_t layoutB,
                                  int64_t M, int64_t N, int64_t K, double alpha,
                                  const void* A, int64_t lda, const void* B, int64_t ldb,
                                  double beta, const void* C, int64_t ldc, void* D, int64_t ldd,
                                  const gemm_epilogue_t* epi, int32_t* status,
                                  gemm_stream_t stream);

/* Synchronise `stream`, then read and clear the library's own error word of
 * gemm_run_s8_noalloc on the current device (the word its calls with
 * status == NULL report to).  *code is 0 when no such call reported a failure
 * since the last read, else the status of the first one (GEMM_ERR_TIMEOUT).
 * Allocates nothing.  Like gemm_run_s8_noalloc, its first use on a device
 * looks up the word's device address; make that first call before any stream
 * capture.  The paper has no counterpart. */
gemm_status_t gemm_noalloc_device_status(int32_t* code, gemm_stream_t stream);

/* Set the bound, in nanoseconds (> 0; default 4e9), of the in-kernel waits of
 * every later gemm_run_s8_noalloc call in this process (all devices).  A wait
 * that runs past it records GEMM_ERR_TIMEOUT and its CTA winds down, as for
 * gemm_plan_set_timeout.  The paper has no counterpart. */
gemm_status_t gemm_noalloc_set_timeout(uint64_t timeout_ns);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_GEMM_EPILOGUES_GB300_GEMM_H */

/*
 * oracle.c -- plain, slow, obviously-correct CPU reference for the generalized
 * GEMM with a fused epilogue:
 *
 *     D[i,j] = cast_out( act( alpha * sum_k a(i,k) * b(k,j) + beta * C[i,j] + bias ) )
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the GPU library is
 * compared against.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load it.  It shares no code, header, table or helper with
 * the CUDA library: every conversion and index function below is written here
 * from its definition.
 *
 * Sources for what is computed (titles and sections of the pages):
 *   - "CUTLASS: Fast Linear Algebra in CUDA C++", section "Efficient Matrix
 *     Multiplication on GPUs": C = alpha*A*B + beta*C with A an MxK matrix,
 *     B a KxN matrix and C an MxN matrix; the plain three-loop dot-product
 *     form (i, j, k) and the reordered form with k outermost.
 *   - same page, "Fusing Element-wise Operations: An Example with SGEMM"
 *     (the fused_bias_relu_epilogue functor): result = alpha*acc + bias +
 *     beta*c, then clamped as max(threshold, result).
 *   - "Flexible Performant GEMM Kernels on GPUs", section 2.3 (Tensor Cores):
 *     D = A*B + C with 16-bit A/B and 32-bit C/D (mixed precision).
 *   - same paper, section 4.3 (Listing 9): D_ij = max(sum_k A_ik B_kj + C_ij, 0);
 *     section 4.3 (BLAS-like interface, Listing 10): C := alpha*A*B + beta*C
 *     with transposition of the inputs; section 5.1: the N (column-major) and
 *     T (row-major) layouts of A and B; section 5.3: a one-dimensional bias
 *     vector added to every row of the product.
 *   - section 3.2 (Figure 4): linearisation of a column-major (m, n) offset
 *     in an M-row parent as n*M + m.
 *
 * Readings where the pages leave a step open (each repeated in the design notes):
 *   - The bias is a vector of length N indexed by the column j ("added to every
 *     row"); BIAS_ROW (length M, indexed by i) is the transposed counterpart.
 *   - Order: alpha*acc + beta*C + bias, then the activation, then one rounding
 *     to the output type.  The ReLU threshold is 0.
 *   - An optional elementwise transform of C as it is read (c_act = ReLU:
 *     C[i,j] -> max(C[i,j], 0) before the beta product): the "ReLU on C" of
 *     "Flexible Performant GEMM Kernels on GPUs", section 5.3, Table 2, an
 *     instance of the transforms applied after every load of section 4.2.
 *   - Floating inputs are accumulated in fp64 (products of fp32/fp16/bf16
 *     values are exact in fp64); int8 inputs in int64 with integral alpha/beta.
 *   - beta == 0 means C is not read (it may be NULL), as in BLAS.
 *   - C and D are row-major M x N with leading dimensions ldc, ldd (>= N).
 *   - Casting to fp16/bf16 rounds to nearest, ties to even (IEEE 754), from
 *     the fp64 value in one step; fp32 output uses C's double->float conversion,
 *     which is the same rounding.  int32 output keeps the low 32 bits of the
 *     int64 value and counts every value outside the int32 range.
 *   - Optional elementwise transforms of A and B as they are read (the
 *     transforms applied after every load of "Flexible Performant GEMM Kernels
 *     on GPUs", section 4.2, Figure 10: a simple scaling, an activation):
 *     t(x) = act(scale * x) with act = none or ReLU (threshold 0), the scale
 *     applied first.  The tensor cores multiply 16-bit operands, so for fp16 and
 *     bf16 operands the transformed value is taken as the product in fp32
 *     (rounded to nearest even), then the activation, then rounded to nearest
 *     even back to the operand's own type; fp32 operands keep the fp32 value;
 *     int8 operands admit the activation only (any scale would leave the
 *     integers).  The sum then runs over t_A(a(i,k)) * t_B(b(k,j)).
 *   - int8 output of an int8 problem (the requantising cast): the int32 result v
 *     (low 32 bits, as above) is converted to fp32, multiplied by the fp32 scale
 *     out_scale, rounded to the nearest integer with ties to even, and saturated
 *     to [-128, 127].  The product is formed in fp32 on purpose: a floating step
 *     that decides an integer is taken in the precision the library takes it in.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* The oracle's own type codes.  (They happen to be small integers; nothing
 * here includes the library's header.) */
enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_S8 = 3, OR_S32 = 4 };
enum { OR_LAYOUT_N = 0, OR_LAYOUT_T = 1 };
enum { OR_ACT_NONE = 0, OR_ACT_RELU = 1 };
enum { OR_BIAS_NONE = 0, OR_BIAS_COL = 1, OR_BIAS_ROW = 2 };

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 and bfloat16 decoding/encoding, from their definitions.  */
/* ------------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)          v = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
    else if (e == 31)    v = f ? NAN : INFINITY;
    else                 v = ldexp((double)(1024 + f), e - 25);   /* (1 + f/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the upper half of a binary32 (1 sign, 8 exponent bits with bias 127,
 * 7 fraction bits). */
double oracle_bf16_to_double(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0)          v = ldexp((double)f, -133);              /* f * 2^(-126-7) */
    else if (e == 255)   v = f ? NAN : INFINITY;
    else                 v = ldexp((double)(128 + f), e - 134);   /* (1 + f/2^7) * 2^(e-127) */
    return sign ? -v : v;
}

/* Round a finite non-negative double x to a format with P fraction bits,
 * minimum normal exponent EMIN, and largest finite value MAXF (bits pattern
 * returned without sign).  Round to nearest, ties to even.  Written directly
 * from the definition: find the spacing (ulp) of the target format at x,
 * divide, round the quotient to the nearest integer (ties to even), scale back.
 * All steps are exact in double for the two formats used here. */
static double round_to_format(double x, int P, int EMIN) {
    if (x == 0.0) return 0.0;
    int ex;
    frexp(x, &ex);                 /* x = m * 2^ex, m in [0.5, 1) -> exponent of x is ex-1 */
    int e = ex - 1;
    if (e < EMIN) e = EMIN;        /* subnormal range shares the spacing of the smallest binade */
    double ulp = ldexp(1.0, e - P);
    double q = x / ulp;            /* exact: ulp is a power of two */
    double fl = floor(q);
    double rem = q - fl;
    double r;
    if (rem > 0.5)       r = fl + 1.0;
    else if (rem < 0.5)  r = fl;
    else                 r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;   /* tie -> even */
    return r * ulp;
}

uint16_t oracle_f16_from_double(double x) {
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return 0x7e00;
    double a = fabs(x);
    if (isinf(a)) return sign | 0x7c00;
    double r = round_to_format(a, 10, -14);
    if (r >= 65536.0) return sign | 0x7c00;   /* rounds past the largest finite value 65504 */
    if (r == 0.0) return sign;
    int ex;
    frexp(r, &ex);
    int e = ex - 1;
    if (e < -14) {                            /* subnormal: r = f * 2^-24 */
        return sign | (uint16_t)(r / ldexp(1.0, -24));
    }
    uint16_t f = (uint16_t)(ldexp(r, -e) * 1024.0 - 1024.0);
    return sign | (uint16_t)((e + 15) << 10) | f;
}

uint16_t oracle_bf16_from_double(double x) {
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return 0x7fc0;
    double a = fabs(x);
    if (isinf(a)) return sign | 0x7f80;
    double r = round_to_format(a, 7, -126);
    if (r >= ldexp(1.0, 128)) return sign | 0x7f80;   /* past the largest finite value */
    if (r == 0.0) return sign;
    int ex;
    frexp(r, &ex);
    int e = ex - 1;
    if (e < -126) {
        return sign | (uint16_t)(r / ldexp(1.0, -133));
    }
    uint16_t f = (uint16_t)(ldexp(r, -e) * 128.0 - 128.0);
    return sign | (uint16_t)((e + 127) << 7) | f;
}

/* ------------------------------------------------------------------------ */
/* Element access.                                                            */
/* ------------------------------------------------------------------------ */

static double load_float(int dtype, const void* p, int64_t idx) {
    switch (dtype) {
    case OR_F32:  return (double)((const float*)p)[idx];
    case OR_F16:  return oracle_f16_to_double(((const uint16_t*)p)[idx]);
    case OR_BF16: return oracle_bf16_to_double(((const uint16_t*)p)[idx]);
    case OR_S8:   return (double)((const int8_t*)p)[idx];
    case OR_S32:  return (double)((const int32_t*)p)[idx];
    default:      return NAN;
    }
}

static int64_t load_int(int dtype, const void* p, int64_t idx) {
    switch (dtype) {
    case OR_S8:  return (int64_t)((const int8_t*)p)[idx];
    case OR_S32: return (int64_t)((const int32_t*)p)[idx];
    default:     return 0;
    }
}

/* Storage offset of logical element (i, k) of A (M x K).
 * N: column-major, element (i, k) at i + k*lda (the linearisation n*M + m with
 *    the leading dimension as the column length).
 * T: row-major, element (i, k) at i*lda + k. */
static int64_t a_offset(int layout, int64_t i, int64_t k, int64_t lda) {
    return layout == OR_LAYOUT_N ? i + k * lda : i * lda + k;
}

/* Storage offset of logical element (k, j) of B (K x N). */
static int64_t b_offset(int layout, int64_t k, int64_t j, int64_t ldb) {
    return layout == OR_LAYOUT_N ? k + j * ldb : k * ldb + j;
}

typedef struct {
    int ab_dtype, layout_a, layout_b;
    int64_t M, N, K;
    double alpha, beta;
    const void *A, *B, *C, *bias;
    int64_t lda, ldb, ldc, ldd;
    int c_dtype, bias_dtype, bias_mode, act, d_dtype;
    int c_act;   /* transform applied to each C element as it is read */
    double out_scale;   /* int8 output: requantisation scale (applied in fp32) */
    int a_act;          /* transforms applied to each A and B element as it is read */
    double a_scale;
    int b_act;
    double b_scale;
} problem_t;

static int is_int_problem(const problem_t* p) { return p->ab_dtype == OR_S8; }

/* The epilogue for a floating-point problem: alpha*acc + beta*C + bias, then
 * the activation.  Returns the value before the output cast. */
static double epilogue_float(const problem_t* p, int64_t i, int64_t j, double acc) {
    double v = p->alpha * acc;
    if (p->beta != 0.0) {
        double c = load_float(p->c_dtype, p->C, i * p->ldc + j);
        if (p->c_act == OR_ACT_RELU) c = (c > 0.0) ? c : 0.0;
        v += p->beta * c;
    }
    if (p->bias_mode == OR_BIAS_COL) v += load_float(p->bias_dtype, p->bias, j);
    else if (p->bias_mode == OR_BIAS_ROW) v += load_float(p->bias_dtype, p->bias, i);
    if (p->act == OR_ACT_RELU) v = (v > 0.0) ? v : 0.0;
    return v;
}

static int64_t epilogue_int(const problem_t* p, int64_t i, int64_t j, int64_t acc) {
    int64_t alpha = (int64_t)p->alpha, beta = (int64_t)p->beta;
    int64_t v = alpha * acc;
    if (beta != 0) {
        int64_t c = load_int(p->c_dtype, p->C, i * p->ldc + j);
        if (p->c_act == OR_ACT_RELU) c = (c > 0) ? c : 0;
        v += beta * c;
    }
    if (p->bias_mode == OR_BIAS_COL) v += load_int(p->bias_dtype, p->bias, j);
    else if (p->bias_mode == OR_BIAS_ROW) v += load_int(p->bias_dtype, p->bias, i);
    if (p->act == OR_ACT_RELU) v = (v > 0) ? v : 0;
    return v;
}

/* Store a finished value into the output buffer at linear index idx. */
static void store_float(int dtype, void* D, int64_t idx, double v) {
    switch (dtype) {
    case OR_F32:  ((float*)D)[idx] = (float)v; break;
    case OR_F16:  ((uint16_t*)D)[idx] = oracle_f16_from_double(v); break;
    case OR_BF16: ((uint16_t*)D)[idx] = oracle_bf16_from_double(v); break;
    default: break;
    }
}

/* Returns 1 when v does not fit int32 (the low 32 bits are stored anyway). */
static int store_int(void* D, int64_t idx, int64_t v) {
    ((int32_t*)D)[idx] = (int32_t)(uint32_t)(uint64_t)v;
    return (v < INT32_MIN || v > INT32_MAX) ? 1 : 0;
}

/* The output of an int problem: int32, or int8 requantised (see the header). */
static int store_int_out(const problem_t* p, void* D, int64_t idx, int64_t v) {
    if (p->d_dtype != OR_S8) return store_int(D, idx, v);
    const int32_t v32 = (int32_t)(uint32_t)(uint64_t)v;
    const float prod = (float)v32 * (float)p->out_scale;    /* both roundings to nearest even, in fp32 */
    float r = nearbyintf(prod);                             /* ties to even (default rounding mode) */
    if (r > 127.0f) r = 127.0f;
    if (r < -128.0f) r = -128.0f;
    ((int8_t*)D)[idx] = (int8_t)r;
    return (v < INT32_MIN || v > INT32_MAX) ? 1 : 0;
}

/* The transform of one operand element after it is read (see the header):
 * act(scale * x), the product in fp32, rounded back to the operand's type. */
static double transform_operand(int dtype, double x, int act, double scale) {
    if (dtype == OR_S8) return (act == OR_ACT_RELU && x < 0.0) ? 0.0 : x;
    double v = (double)((float)scale * (float)x);
    if (act == OR_ACT_RELU) v = (v > 0.0) ? v : 0.0;
    if (dtype == OR_F16) return oracle_f16_to_double(oracle_f16_from_double(v));
    if (dtype == OR_BF16) return oracle_bf16_to_double(oracle_bf16_from_double(v));
    return v;   /* fp32: already an fp32 value */
}

static int has_transform(const problem_t* p) {
    return p->a_act != OR_ACT_NONE || p->b_act != OR_ACT_NONE || p->a_scale != 1.0 || p->b_scale != 1.0;
}

/* Decoding tables for the 16-bit formats: entry b is the value of bit pattern
 * b, filled once from the decoders above. */
static double f16_table[65536], bf16_table[65536];
static int tables_ready = 0;

static void init_tables(void) {
    if (tables_ready) return;
#pragma omp critical(oracle_tables)
    {
        if (!tables_ready) {
            for (int b = 0; b < 65536; ++b) {
                f16_table[b] = oracle_f16_to_double((uint16_t)b);
                bf16_table[b] = oracle_bf16_to_double((uint16_t)b);
            }
            tables_ready = 1;
        }
    }
}

/* sum_k a(i,k) * b(k,j), k ascending.  The storage position of a(i,k) moves by
 * a constant step as k grows (a_offset is affine in k), so the loop walks the
 * offsets from a_offset(i,0) and b_offset(0,j) by those steps. */
static double dot_float(const problem_t* p, int64_t i, int64_t j) {
    const int64_t a0 = a_offset(p->layout_a, i, 0, p->lda);
    const int64_t da = p->K > 1 ? a_offset(p->layout_a, i, 1, p->lda) - a0 : 0;
    const int64_t b0 = b_offset(p->layout_b, 0, j, p->ldb);
    const int64_t db = p->K > 1 ? b_offset(p->layout_b, 1, j, p->ldb) - b0 : 0;
    double acc = 0.0;
    int64_t ia = a0, ib = b0;
    if (has_transform(p)) {
        for (int64_t k = 0; k < p->K; ++k, ia += da, ib += db)
            acc += transform_operand(p->ab_dtype, load_float(p->ab_dtype, p->A, ia), p->a_act, p->a_scale) *
                   transform_operand(p->ab_dtype, load_float(p->ab_dtype, p->B, ib), p->b_act, p->b_scale);
        return acc;
    }
    switch (p->ab_dtype) {
    case OR_F32: {
        const float *A = (const float*)p->A, *B = (const float*)p->B;
        for (int64_t k = 0; k < p->K; ++k, ia += da, ib += db) acc += (double)A[ia] * (double)B[ib];
        break;
    }
    case OR_F16: {
        const uint16_t *A = (const uint16_t*)p->A, *B = (const uint16_t*)p->B;
        for (int64_t k = 0; k < p->K; ++k, ia += da, ib += db) acc += f16_table[A[ia]] * f16_table[B[ib]];
        break;
    }
    case OR_BF16: {
        const uint16_t *A = (const uint16_t*)p->A, *B = (const uint16_t*)p->B;
        for (int64_t k = 0; k < p->K; ++k, ia += da, ib += db) acc += bf16_table[A[ia]] * bf16_table[B[ib]];
        break;
    }
    default:
        for (int64_t k = 0; k < p->K; ++k, ia += da, ib += db)
            acc += load_float(p->ab_dtype, p->A, ia) * load_float(p->ab_dtype, p->B, ib);
    }
    return acc;
}

static int64_t dot_int(const problem_t* p, int64_t i, int64_t j) {
    const int64_t a0 = a_offset(p->layout_a, i, 0, p->lda);
    const int64_t da = p->K > 1 ? a_offset(p->layout_a, i, 1, p->lda) - a0 : 0;
    const int64_t b0 = b_offset(p->layout_b, 0, j, p->ldb);
    const int64_t db = p->K > 1 ? b_offset(p->layout_b, 1, j, p->ldb) - b0 : 0;
    const int8_t *A = (const int8_t*)p->A, *B = (const int8_t*)p->B;
    int64_t acc = 0, ia = a0, ib = b0;
    if (has_transform(p)) {
        for (int64_t k = 0; k < p->K; ++k, ia += da, ib += db) {
            const int64_t a = (p->a_act == OR_ACT_RELU && A[ia] < 0) ? 0 : A[ia];
            const int64_t b = (p->b_act == OR_ACT_RELU && B[ib] < 0) ? 0 : B[ib];
            acc += a * b;
        }
        return acc;
    }
    for (int64_t k = 0; k < p->K; ++k, ia += da, ib += db) acc += (int64_t)A[ia] * (int64_t)B[ib];
    return acc;
}

/* One output element in the dot-product order: sum over k for fixed (i, j). */
static int64_t element_ijk(const problem_t* p, int64_t i, int64_t j, void* D, int64_t out_idx) {
    if (is_int_problem(p)) return store_int_out(p, D, out_idx, epilogue_int(p, i, j, dot_int(p, i, j)));
    store_float(p->d_dtype, D, out_idx, epilogue_float(p, i, j, dot_float(p, i, j)));
    return 0;
}

static int valid_problem(const problem_t* p) {
    if (p->M < 0 || p->N < 0 || p->K < 0) return 0;
    if (p->ab_dtype < OR_F32 || p->ab_dtype > OR_S8) return 0;
    if (p->K > 0) {   /* K == 0 is an empty sum: A and B are not read */
        if (p->layout_a == OR_LAYOUT_N ? p->lda < (p->M > 1 ? p->M : 1) : p->lda < (p->K > 1 ? p->K : 1)) return 0;
        if (p->layout_b == OR_LAYOUT_N ? p->ldb < (p->K > 1 ? p->K : 1) : p->ldb < (p->N > 1 ? p->N : 1)) return 0;
    }
    if (p->ldd < p->N) return 0;
    if (p->beta != 0.0 && (p->C == NULL || p->ldc < p->N)) return 0;
    if (p->bias_mode != OR_BIAS_NONE && p->bias == NULL) return 0;
    if (p->c_act != OR_ACT_NONE && p->c_act != OR_ACT_RELU) return 0;
    if (p->a_act != OR_ACT_NONE && p->a_act != OR_ACT_RELU) return 0;
    if (p->b_act != OR_ACT_NONE && p->b_act != OR_ACT_RELU) return 0;
    if (!isfinite(p->a_scale) || !isfinite(p->b_scale)) return 0;
    if (is_int_problem(p) && (p->a_scale != 1.0 || p->b_scale != 1.0)) return 0;
    if (is_int_problem(p)) {
        if (p->d_dtype != OR_S32 && p->d_dtype != OR_S8) return 0;
        if (p->d_dtype == OR_S8 && !isfinite(p->out_scale)) return 0;
        if (p->alpha != floor(p->alpha) || p->beta != floor(p->beta)) return 0;
    } else if (p->d_dtype == OR_S32 || p->d_dtype == OR_S8) {
        return 0;
    }
    return 1;
}

/*
 * Full GEMM.  loop_order 0: i, j, k (dot-product form, parallel over rows i
 * with nthreads threads).  loop_order 1: k outermost, accumulating outer
 * products of column k of A and row k of B into an M x N accumulator (single
 * thread; for small cross-checks).
 * Returns the number of int32 overflows (int problems), 0, or -1 for invalid
 * arguments.
 */
int64_t oracle_gemm(int ab_dtype, int layout_a, int layout_b,
                    int64_t M, int64_t N, int64_t K,
                    double alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
                    double beta, int c_dtype, const void* C, int64_t ldc,
                    int bias_dtype, const void* bias, int bias_mode, int act, int c_act,
                    int d_dtype, void* D, int64_t ldd,
                    int loop_order, int nthreads, double out_scale,
                    int a_act, double a_scale, int b_act, double b_scale) {
    problem_t p = {ab_dtype, layout_a, layout_b, M, N, K, alpha, beta, A, B, C, bias,
                   lda, ldb, ldc, ldd, c_dtype, bias_dtype, bias_mode, act, d_dtype, c_act, out_scale,
                   a_act, a_scale, b_act, b_scale};
    if (!valid_problem(&p)) return -1;
    if (M == 0 || N == 0) return 0;
    init_tables();
    int64_t overflow = 0;
    if (loop_order == 0) {
        if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(+ : overflow)
        for (int64_t i = 0; i < M; ++i)
            for (int64_t j = 0; j < N; ++j)
                overflow += element_ijk(&p, i, j, D, i * ldd + j);
        return overflow;
    }
    /* k-outer form */
    if (is_int_problem(&p)) {
        int64_t* acc = (int64_t*)calloc((size_t)(M * N), sizeof(int64_t));
        if (!acc) return -1;
        for (int64_t k = 0; k < K; ++k)
            for (int64_t i = 0; i < M; ++i)
                for (int64_t j = 0; j < N; ++j)
                    acc[i * N + j] += (int64_t)transform_operand(OR_S8, (double)load_int(ab_dtype, A, a_offset(layout_a, i, k, lda)), a_act, 1.0) *
                                      (int64_t)transform_operand(OR_S8, (double)load_int(ab_dtype, B, b_offset(layout_b, k, j, ldb)), b_act, 1.0);
        for (int64_t i = 0; i < M; ++i)
            for (int64_t j = 0; j < N; ++j)
                overflow += store_int_out(&p, D, i * ldd + j, epilogue_int(&p, i, j, acc[i * N + j]));
        free(acc);
        return overflow;
    }
    double* acc = (double*)calloc((size_t)(M * N), sizeof(double));
    if (!acc) return -1;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t i = 0; i < M; ++i)
            for (int64_t j = 0; j < N; ++j)
                acc[i * N + j] += transform_operand(ab_dtype, load_float(ab_dtype, A, a_offset(layout_a, i, k, lda)), a_act, a_scale) *
                                  transform_operand(ab_dtype, load_float(ab_dtype, B, b_offset(layout_b, k, j, ldb)), b_act, b_scale);
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            store_float(d_dtype, D, i * ldd + j, epilogue_float(&p, i, j, acc[i * N + j]));
    free(acc);
    return 0;
}

/*
 * Selected entries only: out[e] = D[rows[e], cols[e]] (in d_dtype, packed
 * contiguously), computed in the dot-product order.  Used to check outputs of
 * problems too large for the full oracle.  Returns overflows or -1.
 */
int64_t oracle_gemm_entries(int ab_dtype, int layout_a, int layout_b,
                            int64_t M, int64_t N, int64_t K,
                            double alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
                            double beta, int c_dtype, const void* C, int64_t ldc,
                            int bias_dtype, const void* bias, int bias_mode, int act, int c_act,
                            int d_dtype, int64_t n_entries, const int64_t* rows, const int64_t* cols,
                            void* out, int nthreads, double out_scale,
                            int a_act, double a_scale, int b_act, double b_scale) {
    problem_t p = {ab_dtype, layout_a, layout_b, M, N, K, alpha, beta, A, B, C, bias,
                   lda, ldb, ldc, N, c_dtype, bias_dtype, bias_mode, act, d_dtype, c_act, out_scale,
                   a_act, a_scale, b_act, b_scale};
    if (!valid_problem(&p)) return -1;
    for (int64_t e = 0; e < n_entries; ++e)
        if (rows[e] < 0 || rows[e] >= M || cols[e] < 0 || cols[e] >= N) return -1;
    init_tables();
    int64_t overflow = 0;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 16) num_threads(nthreads) reduction(+ : overflow)
    for (int64_t e = 0; e < n_entries; ++e)
        overflow += element_ijk(&p, rows[e], cols[e], out, e);
    return overflow;
}

/* ------------------------------------------------------------------------ */
/* GEMM over complex or dual numbers.                                         */
/* ------------------------------------------------------------------------ */
/*
 * "Flexible Performant GEMM Kernels on GPUs", section 5.4: a complex GEMM
 * multiplies numbers x + y*i with i*i = -1; a dual-number GEMM numbers
 * x + y*eps with eps*eps = 0.  Writing u for the unit, one product is
 *     (a + b u)(c + d u) = (a c + b d u^2) + (a d + b c) u,
 * so u^2 = -1 gives (ac - bd) + (ad + bc) i and u^2 = 0 gives ac + (ad + bc) eps.
 * The matrices are stored interleaved, as that section describes for global
 * memory: the pair of the logical element at storage offset e (from the layout
 * functions above, in pairs) sits at scalar positions 2e (the real part) and
 * 2e + 1 (the u part); A, B, C, D and the bias all hold such pairs.
 *
 * Readings taken here:
 *   - D = epilogue(alpha * sum_k a(i,k) b(k,j) + beta * C) with REAL alpha and
 *     beta (the section's D = A*B + C is alpha = beta = 1); sums in fp64.
 *   - The bias is a vector of pairs (N of them, by column, or M by row) added
 *     to the pair of each output; c_act and act apply to each of the two parts
 *     on its own (the pages define no activation of a complex number), and
 *     each part is rounded on its own to the output type.
 */
enum { OR_UNIT_IMAGINARY = 0, OR_UNIT_DUAL = 1 };

/* One finished output pair (i, j) into out[2*out_idx], out[2*out_idx + 1]. */
static void element_pair(const problem_t* p, int unit, int64_t i, int64_t j, void* out, int64_t out_idx) {
    const double u2 = unit == OR_UNIT_IMAGINARY ? -1.0 : 0.0;   /* the square of the unit */
    double re = 0.0, im = 0.0;
    for (int64_t k = 0; k < p->K; ++k) {
        const int64_t ea = a_offset(p->layout_a, i, k, p->lda);
        const int64_t eb = b_offset(p->layout_b, k, j, p->ldb);
        const double a = load_float(p->ab_dtype, p->A, 2 * ea), b = load_float(p->ab_dtype, p->A, 2 * ea + 1);
        const double c = load_float(p->ab_dtype, p->B, 2 * eb), d = load_float(p->ab_dtype, p->B, 2 * eb + 1);
        re += a * c + u2 * (b * d);
        im += a * d + b * c;
    }
    double acc[2] = {re, im};
    for (int part = 0; part < 2; ++part) {
        double v = p->alpha * acc[part];
        if (p->beta != 0.0) {
            double cv = load_float(p->c_dtype, p->C, 2 * (i * p->ldc + j) + part);
            if (p->c_act == OR_ACT_RELU) cv = (cv > 0.0) ? cv : 0.0;
            v += p->beta * cv;
        }
        if (p->bias_mode == OR_BIAS_COL) v += load_float(p->bias_dtype, p->bias, 2 * j + part);
        else if (p->bias_mode == OR_BIAS_ROW) v += load_float(p->bias_dtype, p->bias, 2 * i + part);
        if (p->act == OR_ACT_RELU) v = (v > 0.0) ? v : 0.0;
        store_float(p->d_dtype, out, 2 * out_idx + part, v);
    }
}

static int valid_pair_problem(const problem_t* p, int unit) {
    if (unit != OR_UNIT_IMAGINARY && unit != OR_UNIT_DUAL) return 0;
    if (p->ab_dtype == OR_S8 || p->ab_dtype == OR_S32) return 0;   /* floating parts only */
    return valid_problem(p);
}

/* Full complex / dual GEMM (dot-product order, rows in parallel).  Sizes and
 * leading dimensions count pairs.  Returns 0, or -1 for invalid arguments. */
int64_t oracle_gemm_pairs(int unit, int ab_dtype, int layout_a, int layout_b,
                          int64_t M, int64_t N, int64_t K,
                          double alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
                          double beta, int c_dtype, const void* C, int64_t ldc,
                          int bias_dtype, const void* bias, int bias_mode, int act, int c_act,
                          int d_dtype, void* D, int64_t ldd, int nthreads) {
    problem_t p = {ab_dtype, layout_a, layout_b, M, N, K, alpha, beta, A, B, C, bias,
                   lda, ldb, ldc, ldd, c_dtype, bias_dtype, bias_mode, act, d_dtype, c_act, 1.0,
                   OR_ACT_NONE, 1.0, OR_ACT_NONE, 1.0};
    if (!valid_pair_problem(&p, unit)) return -1;
    if (M == 0 || N == 0) return 0;
    init_tables();
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            element_pair(&p, unit, i, j, D, i * ldd + j);
    return 0;
}

/* Selected output pairs only: out[2e], out[2e+1] = D[rows[e], cols[e]]. */
int64_t oracle_gemm_pairs_entries(int unit, int ab_dtype, int layout_a, int layout_b,
                                  int64_t M, int64_t N, int64_t K,
                                  double alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
                                  double beta, int c_dtype, const void* C, int64_t ldc,
                                  int bias_dtype, const void* bias, int bias_mode, int act, int c_act,
                                  int d_dtype, int64_t n_entries, const int64_t* rows,
                                  const int64_t* cols, void* out, int nthreads) {
    problem_t p = {ab_dtype, layout_a, layout_b, M, N, K, alpha, beta, A, B, C, bias,
                   lda, ldb, ldc, N, c_dtype, bias_dtype, bias_mode, act, d_dtype, c_act, 1.0,
                   OR_ACT_NONE, 1.0, OR_ACT_NONE, 1.0};
    if (!valid_pair_problem(&p, unit)) return -1;
    for (int64_t e = 0; e < n_entries; ++e)
        if (rows[e] < 0 || rows[e] >= M || cols[e] < 0 || cols[e] >= N) return -1;
    init_tables();
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 16) num_threads(nthreads)
    for (int64_t e = 0; e < n_entries; ++e)
        element_pair(&p, unit, rows[e], cols[e], out, e);
    return 0;
}

/* Threads the OpenMP runtime would use by default (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

// diag_kernel.cu -- GEMM with one diagonal operand (sm_103a).
//
// "Flexible Performant GEMM Kernels on GPUs", section 5.2: with A (or B) a
// diagonal matrix, a layout that answers zero off the diagonal without touching
// memory, plus a predicate that skips the inner-loop iterations on those
// zeros, leaves exactly one product per output:
//     A = diag(d):  D[i,j] = epilogue(alpha * d[i] * x(i,j) + beta * C[i,j] + bias)
//     B = diag(d):  D[i,j] = epilogue(alpha * x(i,j) * d[j] + beta * C[i,j] + bias)
// where x is the dense operand (B, or A) seen as an M x N matrix.  Taken to its
// end on GB300 that is an HBM-bound elementwise pass over x, C and D: no zero is
// stored or loaded and no tensor-core instruction is issued.
//
// Two kernels share the arithmetic.  The TMA-staged kernel (16-bit x, and C
// absent or fp32/fp16/bf16, every operand TMA-alignable) keeps the bytes in
// flight in shared memory instead of registers: one producer thread per CTA
// streams 64 x 64 boxes of x and C, and the tile's 64 entries of the diagonal
// and of the bias, with TMA into a ring of stages, one CTA per
// SM, and sixteen consumer warps finish each tile from shared memory (lane = row,
// eight consecutive columns per lane, so every D store writes whole 32-byte
// sectors).  The register kernel below serves every other type and alignment.
//
// Register kernel work decomposition: 64 x 64 tiles of D, CTAs persistent over the tiles; each
// thread owns two 8-wide row segments of a tile.  x, C and D move as aligned
// 8-element vectors where the host found the rows (columns) aligned, scalars
// otherwise and at ragged edges.  A column-major x is read column-contiguous
// and turned around in shared memory, so both its reads and D's row-major
// writes stay coalesced.  All loads of a tile (x and C) are issued before the
// first use.
#include <atomic>
#include <type_traits>

#include "kernels.h"

namespace gemmlib {
namespace {

constexpr int DG_THREADS = 256;
constexpr int DG_SEGS = DIAG_TM * DIAG_TN / 8 / DG_THREADS;   // 8-wide segments per thread (2)
static_assert(DIAG_TM % 8 == 0 && DIAG_TN % 8 == 0, "tiles hold whole 8-element vectors");
static_assert(DG_THREADS % (DIAG_TN / 8) == 0, "a thread's segments share one column range");

// --------------------------- 8-element vectors ------------------------------

template <typename T>
__device__ __forceinline__ void ld_vec8(const T* p, T (&v)[8]) {
  if constexpr (sizeof(T) == 1) {
    const uint2 r = *reinterpret_cast<const uint2*>(p);
    memcpy(v, &r, 8);
  } else if constexpr (sizeof(T) == 2) {
    const uint4 r = *reinterpret_cast<const uint4*>(p);
    memcpy(v, &r, 16);
  } else if ((reinterpret_cast<uintptr_t>(p) & 31) == 0) {
    // One 32-byte access per lane: a warp's request covers whole 32-byte sectors.
    uint32_t w[8];
    asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
    memcpy(v, w, 32);
  } else {
    const uint4 r0 = reinterpret_cast<const uint4*>(p)[0];
    const uint4 r1 = reinterpret_cast<const uint4*>(p)[1];
    memcpy(v, &r0, 16);
    memcpy(v + 4, &r1, 16);
  }
}

template <typename T>
__device__ __forceinline__ void st_vec8(T* p, const T (&v)[8]) {
  if constexpr (sizeof(T) == 2) {
    uint4 r;
    memcpy(&r, v, 16);
    *reinterpret_cast<uint4*>(p) = r;
  } else if ((reinterpret_cast<uintptr_t>(p) & 31) == 0) {
    // One 32-byte store per lane writes whole sectors; two 16-byte stores per lane
    // leave every sector half written by each instruction, which halves the
    // write bandwidth.
    uint32_t w[8];
    memcpy(w, v, 32);
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
  } else {
    uint4 r0, r1;
    memcpy(&r0, v, 16);
    memcpy(&r1, v + 4, 16);
    reinterpret_cast<uint4*>(p)[0] = r0;
    reinterpret_cast<uint4*>(p)[1] = r1;
  }
}

template <typename T> __device__ __forceinline__ float to_float(T v) { return (float)v; }
template <> __device__ __forceinline__ float to_float<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_float<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

// Elements idx .. idx+n-1 (n <= 8) of a typed array, widened to Acc; the rest 0.
// `vec`: the 8 elements form one aligned vector (taken only when n == 8).
template <typename T, typename Acc>
__device__ __forceinline__ void load8(const T* p, int64_t idx, bool vec, int n, Acc (&out)[8]) {
  if (vec && n == 8) {
    T v[8];
    ld_vec8(p + idx, v);
#pragma unroll
    for (int t = 0; t < 8; ++t) out[t] = (Acc)to_float(v[t]);
  } else {
#pragma unroll
    for (int t = 0; t < 8; ++t) out[t] = t < n ? (Acc)to_float(p[idx + t]) : (Acc)0;
  }
}

// The same for an int8 array widened to int32 (exact).
__device__ __forceinline__ void load8(const int8_t* p, int64_t idx, bool vec, int n, int32_t (&out)[8]) {
  if (vec && n == 8) {
    int8_t v[8];
    ld_vec8(p + idx, v);
#pragma unroll
    for (int t = 0; t < 8; ++t) out[t] = v[t];
  } else {
#pragma unroll
    for (int t = 0; t < 8; ++t) out[t] = t < n ? (int32_t)p[idx + t] : 0;
  }
}

__device__ __forceinline__ void load8(const int32_t* p, int64_t idx, bool vec, int n, int32_t (&out)[8]) {
  if (vec && n == 8) {
    ld_vec8(p + idx, out);
  } else {
#pragma unroll
    for (int t = 0; t < 8; ++t) out[t] = t < n ? p[idx + t] : 0;
  }
}

// C elements (runtime dtype) as float.
__device__ __forceinline__ void load8_c(const void* C, int dt, int64_t idx, bool vec, int n, float (&out)[8]) {
  switch (dt) {
    case GEMM_F32: load8(static_cast<const float*>(C), idx, vec, n, out); break;
    case GEMM_F16: load8(static_cast<const __half*>(C), idx, vec, n, out); break;
    default: load8(static_cast<const __nv_bfloat16*>(C), idx, vec, n, out); break;
  }
}

template <typename T>
__device__ __forceinline__ T from_float(float v) { return v; }
template <> __device__ __forceinline__ __half from_float<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

template <typename T>
__device__ __forceinline__ void store8_typed(T* p, int64_t idx, bool vec, int n, const float (&v)[8]) {
  if (vec && n == 8) {
    T w[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) w[t] = from_float<T>(v[t]);
    st_vec8(p + idx, w);
  } else {
#pragma unroll
    for (int t = 0; t < 8; ++t)
      if (t < n) p[idx + t] = from_float<T>(v[t]);
  }
}

__device__ __forceinline__ void store8_d(void* D, int dt, int64_t idx, bool vec, int n, const float (&v)[8]) {
  switch (dt) {
    case GEMM_F32: store8_typed(static_cast<float*>(D), idx, vec, n, v); break;
    case GEMM_F16: store8_typed(static_cast<__half*>(D), idx, vec, n, v); break;
    default: store8_typed(static_cast<__nv_bfloat16*>(D), idx, vec, n, v); break;
  }
}

__device__ __forceinline__ void store8_d(void* D, int dt, int64_t idx, bool vec, int n, const int32_t (&v)[8],
                                         float out_scale) {
  if (dt == GEMM_S8) {   // requantised int8 D
    int8_t* q = static_cast<int8_t*>(D);
#pragma unroll
    for (int t = 0; t < 8; ++t)
      if (t < n) q[idx + t] = requant_s8(v[t], out_scale);
    return;
  }
  int32_t* p = static_cast<int32_t*>(D);
  if (vec && n == 8) {
    st_vec8(p + idx, v);
  } else {
#pragma unroll
    for (int t = 0; t < 8; ++t)
      if (t < n) p[idx + t] = v[t];
  }
}

__device__ __forceinline__ int clamp8(int64_t v) { return v <= 0 ? 0 : (v >= 8 ? 8 : (int)v); }

// All lanes of a warp wait; the warp gives up together if any lane gave up.
__device__ __forceinline__ bool warp_all_wait(uint32_t bar, uint32_t parity, const WaitCtx& wc) {
  const bool ok = mbar_wait(bar, parity, wc);
  return __all_sync(0xffffffffu, ok) != 0;
}

// ------------------------------- the kernel ---------------------------------

template <typename XT, bool X_ROW_MAJOR>
__global__ void __launch_bounds__(DG_THREADS) diag_gemm_kernel(const DiagParams p) {
  constexpr bool IS_INT = std::is_same<XT, int8_t>::value;
  using Acc = typename std::conditional<IS_INT, int32_t, float>::type;
  // Column-major x is turned around here (one element of padding per row
  // spreads the transposed accesses over the banks).
  __shared__ Acc turn[X_ROW_MAJOR ? 1 : DIAG_TM][DIAG_TN + 1];

  const XT* X = static_cast<const XT*>(p.X);
  const XT* dg = static_cast<const XT*>(p.diag);
  const EpiParams& e = p.epi;
  const EpiPtrs ptr = epi_ptrs(e, 0);
  const int tid = threadIdx.x;
  // This thread's output segments in every tile: rows r0 + 32*q, columns c8 .. c8+7.
  const int c8 = (tid % (DIAG_TN / 8)) * 8;
  const int r0 = tid / (DIAG_TN / 8);
  constexpr int ROW_STEP = DG_THREADS / (DIAG_TN / 8);

  for (int64_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
    const int64_t i0 = (t / p.tiles_n) * DIAG_TM;
    const int64_t j0 = (t % p.tiles_n) * DIAG_TN;
    const int64_t j = j0 + c8;
    const int n_out = clamp8(p.N - j);

    // 1. x for this thread's segments (row-major: directly; column-major: the
    //    column slices that the thread carries to shared memory).
    Acc x[DG_SEGS][8];
#pragma unroll
    for (int q = 0; q < DG_SEGS; ++q) {
      if constexpr (X_ROW_MAJOR) {
        const int64_t i = i0 + r0 + q * ROW_STEP;
        load8(X, i * p.ldx + j, p.vec_x != 0, i < p.M ? n_out : 0, x[q]);
      } else {
        const int v = tid + q * DG_THREADS;
        const int64_t ci = i0 + (v % (DIAG_TM / 8)) * 8;   // 8 consecutive rows ...
        const int64_t cj = j0 + v / (DIAG_TM / 8);         // ... of one column
        load8(X, ci + cj * p.ldx, p.vec_x != 0, cj < p.N ? clamp8(p.M - ci) : 0, x[q]);
      }
    }

    // 2. C for the same output segments (in flight together with x).
    Acc c[DG_SEGS][8];
    if (e.read_c) {
#pragma unroll
      for (int q = 0; q < DG_SEGS; ++q) {
        const int64_t i = i0 + r0 + q * ROW_STEP;
        const int n = i < p.M ? n_out : 0;
        if constexpr (IS_INT) load8(static_cast<const int32_t*>(ptr.C), i * e.ldc + j, e.vec_c != 0, n, c[q]);
        else load8_c(ptr.C, e.c_dtype, i * e.ldc + j, e.vec_c != 0, n, c[q]);
        if (e.c_relu) {
#pragma unroll
          for (int u = 0; u < 8; ++u) c[q][u] = c[q][u] > (Acc)0 ? c[q][u] : (Acc)0;
        }
      }
    }

    // 3. Column-major x: through shared memory into the output segments.
    if constexpr (!X_ROW_MAJOR) {
      __syncthreads();   // the previous tile's reads of `turn` are done
#pragma unroll
      for (int q = 0; q < DG_SEGS; ++q) {
        const int v = tid + q * DG_THREADS;
        const int rr = (v % (DIAG_TM / 8)) * 8, cc = v / (DIAG_TM / 8);
#pragma unroll
        for (int u = 0; u < 8; ++u) turn[rr + u][cc] = x[q][u];
      }
      __syncthreads();
#pragma unroll
      for (int q = 0; q < DG_SEGS; ++q) {
        const int rr = r0 + q * ROW_STEP;
#pragma unroll
        for (int u = 0; u < 8; ++u) x[q][u] = turn[rr][c8 + u];
      }
    }

    // 4. The one product per output, the fused epilogue, row-major D.
    Acc dcol[8];   // right diagonal: d[j .. j+7]
    if (!p.left) load8(dg, j, p.vec_diag != 0, n_out, dcol);
#pragma unroll
    for (int q = 0; q < DG_SEGS; ++q) {
      const int64_t i = i0 + r0 + q * ROW_STEP;
      if (i >= p.M || n_out == 0) continue;
      const Acc drow = p.left ? (Acc)to_float(dg[i]) : (Acc)0;
      Acc v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const Acc d = p.left ? drow : dcol[u];
        if constexpr (IS_INT) {
          v[u] = wrap_madd(e.alpha_i, d * x[q][u], 0);   // |d * x| <= 2^14: exact
          if (e.read_c) v[u] = wrap_madd(e.beta_i, c[q][u], v[u]);
        } else {
          v[u] = e.alpha * (d * x[q][u]);
          if (e.read_c) v[u] = fmaf(e.beta, c[q][u], v[u]);
        }
      }
      if (e.bias_mode == GEMM_BIAS_COL) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (u >= n_out) break;
          if constexpr (IS_INT) v[u] = wrap_madd(1, load_as_int(ptr.bias, GEMM_S32, j + u), v[u]);
          else v[u] += load_as_float(ptr.bias, e.bias_dtype, j + u);
        }
      } else if (e.bias_mode == GEMM_BIAS_ROW) {
        if constexpr (IS_INT) {
          const int32_t b = load_as_int(ptr.bias, GEMM_S32, i);
#pragma unroll
          for (int u = 0; u < 8; ++u) v[u] = wrap_madd(1, b, v[u]);
        } else {
          const float b = load_as_float(ptr.bias, e.bias_dtype, i);
#pragma unroll
          for (int u = 0; u < 8; ++u) v[u] += b;
        }
      }
      if (e.relu) {
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = v[u] > (Acc)0 ? v[u] : (Acc)0;
      }
      if constexpr (IS_INT) store8_d(ptr.D, e.d_dtype, i * e.ldd + j, e.vec_d != 0, n_out, v, e.out_scale);
      else store8_d(ptr.D, e.d_dtype, i * e.ldd + j, e.vec_d != 0, n_out, v);
    }
  }
}

// ------------------------- the TMA-staged kernel ----------------------------

// Sixteen consumer warps, one 32-row x 8-column task each per tile: with eight
// (two tasks each) the consumers could not keep up (4096^2, fp16 x, fp32 C and
// D: 30.5 / 33.2 us for row- / column-major x against 27.8 / 28.5 us with 16).
constexpr int DT_CONS_WARPS = 16;
constexpr int DT_THREADS = 32 * (DT_CONS_WARPS + 1);        // + one producer warp
constexpr int DT_X_BYTES = DIAG_TM * DIAG_TN * 2;           // 8 KiB: a 16-bit x box
constexpr int DT_C_BYTES = DIAG_TM * DIAG_TN * 4;           // 16 KiB: fp32 C (16-bit C uses half)
constexpr int DT_V_OFF = DT_X_BYTES + DT_C_BYTES;           // the tile's 64 diagonal entries (16-bit)
constexpr int DT_BIAS_OFF = DT_V_OFF + 128;                 // the tile's 64 bias entries (up to fp32)
constexpr int DT_STAGE_BYTES = DT_X_BYTES + DT_C_BYTES + 1024;   // whole KiBs keep the boxes 1024-aligned
constexpr size_t DT_SMEM = 1024 + (size_t)DIAG_TMA_STAGES * DT_STAGE_BYTES + 2 * DIAG_TMA_STAGES * 8 + 16;
static_assert(DIAG_TM == 64 && DIAG_TN == 64 && DT_CONS_WARPS == 16, "16 tasks of 32 rows x 8 columns per 64 x 64 box");

// Byte offset of 16-byte chunk q of row R in a box stored with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128(uint32_t R, uint32_t q) { return R * 128u + ((q ^ (R & 7u)) << 4); }

__device__ __forceinline__ float h16_to_float(uint16_t b, bool bf16) {
  if (bf16) return __uint_as_float((uint32_t)b << 16);
  return __half2float(__ushort_as_half(b));
}

template <bool X_ROW_MAJOR>
__global__ void __launch_bounds__(DT_THREADS, 1) diag_tma_kernel(const __grid_constant__ DiagParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;        // swizzle atoms need 1024-byte alignment
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bar0 = base + (uint32_t)(DIAG_TMA_STAGES * DT_STAGE_BYTES);
  volatile int32_t* abort_flag =
      reinterpret_cast<volatile int32_t*>(base_ptr + DIAG_TMA_STAGES * DT_STAGE_BYTES + 2 * DIAG_TMA_STAGES * 8);
  auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(DIAG_TMA_STAGES + s); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const EpiParams& e = p.epi;
  const bool c_f32 = e.c_dtype == GEMM_F32;
  const uint32_t c_bytes = e.read_c ? (c_f32 ? (uint32_t)DT_C_BYTES : (uint32_t)DT_C_BYTES / 2) : 0u;
  const bool has_bias = e.bias_mode != GEMM_BIAS_NONE;
  const uint32_t bias_bytes = has_bias ? 64u * (uint32_t)dtype_bytes(e.bias_dtype) : 0u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < DIAG_TMA_STAGES; ++s) {
      mbar_init(full_bar(s), 1);               // the producer's expect_tx arrival + the copies' bytes
      mbar_init(empty_bar(s), DT_CONS_WARPS);  // one arrival per consumer warp
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};

  if (warp == DT_CONS_WARPS) {
    // ------------------------------- producer -------------------------------
    if (lane == 0) {
      tma_prefetch_desc(&p.tmX);
      if (e.read_c) tma_prefetch_desc(&p.tmC);
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_parity = 0;
      for (int64_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
        const int32_t i0 = (int32_t)((t / p.tiles_n) * DIAG_TM);
        const int32_t j0 = (int32_t)((t % p.tiles_n) * DIAG_TN);
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, wc)) break;
        const uint32_t fb = full_bar(stage);
        const uint32_t sx = base + (uint32_t)(stage * DT_STAGE_BYTES);
        mbar_expect_tx(fb, (uint32_t)DT_X_BYTES + c_bytes + 128u + bias_bytes);
        tma_load_1d(sx + DT_V_OFF, &p.tmDiag, p.left ? i0 : j0, fb);
        if (has_bias) tma_load_1d(sx + DT_BIAS_OFF, &p.tmBias, e.bias_mode == GEMM_BIAS_ROW ? i0 : j0, fb);
        if (X_ROW_MAJOR) tma_load_2d(sx, &p.tmX, j0, i0, fb);   // rows of x: (columns, rows)
        else tma_load_2d(sx, &p.tmX, i0, j0, fb);               // columns of x: (rows, columns)
        if (e.read_c) {
          tma_load_2d(sx + DT_X_BYTES, &p.tmC, j0, i0, fb);
          if (c_f32) tma_load_2d(sx + DT_X_BYTES + DT_C_BYTES / 2, &p.tmC, j0 + 32, i0, fb);
        }
        issued |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == DIAG_TMA_STAGES) { stage = 0; phase ^= 1u; }
      }
      // Every copy this thread started lands before the CTA may exit.
      for (int s = 0; s < DIAG_TMA_STAGES; ++s)
        if (issued & (1u << s)) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(full_bar(s), (last_parity >> s) & 1u))
            if (globaltimer_ns() - t0 > 1000000000ull) break;
        }
    }
  } else {
    // ------------------------------- consumers ------------------------------
    const bool bf16 = p.ab_dtype == GEMM_BF16;
    const EpiPtrs ptr = epi_ptrs(e, 0);
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      const int64_t i0 = (t / p.tiles_n) * DIAG_TM;
      const int64_t j0 = (t % p.tiles_n) * DIAG_TN;
      if (!warp_all_wait(full_bar(stage), phase, wc)) break;
      const uint8_t* sx = base_ptr + stage * DT_STAGE_BYTES;
      const uint8_t* sc = sx + DT_X_BYTES;
      const uint16_t* sv = reinterpret_cast<const uint16_t*>(sx + DT_V_OFF);
      const uint8_t* sbias = sx + DT_BIAS_OFF;
      {
        // Task: rows 32h .. 32h + 31 of the tile (one per lane), columns 8g .. 8g + 7.
        const int task = warp;
        const int h = task / 8, g = task % 8;
        const int r = 32 * h + lane;
        const int64_t i = i0 + r, j = j0 + 8 * g;
        float x[8];
        if constexpr (X_ROW_MAJOR) {
          const uint4 w = *reinterpret_cast<const uint4*>(sx + sw128((uint32_t)r, (uint32_t)g));
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            x[2 * u] = h16_to_float((uint16_t)(ww[u] & 0xffffu), bf16);
            x[2 * u + 1] = h16_to_float((uint16_t)(ww[u] >> 16), bf16);
          }
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u)
            x[u] = h16_to_float(*reinterpret_cast<const uint16_t*>(
                                    sx + sw128((uint32_t)(8 * g + u), (uint32_t)(r >> 3)) + (uint32_t)(r & 7) * 2u),
                                bf16);
        }
        float c[8];
        if (e.read_c) {
          if (c_f32) {
            const uint8_t* box = sc + (g >> 2) * (DT_C_BYTES / 2);
            const uint4 a = *reinterpret_cast<const uint4*>(box + sw128((uint32_t)r, (uint32_t)(2 * (g & 3))));
            const uint4 b = *reinterpret_cast<const uint4*>(box + sw128((uint32_t)r, (uint32_t)(2 * (g & 3) + 1)));
            c[0] = __uint_as_float(a.x); c[1] = __uint_as_float(a.y); c[2] = __uint_as_float(a.z);
            c[3] = __uint_as_float(a.w); c[4] = __uint_as_float(b.x); c[5] = __uint_as_float(b.y);
            c[6] = __uint_as_float(b.z); c[7] = __uint_as_float(b.w);
          } else {
            const uint4 w = *reinterpret_cast<const uint4*>(sc + sw128((uint32_t)r, (uint32_t)g));
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
            const bool cb = e.c_dtype == GEMM_BF16;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              c[2 * u] = h16_to_float((uint16_t)(ww[u] & 0xffffu), cb);
              c[2 * u + 1] = h16_to_float((uint16_t)(ww[u] >> 16), cb);
            }
          }
          if (e.c_relu) {
#pragma unroll
            for (int u = 0; u < 8; ++u) c[u] = fmaxf(c[u], 0.0f);
          }
        }
        if (i < p.M && j < p.N) {
          const int n_out = clamp8(p.N - j);
          float v[8];
          const float drow = p.left ? h16_to_float(sv[r], bf16) : 0.0f;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float d = p.left ? drow : h16_to_float(sv[8 * g + u], bf16);
            v[u] = e.alpha * (d * x[u]);
            if (e.read_c) v[u] = fmaf(e.beta, c[u], v[u]);
          }
          if (e.bias_mode == GEMM_BIAS_COL) {
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] += load_as_float(sbias, e.bias_dtype, 8 * g + u);
          } else if (e.bias_mode == GEMM_BIAS_ROW) {
            const float b = load_as_float(sbias, e.bias_dtype, r);
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] += b;
          }
          if (e.relu) {
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = fmaxf(v[u], 0.0f);
          }
          store8_d(ptr.D, e.d_dtype, i * e.ldd + j, e.vec_d != 0, n_out, v);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(stage));
      if (++stage == DIAG_TMA_STAGES) { stage = 0; phase ^= 1u; }
    }
  }
  __syncthreads();
}

cudaError_t launch_tma(const DiagParams& p, int x_row_major, int sm_count, int* grid_out, cudaStream_t stream) {
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return ce;
  if (dev < 64 && !configured[dev]) {
    ce = cudaFuncSetAttribute(diag_tma_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DT_SMEM);
    if (ce == cudaSuccess)
      ce = cudaFuncSetAttribute(diag_tma_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DT_SMEM);
    if (ce != cudaSuccess) return ce;
    configured[dev] = true;
  }
  const int grid = (int)std::min<int64_t>(p.num_tiles, std::max(1, sm_count));
  if (x_row_major) diag_tma_kernel<true><<<grid, DT_THREADS, DT_SMEM, stream>>>(p);
  else diag_tma_kernel<false><<<grid, DT_THREADS, DT_SMEM, stream>>>(p);
  *grid_out = grid;
  return cudaGetLastError();
}

template <typename XT, bool RM>
cudaError_t launch_one(const DiagParams& p, int sm_count, int* grid_out, cudaStream_t stream) {
  // Resident CTAs per SM of this instantiation (looked up once per process).
  static std::atomic<int> resident{0};
  int per_sm = resident.load(std::memory_order_relaxed);
  if (per_sm == 0) {
    cudaError_t ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, diag_gemm_kernel<XT, RM>, DG_THREADS, 0);
    if (ce != cudaSuccess) return ce;
    resident.store(per_sm, std::memory_order_relaxed);
  }
  const int64_t cap = (int64_t)std::max(1, sm_count) * std::max(1, per_sm);
  const int grid = (int)std::min<int64_t>(p.num_tiles, cap);
  diag_gemm_kernel<XT, RM><<<grid, DG_THREADS, 0, stream>>>(p);
  *grid_out = grid;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_diag(const DiagParams& p, int x_row_major, int sm_count, int* grid_out, cudaStream_t stream) {
  if (p.num_tiles <= 0) return cudaErrorInvalidValue;
  if (p.use_tma) {
    if (p.ab_dtype != GEMM_F16 && p.ab_dtype != GEMM_BF16) return cudaErrorInvalidValue;
    return launch_tma(p, x_row_major, sm_count, grid_out, stream);
  }
  switch (p.ab_dtype) {
    case GEMM_F16:
      return x_row_major ? launch_one<__half, true>(p, sm_count, grid_out, stream)
                         : launch_one<__half, false>(p, sm_count, grid_out, stream);
    case GEMM_BF16:
      return x_row_major ? launch_one<__nv_bfloat16, true>(p, sm_count, grid_out, stream)
                         : launch_one<__nv_bfloat16, false>(p, sm_count, grid_out, stream);
    case GEMM_F32:
      return x_row_major ? launch_one<float, true>(p, sm_count, grid_out, stream)
                         : launch_one<float, false>(p, sm_count, grid_out, stream);
    case GEMM_S8:
      return x_row_major ? launch_one<int8_t, true>(p, sm_count, grid_out, stream)
                         : launch_one<int8_t, false>(p, sm_count, grid_out, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gemmlib

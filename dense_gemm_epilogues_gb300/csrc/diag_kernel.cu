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
// Work decomposition: 64 x 64 tiles of D, CTAs persistent over the tiles; each
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

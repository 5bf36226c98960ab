// pair_kernel.cu -- operand staging of the complex / dual-number GEMM (sm_103a).
//
// "Flexible Performant GEMM Kernels on GPUs", section 5.4: numbers x + y u with
// u = i (i*i = -1, complex) or u = eps (eps*eps = 0, dual), stored interleaved
// (real part, then u part) in global memory.  One product is
//     (a + b u)(c + d u) = (a c + b d u^2) + (a d + b c) u.
// The library maps the pair GEMM onto ONE real GEMM of size M x 2N x 2K that the
// tensor-core kernels run unchanged:
//   - A as an M x 2K real matrix: real column 2k holds Re a(i,k), column 2k+1
//     holds its u part.  A row-major interleaved A already IS that matrix
//     (leading dimension 2*lda); a column-major one is split here into two
//     real columns per pair column.
//   - B as a 2K x 2N real matrix Bx whose column 2j yields the real part and
//     column 2j+1 the u part of each output:
//         Bx[2k, 2j] = c,  Bx[2k+1, 2j] = u^2 d  (-d complex, 0 dual),
//         Bx[2k, 2j+1] = d, Bx[2k+1, 2j+1] = c,   with b(k,j) = c + d u,
//     so sum_kk Ax[i,kk] Bx[kk,2j] = sum_k a c + u^2 b d and
//        sum_kk Ax[i,kk] Bx[kk,2j+1] = sum_k a d + b c.
//     It is built here, in B's own layout (K-major for N, N-major for T).
//   - C, D and the bias are interleaved, i.e. already M x 2N real row-major
//     matrices (leading dimension 2*ld) and a 2N real vector.
// The complex case wastes no multiply (4 real products per complex one); the
// dual case multiplies by the zeros of u^2 d (4 real products where 3 suffice).
//
// The copies below only move bits (negation flips the sign bit), so staging is
// exact for every element type.
#include "kernels.h"

namespace gemmlib {
namespace {

constexpr int PS_THREADS = 256;
constexpr int PS_V = 4;   // pairs per thread step (16 bytes of fp16 pairs)

template <typename U> struct Sign;
template <> struct Sign<uint16_t> { static constexpr uint16_t BIT = 0x8000u; };
template <> struct Sign<uint32_t> { static constexpr uint32_t BIT = 0x80000000u; };

// n (<= 8) consecutive elements; `vec`: all 8 present and the address 16-byte aligned.
template <typename U>
__device__ __forceinline__ void load8u(const U* p, bool vec, int n, U (&v)[8]) {
  if (vec) {
    if constexpr (sizeof(U) == 2) {
      const uint4 r = *reinterpret_cast<const uint4*>(p);
      memcpy(v, &r, 16);
    } else {
      const uint4 r0 = reinterpret_cast<const uint4*>(p)[0], r1 = reinterpret_cast<const uint4*>(p)[1];
      memcpy(v, &r0, 16);
      memcpy(v + 4, &r1, 16);
    }
  } else {
#pragma unroll
    for (int t = 0; t < 8; ++t) v[t] = t < n ? p[t] : (U)0;
  }
}

template <typename U>
__device__ __forceinline__ void store8u(U* p, bool vec, int n, const U (&v)[8]) {
  if (vec) {
    if constexpr (sizeof(U) == 2) {
      uint4 r;
      memcpy(&r, v, 16);
      *reinterpret_cast<uint4*>(p) = r;
    } else {
      uint4 r0, r1;
      memcpy(&r0, v, 16);
      memcpy(&r1, v + 4, 16);
      reinterpret_cast<uint4*>(p)[0] = r0;
      reinterpret_cast<uint4*>(p)[1] = r1;
    }
  } else {
#pragma unroll
    for (int t = 0; t < 8; ++t)
      if (t < n) p[t] = v[t];
  }
}

// Bx from B (see the file header).  B's storage: pair (k, j) at pair offset
// k + j*ldb (column-major) or k*ldb + j (row-major).  Bx keeps B's layout with
// leading dimension ldo (a multiple of 8): column-major 2K x 2N, or row-major
// 2K x 2N.  Each thread step moves PS_V consecutive pairs of one column (row).
template <typename U, bool ROW_MAJOR>
__global__ void __launch_bounds__(PS_THREADS)
pair_stage_b_kernel(const U* __restrict__ B, int64_t ldb, int64_t K, int64_t N, int dual, int vec_in,
                    U* __restrict__ out, int64_t ldo) {
  const int64_t n_outer = ROW_MAJOR ? K : N, n_inner = ROW_MAJOR ? N : K;
  const int64_t step = (int64_t)gridDim.x * PS_THREADS * PS_V;
  for (int64_t o = blockIdx.y; o < n_outer; o += gridDim.y) {
    for (int64_t in = ((int64_t)blockIdx.x * PS_THREADS + threadIdx.x) * PS_V; in < n_inner; in += step) {
      const int n = n_inner - in < PS_V ? (int)(n_inner - in) : PS_V;
      const bool full = n == PS_V;
      U x[8];   // PS_V pairs: c0 d0 c1 d1 ...
      load8u(B + 2 * (o * ldb + in), full && vec_in != 0, 2 * n, x);
      U r0[8], r1[8];
#pragma unroll
      for (int t = 0; t < PS_V; ++t) {
        const U c = x[2 * t], d = x[2 * t + 1];
        const U ud = dual ? (U)0 : (U)(d ^ Sign<U>::BIT);   // u^2 * d
        if constexpr (ROW_MAJOR) {   // rows 2k and 2k+1 of Bx, columns 2j and 2j+1
          r0[2 * t] = c;  r0[2 * t + 1] = d;
          r1[2 * t] = ud; r1[2 * t + 1] = c;
        } else {                     // columns 2j and 2j+1 of Bx, rows 2k and 2k+1
          r0[2 * t] = c;  r0[2 * t + 1] = ud;
          r1[2 * t] = d;  r1[2 * t + 1] = c;
        }
      }
      store8u(out + (2 * o) * ldo + 2 * in, full, 2 * n, r0);
      store8u(out + (2 * o + 1) * ldo + 2 * in, full, 2 * n, r1);
    }
  }
}

// Ax from A: row-major A is copied to a row-major M x 2K matrix (leading
// dimension lds, a multiple of 8); column-major A is split into a column-major
// M x 2K matrix (real parts in column 2k, u parts in column 2k+1, leading
// dimension lds).  Each thread step moves PS_V (row-major) or 2*PS_V
// (column-major) consecutive pairs.
template <typename U, bool ROW_MAJOR>
__global__ void __launch_bounds__(PS_THREADS)
pair_stage_a_kernel(const U* __restrict__ A, int64_t lda, int64_t M, int64_t K, int vec_in,
                    U* __restrict__ out, int64_t lds) {
  constexpr int V = ROW_MAJOR ? PS_V : 2 * PS_V;
  const int64_t n_outer = ROW_MAJOR ? M : K, n_inner = ROW_MAJOR ? K : M;
  const int64_t step = (int64_t)gridDim.x * PS_THREADS * V;
  for (int64_t o = blockIdx.y; o < n_outer; o += gridDim.y) {
    for (int64_t in = ((int64_t)blockIdx.x * PS_THREADS + threadIdx.x) * V; in < n_inner; in += step) {
      const int n = n_inner - in < V ? (int)(n_inner - in) : V;
      const bool full = n == V;
      const U* src = A + 2 * (o * lda + in);
      if constexpr (ROW_MAJOR) {   // o = i, in = k: a plain copy of PS_V pairs
        U x[8];
        load8u(src, full && vec_in != 0, 2 * n, x);
        store8u(out + o * lds + 2 * in, full, 2 * n, x);
      } else {                     // o = k, in = i: 8 pairs -> 8 real parts and 8 u parts
        U x0[8], x1[8];
        load8u(src, full && vec_in != 0, min(2 * n, 8), x0);
        load8u(src + 8, full && vec_in != 0, max(2 * n - 8, 0), x1);
        U re[8], im[8];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          re[t] = x0[2 * t];     im[t] = x0[2 * t + 1];
          re[4 + t] = x1[2 * t]; im[4 + t] = x1[2 * t + 1];
        }
        store8u(out + in + (2 * o) * lds, full, n, re);
        store8u(out + in + (2 * o + 1) * lds, full, n, im);
      }
    }
  }
}

dim3 stage_grid(int64_t n_outer, int64_t n_inner, int per_thread) {
  const int64_t chunk = (int64_t)PS_THREADS * per_thread;
  const int64_t gx = std::min<int64_t>((n_inner + chunk - 1) / chunk, 64);
  const int64_t gy = std::min<int64_t>(n_outer, std::max<int64_t>(1, 4096 / gx));
  return dim3((unsigned)std::max<int64_t>(gx, 1), (unsigned)std::min<int64_t>(gy, 65535));
}

}  // namespace

cudaError_t launch_pair_stage_b(const void* B, int64_t ldb, int b_row_major, int64_t K, int64_t N, int elem_bytes,
                                int dual, void* out, int64_t ldo, cudaStream_t stream) {
  if (K <= 0 || N <= 0) return cudaSuccess;
  // 16-byte vectors when every column (row) of B starts 16-byte aligned.
  const int aligned = (reinterpret_cast<uintptr_t>(B) % 16) == 0 && (ldb * 2 * elem_bytes) % 16 == 0;
  const dim3 grid = b_row_major ? stage_grid(K, N, PS_V) : stage_grid(N, K, PS_V);
  if (elem_bytes == 2) {
    const uint16_t* b = static_cast<const uint16_t*>(B);
    uint16_t* o = static_cast<uint16_t*>(out);
    if (b_row_major) pair_stage_b_kernel<uint16_t, true><<<grid, PS_THREADS, 0, stream>>>(b, ldb, K, N, dual, aligned, o, ldo);
    else pair_stage_b_kernel<uint16_t, false><<<grid, PS_THREADS, 0, stream>>>(b, ldb, K, N, dual, aligned, o, ldo);
  } else if (elem_bytes == 4) {
    const uint32_t* b = static_cast<const uint32_t*>(B);
    uint32_t* o = static_cast<uint32_t*>(out);
    if (b_row_major) pair_stage_b_kernel<uint32_t, true><<<grid, PS_THREADS, 0, stream>>>(b, ldb, K, N, dual, aligned, o, ldo);
    else pair_stage_b_kernel<uint32_t, false><<<grid, PS_THREADS, 0, stream>>>(b, ldb, K, N, dual, aligned, o, ldo);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_pair_stage_a(const void* A, int64_t lda, int a_row_major, int64_t M, int64_t K, int elem_bytes,
                                void* out, int64_t lds, cudaStream_t stream) {
  if (M <= 0 || K <= 0) return cudaSuccess;
  const int aligned = (reinterpret_cast<uintptr_t>(A) % 16) == 0 && (lda * 2 * elem_bytes) % 16 == 0;
  const dim3 grid = a_row_major ? stage_grid(M, K, PS_V) : stage_grid(K, M, 2 * PS_V);
  if (elem_bytes == 2) {
    const uint16_t* a = static_cast<const uint16_t*>(A);
    uint16_t* o = static_cast<uint16_t*>(out);
    if (a_row_major) pair_stage_a_kernel<uint16_t, true><<<grid, PS_THREADS, 0, stream>>>(a, lda, M, K, aligned, o, lds);
    else pair_stage_a_kernel<uint16_t, false><<<grid, PS_THREADS, 0, stream>>>(a, lda, M, K, aligned, o, lds);
  } else if (elem_bytes == 4) {
    const uint32_t* a = static_cast<const uint32_t*>(A);
    uint32_t* o = static_cast<uint32_t*>(out);
    if (a_row_major) pair_stage_a_kernel<uint32_t, true><<<grid, PS_THREADS, 0, stream>>>(a, lda, M, K, aligned, o, lds);
    else pair_stage_a_kernel<uint32_t, false><<<grid, PS_THREADS, 0, stream>>>(a, lda, M, K, aligned, o, lds);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace gemmlib

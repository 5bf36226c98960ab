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

template <typename U> struct PairWord;
template <> struct PairWord<uint16_t> { using T = uint32_t; static constexpr uint16_t SIGN = 0x8000u; };
template <> struct PairWord<uint32_t> { using T = uint2; static constexpr uint32_t SIGN = 0x80000000u; };

template <typename U>
__device__ __forceinline__ void load_pair(const U* p, int64_t e, bool aligned, U& re, U& im) {
  if (aligned) {
    const typename PairWord<U>::T w = reinterpret_cast<const typename PairWord<U>::T*>(p)[e];
    U v[2];
    memcpy(v, &w, sizeof(v));
    re = v[0];
    im = v[1];
  } else {
    re = p[2 * e];
    im = p[2 * e + 1];
  }
}

// Two adjacent elements at an even element offset of a 256-byte aligned buffer.
template <typename U>
__device__ __forceinline__ void store_pair(U* p, int64_t off, U x, U y) {
  const U v[2] = {x, y};
  typename PairWord<U>::T w;
  memcpy(&w, v, sizeof(v));
  *reinterpret_cast<typename PairWord<U>::T*>(p + off) = w;
}

// Bx from B (see the file header).  B's storage: pair (k, j) at pair offset
// k + j*ldb (column-major) or k*ldb + j (row-major).  Bx keeps B's layout with
// leading dimension ldo (even): column-major 2K x 2N, or row-major 2K x 2N.
template <typename U, bool ROW_MAJOR>
__global__ void __launch_bounds__(PS_THREADS)
pair_stage_b_kernel(const U* __restrict__ B, int64_t ldb, int64_t K, int64_t N, int dual, int aligned,
                    U* __restrict__ out, int64_t ldo) {
  const int64_t n_outer = ROW_MAJOR ? K : N, n_inner = ROW_MAJOR ? N : K;
  const int64_t step = (int64_t)gridDim.x * PS_THREADS;
  for (int64_t o = blockIdx.y; o < n_outer; o += gridDim.y) {
    for (int64_t in = (int64_t)blockIdx.x * PS_THREADS + threadIdx.x; in < n_inner; in += step) {
      U c, d;
      load_pair(B, o * ldb + in, aligned != 0, c, d);
      const U ud = dual ? (U)0 : (U)(d ^ PairWord<U>::SIGN);   // u^2 * d
      if constexpr (ROW_MAJOR) {   // o = k, in = j: rows 2k and 2k+1, columns 2j and 2j+1
        store_pair(out, (2 * o) * ldo + 2 * in, c, d);
        store_pair(out, (2 * o + 1) * ldo + 2 * in, ud, c);
      } else {                     // o = j, in = k: columns 2j and 2j+1, rows 2k and 2k+1
        store_pair(out, (2 * o) * ldo + 2 * in, c, ud);
        store_pair(out, (2 * o + 1) * ldo + 2 * in, d, c);
      }
    }
  }
}

// Ax from A: row-major A is copied to a row-major M x 2K matrix (leading
// dimension lds, even); column-major A is split into a column-major M x 2K
// matrix (real parts in column 2k, u parts in column 2k+1, leading dimension lds).
template <typename U, bool ROW_MAJOR>
__global__ void __launch_bounds__(PS_THREADS)
pair_stage_a_kernel(const U* __restrict__ A, int64_t lda, int64_t M, int64_t K, int aligned,
                    U* __restrict__ out, int64_t lds) {
  const int64_t n_outer = ROW_MAJOR ? M : K, n_inner = ROW_MAJOR ? K : M;
  const int64_t step = (int64_t)gridDim.x * PS_THREADS;
  for (int64_t o = blockIdx.y; o < n_outer; o += gridDim.y) {
    for (int64_t in = (int64_t)blockIdx.x * PS_THREADS + threadIdx.x; in < n_inner; in += step) {
      U re, im;
      load_pair(A, o * lda + in, aligned != 0, re, im);
      if constexpr (ROW_MAJOR) {   // o = i, in = k
        store_pair(out, o * lds + 2 * in, re, im);
      } else {                     // o = k, in = i
        out[in + (2 * o) * lds] = re;
        out[in + (2 * o + 1) * lds] = im;
      }
    }
  }
}

dim3 stage_grid(int64_t n_outer, int64_t n_inner) {
  const int64_t gx = std::min<int64_t>((n_inner + PS_THREADS - 1) / PS_THREADS, 64);
  const int64_t gy = std::min<int64_t>(n_outer, std::max<int64_t>(1, 4096 / gx));
  return dim3((unsigned)std::max<int64_t>(gx, 1), (unsigned)std::min<int64_t>(gy, 65535));
}

}  // namespace

cudaError_t launch_pair_stage_b(const void* B, int64_t ldb, int b_row_major, int64_t K, int64_t N, int elem_bytes,
                                int dual, void* out, int64_t ldo, cudaStream_t stream) {
  if (K <= 0 || N <= 0) return cudaSuccess;
  const int aligned = (reinterpret_cast<uintptr_t>(B) % (2 * elem_bytes)) == 0;
  const dim3 grid = b_row_major ? stage_grid(K, N) : stage_grid(N, K);
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
  const int aligned = (reinterpret_cast<uintptr_t>(A) % (2 * elem_bytes)) == 0;
  const dim3 grid = a_row_major ? stage_grid(M, K) : stage_grid(K, M);
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

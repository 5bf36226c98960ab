// simt_kernels.cu -- CUDA-core kernels of the library (sm_103a):
//   * ffma_sgemm_kernel: fp32 SGEMM, register-blocked paired FFMA, double-
//     buffered shared memory, fused epilogue (see the kernel for its tiling),
//     and ffma_tail_reduce_kernel, which finishes a last wave split over K;
//   * simt_gemm_kernel: the generic path for every type, layout and alignment
//     (and K == 0), used where TMA cannot describe the operands;
//   * xf_stage_kernel: the operand-transform staging pass of 16-bit operands;
//   * s8_to_f16_kernel: the int8 -> fp16 staging copy of the exact int8 path.
#include "kernels.h"

namespace gemmlib {
namespace {

// ================================ FFMA SGEMM =================================

constexpr int SG_THREADS = 128;
constexpr int SG_PAD = 4;                       // row padding: conflict-free transposed stores
constexpr int SG_LDS = FFMA_BM + SG_PAD;        // 132 floats per K row (BM == BN)

// Loads one BK x 128 slice of op(A) (as A^T: [k][m]) or of op(B) ([k][n]) into
// registers as 2 x SG_NV groups of four values per thread (each thread stands
// for two of the 256 "loader lanes" v = tid and tid + 128).  `KMAJOR`: the
// operand is K-contiguous in global memory (A row-major / B column-major), so a
// lane loads 4 consecutive K values of one row/column per group; otherwise 4
// consecutive M/N values of one K row.
constexpr int SG_NV = FFMA_BK / 8;

template <bool KMAJOR>
struct SliceLoader {
  const float* ptr;
  int64_t ld;
  int64_t extent_mn;   // M (for A) or N (for B)
  int64_t K;
  int xf_on, xf_relu;  // operand transform t(x) = act(scale * x) after the load
  float xf_scale;

  __device__ __forceinline__ void load(int64_t mn0, int64_t k0, int v, float (&out)[SG_NV][4]) const {
#pragma unroll
    for (int g = 0; g < SG_NV; ++g) {
      if constexpr (KMAJOR) {
        const int64_t r = mn0 + (v >> 1);
        const int64_t k = k0 + (v & 1) * 4 + g * 8;
        const float* src = ptr + r * ld + k;
        if (r < extent_mn && k + 4 <= K) {
          const float4 f = *reinterpret_cast<const float4*>(src);
          out[g][0] = f.x; out[g][1] = f.y; out[g][2] = f.z; out[g][3] = f.w;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) out[g][j] = (r < extent_mn && k + j < K) ? src[j] : 0.0f;
        }
      } else {
        const int64_t k = k0 + (v >> 5) + g * 8;
        const int64_t c = mn0 + (v & 31) * 4;
        const float* src = ptr + k * ld + c;
        if (k < K && c + 4 <= extent_mn) {
          const float4 f = *reinterpret_cast<const float4*>(src);
          out[g][0] = f.x; out[g][1] = f.y; out[g][2] = f.z; out[g][3] = f.w;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) out[g][j] = (k < K && c + j < extent_mn) ? src[j] : 0.0f;
        }
      }
      if (xf_on) {   // zero fill stays zero: t(0) = 0
#pragma unroll
        for (int j = 0; j < 4; ++j) out[g][j] = xf_f32(out[g][j], xf_scale, xf_relu);
      }
    }
  }

  // Store the values into the [BK][SG_LDS] shared buffer.
  __device__ __forceinline__ void store(float* s, int v, const float (&in)[SG_NV][4]) const {
#pragma unroll
    for (int g = 0; g < SG_NV; ++g) {
      if constexpr (KMAJOR) {
        const int r = v >> 1, k = (v & 1) * 4 + g * 8;
#pragma unroll
        for (int j = 0; j < 4; ++j) s[(k + j) * SG_LDS + r] = in[g][j];
      } else {
        const int k = (v >> 5) + g * 8, c = (v & 31) * 4;
        *reinterpret_cast<float4*>(&s[k * SG_LDS + c]) = make_float4(in[g][0], in[g][1], in[g][2], in[g][3]);
      }
    }
  }
};

// Paired FP32 FMA (fma.rn.f32x2): two independent fp32 FMAs, each rounded as
// fmaf would, in one instruction -- half the issue slots of scalar FFMA for the
// same FMA-pipe work.  Adjacent columns of a thread's tile share one packed
// B operand; the A value is duplicated into both halves.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ void ffma2(uint64_t& acc, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

// The fused epilogue of four consecutive outputs (row m, columns nb .. nb+3) from
// their fp32 sums x: alpha, beta * c_act(C), bias, ReLU, cast, store.
__device__ __forceinline__ void ffma_finish4(const EpiParams& e, const EpiPtrs& ptr, int64_t m, int64_t nb,
                                             int64_t N, float (&x)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) x[j] *= e.alpha;
  const bool full = nb + 4 <= N;
  if (e.read_c) {
    const int64_t off = m * e.ldc + nb;
    if (full && e.vec_c && e.c_dtype == GEMM_F32) {
      float4 c = *reinterpret_cast<const float4*>(static_cast<const float*>(ptr.C) + off);
      if (e.c_relu) {
        c.x = fmaxf(c.x, 0.0f); c.y = fmaxf(c.y, 0.0f); c.z = fmaxf(c.z, 0.0f); c.w = fmaxf(c.w, 0.0f);
      }
      x[0] = fmaf(e.beta, c.x, x[0]); x[1] = fmaf(e.beta, c.y, x[1]);
      x[2] = fmaf(e.beta, c.z, x[2]); x[3] = fmaf(e.beta, c.w, x[3]);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (nb + j < N) {
          float c = load_as_float(ptr.C, e.c_dtype, off + j);
          if (e.c_relu) c = fmaxf(c, 0.0f);
          x[j] = fmaf(e.beta, c, x[j]);
        }
    }
  }
  if (e.bias_mode == GEMM_BIAS_COL) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (nb + j < N) x[j] += load_as_float(ptr.bias, e.bias_dtype, nb + j);
  } else if (e.bias_mode == GEMM_BIAS_ROW) {
    const float b = load_as_float(ptr.bias, e.bias_dtype, m);
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] += b;
  }
  if (e.relu) {
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = fmaxf(x[j], 0.0f);
  }
  const int64_t doff = m * e.ldd + nb;
  if (full && e.vec_d && e.d_dtype == GEMM_F32) {
    *reinterpret_cast<float4*>(static_cast<float*>(ptr.D) + doff) = make_float4(x[0], x[1], x[2], x[3]);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (nb + j < N) store_float_as(ptr.D, e.d_dtype, doff + j, x[j]);
  }
}

// The CUTLASS page's hierarchy ("Thread Block Tile", "Warp Tile", "Thread
// Tile", "Software Pipelining"): a 128 x 128 block tile over 128 threads, each
// accumulating an 8 x 16 register tile from 8 x 1 and 1 x 16 fragments of A and B
// in shared memory (outer products, 64 paired FMAs per K step), with global
// loads for the next K slice in flight while the current one is multiplied and
// two shared-memory buffers, one __syncthreads() per slice of 16.  Thread (tx,
// ty) owns rows 4ty .. 4ty+3 and 64+4ty .. 64+4ty+3, columns 4tx + 32j .. +3
// (j = 0..3): eight lanes of a quarter warp read 128 contiguous bytes of B, and
// a quarter warp shares one A address (broadcast).  8 x 16 per thread needs 6
// shared loads per 64 paired FMAs where 8 x 8 needed 4 per 32: shared-memory
// throughput bound the 8 x 8 kernel (measured 51.7 against 55.5 TFLOP/s at
// 4096^3 TN, 54.9 against 60.2 at 8192^3).
template <bool A_KMAJOR, bool B_KMAJOR>
__global__ void __launch_bounds__(SG_THREADS, FFMA_CTAS_PER_SM) ffma_sgemm_kernel(const FfmaParams p) {
  __shared__ __align__(16) float As[2][FFMA_BK * SG_LDS];
  __shared__ __align__(16) float Bs[2][FFMA_BK * SG_LDS];

  const int tid = threadIdx.x;
  const int tx = tid & 7, ty = tid >> 3;
  const int64_t tiles_n = (p.N + FFMA_BN - 1) / FFMA_BN;
  // A tail tile is shared by `split` CTAs, each over its own range of K slices.
  int64_t tile = blockIdx.x;
  int part = -1;
  if ((int)blockIdx.x >= p.full_tiles) {
    const int idx = (int)blockIdx.x - p.full_tiles;
    tile = p.full_tiles + idx / p.split;
    part = idx % p.split;
  }
  const int64_t m0 = (tile / tiles_n) * FFMA_BM;
  const int64_t n0 = (tile % tiles_n) * FFMA_BN;
  const int64_t bz = blockIdx.y;                      // problem of the batch

  const SliceLoader<A_KMAJOR> la{p.A + bz * p.stride_a, p.lda, p.M, p.K, p.xf.a_on, p.xf.a_relu, p.xf.a_scale};
  const SliceLoader<B_KMAJOR> lb{p.B + bz * p.stride_b, p.ldb, p.N, p.K, p.xf.b_on, p.xf.b_relu, p.xf.b_scale};

  uint64_t acc2[8][8];   // acc2[i][q]: row i of the thread, columns 2q and 2q+1 of its 16
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int q = 0; q < 8; ++q) acc2[i][q] = 0ull;

  const int nkt_all = (p.K + FFMA_BK - 1) / FFMA_BK;
  const int kt0 = part < 0 ? 0 : min(nkt_all, part * p.kb_per_part);
  const int kt1 = part < 0 ? nkt_all : min(nkt_all, kt0 + p.kb_per_part);
  float ra[2][SG_NV][4], rb[2][SG_NV][4];
  if (kt0 < kt1) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      la.load(m0, (int64_t)kt0 * FFMA_BK, tid + SG_THREADS * h, ra[h]);
      lb.load(n0, (int64_t)kt0 * FFMA_BK, tid + SG_THREADS * h, rb[h]);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      la.store(As[0], tid + SG_THREADS * h, ra[h]);
      lb.store(Bs[0], tid + SG_THREADS * h, rb[h]);
    }
  }
  __syncthreads();

  int buf = 0;
  for (int kt = kt0; kt < kt1; ++kt) {
    const bool more = kt + 1 < kt1;
    if (more) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        la.load(m0, (int64_t)(kt + 1) * FFMA_BK, tid + SG_THREADS * h, ra[h]);
        lb.load(n0, (int64_t)(kt + 1) * FFMA_BK, tid + SG_THREADS * h, rb[h]);
      }
    }
    const float* as = As[buf];
    const float* bs = Bs[buf];
#pragma unroll
    for (int kk = 0; kk < FFMA_BK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&as[kk * SG_LDS + ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&as[kk * SG_LDS + 64 + ty * 4]);
      float4 b[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = *reinterpret_cast<const float4*>(&bs[kk * SG_LDS + tx * 4 + 32 * j]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      uint64_t b2[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        b2[2 * j] = pack2(b[j].x, b[j].y);
        b2[2 * j + 1] = pack2(b[j].z, b[j].w);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint64_t ai = pack2(a[i], a[i]);
#pragma unroll
        for (int q = 0; q < 8; ++q) ffma2(acc2[i][q], ai, b2[q]);
      }
    }
    if (more) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        la.store(As[buf ^ 1], tid + SG_THREADS * h, ra[h]);
        lb.store(Bs[buf ^ 1], tid + SG_THREADS * h, rb[h]);
      }
    }
    __syncthreads();
    buf ^= 1;
  }

  if (part >= 0) {
    // A part of a tail tile: its raw fp32 sums, 128 x 128 row-major per (tile, part).
    float* w = p.ws + ((size_t)(tile - p.full_tiles) * p.split + part) * (FFMA_BM * FFMA_BN);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float x[4];
        unpack2(acc2[i][2 * j], x[0], x[1]);
        unpack2(acc2[i][2 * j + 1], x[2], x[3]);
        __stcg(reinterpret_cast<float4*>(w + r * FFMA_BN + 32 * j + tx * 4), make_float4(x[0], x[1], x[2], x[3]));
      }
    }
    return;
  }
  // Fused epilogue.
  const EpiPtrs ptr = epi_ptrs(p.epi, bz);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
    if (m >= p.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t nb = n0 + 32 * j + tx * 4;
      if (nb >= p.N) continue;
      float x[4];
      unpack2(acc2[i][2 * j], x[0], x[1]);
      unpack2(acc2[i][2 * j + 1], x[2], x[3]);
      ffma_finish4(p.epi, ptr, m, nb, p.N, x);
    }
  }
}

// The tail tiles' parts summed in part order (K order), then the fused epilogue;
// one thread per four consecutive outputs of a tail tile.
__global__ void __launch_bounds__(256) ffma_tail_reduce_kernel(const FfmaParams p) {
  const int64_t tiles_n = (p.N + FFMA_BN - 1) / FFMA_BN;
  const int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // float4 index over the tail tiles
  constexpr int Q_PER_TILE = FFMA_BM * FFMA_BN / 4;
  const int64_t t = q / Q_PER_TILE;
  const int rem = (int)(q - t * Q_PER_TILE);
  const int r = rem / (FFMA_BN / 4), c4 = (rem % (FFMA_BN / 4)) * 4;
  const int64_t tile = p.full_tiles + t;
  const int64_t m = (tile / tiles_n) * FFMA_BM + r;
  const int64_t nb = (tile % tiles_n) * FFMA_BN + c4;
  if (m >= p.M || nb >= p.N) return;
  float x[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int part = 0; part < p.split; ++part) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(
        p.ws + ((size_t)t * p.split + part) * (FFMA_BM * FFMA_BN) + r * FFMA_BN + c4));
    x[0] += v.x; x[1] += v.y; x[2] += v.z; x[3] += v.w;
  }
  ffma_finish4(p.epi, epi_ptrs(p.epi, 0), m, nb, p.N, x);
}

// ============================ generic SIMT kernel ============================

constexpr int GT = 16;   // 16 x 16 outputs per block, one per thread, K slices of 16

__device__ __forceinline__ int64_t a_index(const SimtParams& p, int64_t i, int64_t k) {
  return p.a_row_major ? i * p.lda + k : i + k * p.lda;
}
__device__ __forceinline__ int64_t b_index(const SimtParams& p, int64_t k, int64_t j) {
  return p.b_row_major ? k * p.ldb + j : k + j * p.ldb;
}

// The operand transform of one element of a floating problem: t(x) =
// act(scale * x) in fp32, rounded back to the operand's type for 16-bit operands.
__device__ __forceinline__ float xf_elem(float x, int dt, float scale, int relu) {
  const float v = xf_f32(x, scale, relu);
  if (dt == GEMM_F16) return __half2float(__float2half_rn(v));
  if (dt == GEMM_BF16) return __bfloat162float(__float2bfloat16_rn(v));
  return v;
}

template <bool IS_INT>
__global__ void __launch_bounds__(GT* GT) simt_gemm_kernel(const SimtParams p) {
  using Acc = typename std::conditional<IS_INT, int32_t, float>::type;
  __shared__ Acc As[GT][GT + 1];
  __shared__ Acc Bs[GT][GT + 1];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int64_t bz = blockIdx.y;                      // problem of the batch
  const void* Ab = static_cast<const char*>(p.A) + bz * p.stride_a * dtype_bytes(p.ab_dtype);
  const void* Bb = static_cast<const char*>(p.B) + bz * p.stride_b * dtype_bytes(p.ab_dtype);
  const int64_t tiles_n = (p.N + GT - 1) / GT;
  const int64_t bm = (int64_t)blockIdx.x / tiles_n, bn = (int64_t)blockIdx.x % tiles_n;
  const int64_t i = bm * GT + ty;
  const int64_t j = bn * GT + tx;
  Acc acc = 0;
  for (int64_t k0 = 0; k0 < p.K; k0 += GT) {
    {
      const int64_t ai = bm * GT + ty, ak = k0 + tx;
      Acc v = 0;
      if (ai < p.M && ak < p.K) {
        if constexpr (IS_INT) {
          v = load_as_int(Ab, p.ab_dtype, a_index(p, ai, ak));
          if (p.xf.a_on && p.xf.a_relu && v < 0) v = 0;   // int8: the activation only
        } else {
          v = load_as_float(Ab, p.ab_dtype, a_index(p, ai, ak));
          if (p.xf.a_on) v = xf_elem(v, p.ab_dtype, p.xf.a_scale, p.xf.a_relu);
        }
      }
      As[ty][tx] = v;
      const int64_t bk = k0 + ty, bj = bn * GT + tx;
      Acc w = 0;
      if (bk < p.K && bj < p.N) {
        if constexpr (IS_INT) {
          w = load_as_int(Bb, p.ab_dtype, b_index(p, bk, bj));
          if (p.xf.b_on && p.xf.b_relu && w < 0) w = 0;
        } else {
          w = load_as_float(Bb, p.ab_dtype, b_index(p, bk, bj));
          if (p.xf.b_on) w = xf_elem(w, p.ab_dtype, p.xf.b_scale, p.xf.b_relu);
        }
      }
      Bs[ty][tx] = w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < GT; ++kk) {
      if constexpr (IS_INT) acc += As[ty][kk] * Bs[kk][tx];
      else acc = fmaf(As[ty][kk], Bs[kk][tx], acc);
    }
    __syncthreads();
  }
  if (i >= p.M || j >= p.N) return;
  const EpiParams& e = p.epi;
  const EpiPtrs ptr = epi_ptrs(e, bz);
  if constexpr (IS_INT) {
    int32_t v = wrap_madd(e.alpha_i, acc, 0);
    if (e.read_c) {
      int32_t c = load_as_int(ptr.C, GEMM_S32, i * e.ldc + j);
      if (e.c_relu) c = c > 0 ? c : 0;
      v = wrap_madd(e.beta_i, c, v);
    }
    if (e.bias_mode == GEMM_BIAS_COL) v = wrap_madd(1, load_as_int(ptr.bias, GEMM_S32, j), v);
    else if (e.bias_mode == GEMM_BIAS_ROW) v = wrap_madd(1, load_as_int(ptr.bias, GEMM_S32, i), v);
    if (e.relu) v = v > 0 ? v : 0;
    if (e.d_dtype == GEMM_S8) static_cast<int8_t*>(ptr.D)[i * e.ldd + j] = requant_s8(v, e.out_scale);
    else static_cast<int32_t*>(ptr.D)[i * e.ldd + j] = v;
  } else {
    float v = acc * e.alpha;
    if (e.read_c) {
      float c = load_as_float(ptr.C, e.c_dtype, i * e.ldc + j);
      if (e.c_relu) c = fmaxf(c, 0.0f);
      v = fmaf(e.beta, c, v);
    }
    if (e.bias_mode == GEMM_BIAS_COL) v += load_as_float(ptr.bias, e.bias_dtype, j);
    else if (e.bias_mode == GEMM_BIAS_ROW) v += load_as_float(ptr.bias, e.bias_dtype, i);
    if (e.relu) v = fmaxf(v, 0.0f);
    store_float_as(ptr.D, e.d_dtype, i * e.ldd + j, v);
  }
}

// ============================ int8 -> fp16 staging ===========================

// One thread converts 16 consecutive elements of a row (vector path when the
// row start and leading dimension keep 16-byte alignment), grid-stride.
// RELU: the int8 operand transform (the activation) is applied as it is staged.
template <bool RELU>
__global__ void s8_to_f16_kernel(const int8_t* __restrict__ src, __half* __restrict__ dst, int64_t outer,
                                 int64_t inner, int64_t ld, int vec) {
  auto cv = [](int8_t x) { return __int2half_rn(RELU && x < 0 ? 0 : (int)x); };
  const int64_t groups_per_row = (inner + 15) / 16;
  const int64_t total = outer * groups_per_row;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = g / groups_per_row;
    const int64_t c = (g - r * groups_per_row) * 16;
    const int8_t* s = src + r * ld + c;
    __half* d = dst + r * ld + c;
    if (vec && c + 16 <= inner) {
      const int4 w = *reinterpret_cast<const int4*>(s);
      const int8_t* b = reinterpret_cast<const int8_t*>(&w);
      uint32_t out[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        __half2 v = __halves2half2(cv(b[2 * h]), cv(b[2 * h + 1]));
        out[h] = *reinterpret_cast<uint32_t*>(&v);
      }
      // One 32-byte store (d is 32-byte aligned on this path): each lane writes a
      // whole sector, where two 16-byte stores would half-write every sector per
      // warp request and halve the write bandwidth.
      asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(d), "r"(out[0]), "r"(out[1]),
                   "r"(out[2]), "r"(out[3]), "r"(out[4]), "r"(out[5]), "r"(out[6]), "r"(out[7])
                   : "memory");
    } else {
      for (int j = 0; j < 16 && c + j < inner; ++j) d[j] = cv(s[j]);
    }
  }
}

// ========================== operand transform staging ==========================

// One thread transforms 8 consecutive 16-bit elements of a row (one 16-byte
// vector when the row start and leading dimension keep 16-byte alignment),
// grid-stride; consecutive threads cover consecutive vectors of a row, so every
// warp store writes whole 32-byte sectors.
template <int KIND>
__global__ void xf_stage_kernel(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst, int64_t outer,
                                int64_t inner, int64_t ld, int vec, float scale, uint32_t scale2, int relu) {
  const int64_t groups_per_row = (inner + 7) / 8;
  const int64_t total = outer * groups_per_row;
  const bool mul = scale != 1.0f;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = g / groups_per_row;
    const int64_t c = (g - r * groups_per_row) * 8;
    const uint16_t* s = src + r * ld + c;
    uint16_t* d = dst + r * ld + c;
    if (vec && c + 8 <= inner) {
      uint4 w = __ldcs(reinterpret_cast<const uint4*>(s));
      w.x = xf_word<KIND>(w.x, scale, scale2, mul, relu != 0);
      w.y = xf_word<KIND>(w.y, scale, scale2, mul, relu != 0);
      w.z = xf_word<KIND>(w.z, scale, scale2, mul, relu != 0);
      w.w = xf_word<KIND>(w.w, scale, scale2, mul, relu != 0);
      *reinterpret_cast<uint4*>(d) = w;
    } else {
      // Ragged row end: one element at a time (the other half of the pair is a copy of it).
      for (int j = 0; j < 8 && c + j < inner; ++j) {
        const uint32_t w = (uint32_t)s[j] | ((uint32_t)s[j] << 16);
        d[j] = (uint16_t)(xf_word<KIND>(w, scale, scale2, mul, relu != 0) & 0xffffu);
      }
    }
  }
}

}  // namespace

cudaError_t launch_xf_stage(const void* src, void* dst, int64_t outer, int64_t inner, int64_t ld, const LoadXf& x,
                            int op, cudaStream_t stream) {
  if (outer <= 0 || inner <= 0) return cudaSuccess;
  const int vec = ((reinterpret_cast<uintptr_t>(src) & 15) == 0 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0 &&
                   (ld % 8) == 0) ? 1 : 0;
  const int64_t total = outer * ((inner + 7) / 8);
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  const int kind = op ? x.b_kind : x.a_kind;
  const float scale = op ? x.b_scale : x.a_scale;
  const uint32_t scale2 = op ? x.b_scale2 : x.a_scale2;
  const int relu = op ? x.b_relu : x.a_relu;
  const uint16_t* s = static_cast<const uint16_t*>(src);
  uint16_t* d = static_cast<uint16_t*>(dst);
  if (kind == XF_F16_PACKED)
    xf_stage_kernel<XF_F16_PACKED><<<(unsigned)blocks, 256, 0, stream>>>(s, d, outer, inner, ld, vec, scale, scale2, relu);
  else if (kind == XF_BF16)
    xf_stage_kernel<XF_BF16><<<(unsigned)blocks, 256, 0, stream>>>(s, d, outer, inner, ld, vec, scale, scale2, relu);
  else
    xf_stage_kernel<XF_F16_F32><<<(unsigned)blocks, 256, 0, stream>>>(s, d, outer, inner, ld, vec, scale, scale2, relu);
  return cudaGetLastError();
}

int64_t ffma_tail_split(int64_t tiles, int64_t K, int sm_count, int* split) {
  *split = 0;
  const int64_t slots = (int64_t)std::max(1, sm_count) * FFMA_CTAS_PER_SM;
  const int64_t nkt = (K + FFMA_BK - 1) / FFMA_BK;
  if (tiles <= slots) return 0;
  const int64_t rem = tiles % slots;
  if (rem == 0 || 2 * rem > slots) return 0;
  // Parts of at least 8 K slices each, at most 4 parts.
  const int64_t s = std::min<int64_t>(std::min<int64_t>(slots / rem, 4), nkt / 8);
  if (s < 2) return 0;
  *split = (int)s;
  return rem;
}

cudaError_t launch_ffma(const FfmaParams& p, int a_row_major, int b_row_major, int batch, cudaStream_t stream) {
  const int64_t tiles = ((p.N + FFMA_BN - 1) / FFMA_BN) * ((p.M + FFMA_BM - 1) / FFMA_BM);
  if (tiles > 0x7fffffffLL || batch < 1 || batch > 65535) return cudaErrorInvalidValue;
  const bool tail = p.full_tiles < tiles;
  if (tail && (batch != 1 || p.split < 2 || p.ws == nullptr || p.kb_per_part < 1)) return cudaErrorInvalidValue;
  const int64_t ctas = tail ? p.full_tiles + (tiles - p.full_tiles) * p.split : tiles;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)ctas, (unsigned)batch);
  // A row-major (T) is K-contiguous; B column-major (N) is K-contiguous.
  const bool ak = a_row_major != 0, bk = b_row_major == 0;
  if (ak && bk) ffma_sgemm_kernel<true, true><<<grid, SG_THREADS, 0, stream>>>(p);
  else if (ak) ffma_sgemm_kernel<true, false><<<grid, SG_THREADS, 0, stream>>>(p);
  else if (bk) ffma_sgemm_kernel<false, true><<<grid, SG_THREADS, 0, stream>>>(p);
  else ffma_sgemm_kernel<false, false><<<grid, SG_THREADS, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !tail) return e;
  const int64_t quads = (tiles - p.full_tiles) * (FFMA_BM * FFMA_BN / 4);
  ffma_tail_reduce_kernel<<<(unsigned)((quads + 255) / 256), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_simt(const SimtParams& p, int batch, cudaStream_t stream) {
  const dim3 block(GT, GT);
  const int64_t tiles = ((p.N + GT - 1) / GT) * ((p.M + GT - 1) / GT);
  if (tiles > 0x7fffffffLL || batch < 1 || batch > 65535) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)tiles, (unsigned)batch);
  if (p.ab_dtype == GEMM_S8) simt_gemm_kernel<true><<<grid, block, 0, stream>>>(p);
  else simt_gemm_kernel<false><<<grid, block, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_s8_to_f16(const int8_t* src, __half* dst, int64_t outer, int64_t inner, int64_t ld,
                             cudaStream_t stream, int relu) {
  if (outer <= 0 || inner <= 0) return cudaSuccess;
  const int vec = ((reinterpret_cast<uintptr_t>(src) & 15) == 0 && (reinterpret_cast<uintptr_t>(dst) & 31) == 0 &&
                   (ld % 16) == 0) ? 1 : 0;
  const int64_t total = outer * ((inner + 15) / 16);
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (relu) s8_to_f16_kernel<true><<<(unsigned)blocks, 256, 0, stream>>>(src, dst, outer, inner, ld, vec);
  else s8_to_f16_kernel<false><<<(unsigned)blocks, 256, 0, stream>>>(src, dst, outer, inner, ld, vec);
  return cudaGetLastError();
}

}  // namespace gemmlib

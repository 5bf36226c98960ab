// common.cuh -- types and device helpers shared by the library's kernels.
//
// Everything here is the GPU side of libgemm.so; it shares nothing with the
// CPU oracle.  The PTX wrappers cover the Blackwell (sm_100-family) features the
// tensor-core kernel is built on: mbarrier phase waits (bounded), TMA tiled
// loads (cp.async.bulk.tensor), tcgen05 MMA/commit/ld into and out of tensor
// memory, and the 64-bit shared-memory matrix descriptor.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gemm.h"

namespace gemmlib {

// ---------------------------------------------------------------------------
// Fused epilogue parameters: v = alpha*acc + beta*C[i,j] + bias; v = act(v);
// D[i,j] = cast(v).  (The fused_bias_relu_epilogue functor of the CUTLASS page,
// "Fusing Element-wise Operations: An Example with SGEMM", with the bias
// indexed per column as in section 5.3 of "Flexible Performant GEMM Kernels on
// GPUs"; threshold 0.)
// ---------------------------------------------------------------------------
struct EpiParams {
  float alpha, beta;          // floating paths (fp32 arithmetic)
  int32_t alpha_i, beta_i;    // integer path (int32 arithmetic)
  const void* C;              // row-major, ldc elements per row (unused when beta == 0)
  int64_t ldc;
  int32_t c_dtype;            // gemm_dtype_t
  int32_t d_dtype;
  void* D;                    // row-major, ldd elements per row
  int64_t ldd;
  const void* bias;
  int32_t bias_dtype;
  int32_t bias_mode;          // gemm_bias_mode_t
  int32_t relu;
  int32_t c_relu;             // ReLU applied to each C element as it is read
  float out_scale;            // int8 D: requantisation scale
  int32_t vec_c;              // C rows may be read with 16-byte vectors
  int32_t vec_d;              // D rows may be written with 16-byte vectors
  int32_t read_c;             // beta != 0
  int64_t stride_c;           // batched problems: elements between consecutive C, D and bias
  int64_t stride_d;
  int64_t stride_bias;
};

// ---------------------------------------------------------------------------
// Operand transforms after load ("Flexible Performant GEMM Kernels on GPUs",
// section 4.2, "Transforms", Figure 10): every element x of A (of B) enters the
// product as t(x) = act(scale * x) -- the product rounded to nearest even in
// fp32, then ReLU (threshold 0) if asked, then, for 16-bit operands, rounded to
// nearest even back to the operand's type.  t(0) = 0 for every finite scale,
// so zero fill past the matrix edges stays zero after the transform.
// ---------------------------------------------------------------------------
struct LoadXf {
  int32_t a_on, b_on;         // transform A / B
  int32_t a_relu, b_relu;
  float a_scale, b_scale;
  // Tensor-core kernels, 16-bit operands: how a packed pair is transformed
  // (XF_F16_PACKED, XF_BF16 or XF_F16_F32, below), and for XF_F16_PACKED the
  // scale as an fp16 pair.
  int32_t a_kind, b_kind;
  uint32_t a_scale2, b_scale2;
};

// The C, D and bias of one problem of a (strided) batch.
struct EpiPtrs {
  const void* C;
  void* D;
  const void* bias;
};

__host__ __device__ inline int dtype_bytes(int dt) {
  return dt == GEMM_F32 || dt == GEMM_S32 ? 4 : (dt == GEMM_S8 ? 1 : 2);
}

#if defined(__CUDACC__)

__device__ __forceinline__ EpiPtrs epi_ptrs(const EpiParams& e, int64_t bz) {
  EpiPtrs q;
  q.C = static_cast<const char*>(e.C) + bz * e.stride_c * dtype_bytes(e.c_dtype);
  q.D = static_cast<char*>(e.D) + bz * e.stride_d * dtype_bytes(e.d_dtype);
  q.bias = static_cast<const char*>(e.bias) + bz * e.stride_bias * dtype_bytes(e.bias_dtype);
  return q;
}

// --------------------------- scalar element access -------------------------

__device__ __forceinline__ float load_as_float(const void* p, int dt, int64_t idx) {
  switch (dt) {
    case GEMM_F32: return static_cast<const float*>(p)[idx];
    case GEMM_F16: return __half2float(static_cast<const __half*>(p)[idx]);
    case GEMM_BF16: return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[idx]);
    case GEMM_S8: return (float)static_cast<const int8_t*>(p)[idx];
    default: return (float)static_cast<const int32_t*>(p)[idx];
  }
}

__device__ __forceinline__ int32_t load_as_int(const void* p, int dt, int64_t idx) {
  return dt == GEMM_S8 ? (int32_t) static_cast<const int8_t*>(p)[idx]
                       : static_cast<const int32_t*>(p)[idx];
}

__device__ __forceinline__ void store_float_as(void* p, int dt, int64_t idx, float v) {
  switch (dt) {
    case GEMM_F32: static_cast<float*>(p)[idx] = v; break;
    case GEMM_F16: static_cast<__half*>(p)[idx] = __float2half_rn(v); break;
    default: static_cast<__nv_bfloat16*>(p)[idx] = __float2bfloat16_rn(v); break;
  }
}

// int8 D of the integer path: saturate_int8(round_half_even(fp32(v) * scale)),
// with the conversion and the product each rounded to nearest even in fp32.
__device__ __forceinline__ int8_t requant_s8(int32_t v, float scale) {
  float r = rintf(__fmul_rn(__int2float_rn(v), scale));
  r = fminf(fmaxf(r, -128.0f), 127.0f);
  return (int8_t)__float2int_rn(r);
}

// t(x) = act(scale * x) in fp32 (the transform of one operand element).
__device__ __forceinline__ float xf_f32(float x, float scale, int relu) {
  const float v = __fmul_rn(scale, x);
  return relu ? fmaxf(v, 0.0f) : v;
}

// How the tensor-core kernels transform a 32-bit word of two 16-bit elements
// (a per-operand choice made on the host, LoadXf::a_kind / b_kind):
//   XF_F16_PACKED  fp16 with a scale that fp16 holds exactly: the product of two
//                  fp16 values is exact in fp32, so rounding it once to fp16
//                  (mul.rn.f16x2) is the fp32 product rounded back to fp16;
//   XF_BF16        bf16: widen each half to fp32 (a shift), multiply in fp32,
//                  round both to bf16 with one cvt;
//   XF_F16_F32     fp16 with any other scale: widen, multiply in fp32, round.
// ReLU is applied to the rounded pair (max with +0): rounding to nearest even
// is monotone and keeps the sign, so it commutes with the ReLU.
enum { XF_F16_PACKED = 0, XF_BF16 = 1, XF_F16_F32 = 2 };

template <int KIND>
__device__ __forceinline__ uint32_t xf_word(uint32_t w, float scale, uint32_t scale2, bool mul, bool relu) {
  if (mul) {
    if constexpr (KIND == XF_F16_PACKED) {
      asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(w) : "r"(w), "r"(scale2));
    } else if constexpr (KIND == XF_BF16) {
      const float lo = __fmul_rn(__uint_as_float(w << 16), scale);
      const float hi = __fmul_rn(__uint_as_float(w & 0xffff0000u), scale);
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(hi), "f"(lo));
    } else {
      const __half2 h = *reinterpret_cast<const __half2*>(&w);
      const float2 f = __half22float2(h);
      asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(__fmul_rn(f.y, scale)), "f"(__fmul_rn(f.x, scale)));
    }
  }
  if (relu) {
    if constexpr (KIND == XF_BF16) asm("max.bf16x2 %0, %1, %2;" : "=r"(w) : "r"(w), "r"(0u));
    else asm("max.f16x2 %0, %1, %2;" : "=r"(w) : "r"(w), "r"(0u));
  }
  return w;
}

// Transform, in place, `bytes` (a multiple of 16) of 16-bit operand elements in
// shared memory starting at `saddr`, shared by `nthr` threads (this one is `tid`).
// Elementwise, so the layout of the staged tile (swizzle, K- or MN-major) does
// not matter.  Eight 16-byte vectors per thread are in flight at a time.
template <int KIND>
__device__ __forceinline__ void xf_smem_k(uint32_t saddr, uint32_t bytes, float scale, uint32_t scale2, bool mul,
                                          bool relu, int tid, int nthr) {
  constexpr int U = 8;
  const uint32_t step = (uint32_t)nthr * 16u;
  uint32_t off = (uint32_t)tid * 16u;
  for (; off + (U - 1) * step < bytes; off += U * step) {
    uint32_t w[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u)
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(w[u][0]), "=r"(w[u][1]), "=r"(w[u][2]), "=r"(w[u][3])
                   : "r"(saddr + off + (uint32_t)u * step));
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int q = 0; q < 4; ++q) w[u][q] = xf_word<KIND>(w[u][q], scale, scale2, mul, relu);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(saddr + off + (uint32_t)u * step),
                   "r"(w[u][0]), "r"(w[u][1]), "r"(w[u][2]), "r"(w[u][3])
                   : "memory");
    }
  }
  for (; off < bytes; off += step) {
    uint32_t w[4];
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "r"(saddr + off));
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = xf_word<KIND>(w[q], scale, scale2, mul, relu);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(saddr + off), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                 "r"(w[3])
                 : "memory");
  }
}

// The transform of operand A (op = 0) or B (op = 1) of a staged tile region.
__device__ __forceinline__ void xf_smem(uint32_t saddr, uint32_t bytes, const LoadXf& x, int op, int tid, int nthr) {
  const int kind = op ? x.b_kind : x.a_kind;
  const float scale = op ? x.b_scale : x.a_scale;
  const uint32_t scale2 = op ? x.b_scale2 : x.a_scale2;
  const bool relu = (op ? x.b_relu : x.a_relu) != 0;
  const bool mul = scale != 1.0f;
  if (kind == XF_F16_PACKED) xf_smem_k<XF_F16_PACKED>(saddr, bytes, scale, scale2, mul, relu, tid, nthr);
  else if (kind == XF_BF16) xf_smem_k<XF_BF16>(saddr, bytes, scale, scale2, mul, relu, tid, nthr);
  else xf_smem_k<XF_F16_F32>(saddr, bytes, scale, scale2, mul, relu, tid, nthr);
}

// Make this thread's generic-proxy writes to its CTA's shared memory visible to
// the async proxy (the tensor cores read the transformed tiles through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async;" ::: "memory");
}

// Integer epilogue arithmetic wraps modulo 2^32 (done in unsigned to keep it defined).
__device__ __forceinline__ int32_t wrap_madd(int32_t a, int32_t b, int32_t c) {
  return (int32_t)((uint32_t)a * (uint32_t)b + (uint32_t)c);
}

// ------------------ a row of 32 consecutive outputs (one thread) -------------
// The tensor-core epilogue gives each thread one row of the tile and 32
// consecutive columns per TMEM load; these helpers finish such a chunk.

// Row-contiguous store of a warp's finished 32 x 32 chunk.  Lane r holds row
// m0 + r in x (already in fp32, finished); the rows are converted, written to
// the warp's shared buffer `stage` (16-byte pieces XOR-swizzled by row, so that
// neither side conflicts on banks) and read back so that every store
// instruction writes whole 32-byte sectors of 8 rows x 64 bytes (16-bit D) or
// 4 rows x 128 bytes (fp32 D).  A warp storing 16 bytes to each of 32 rows
// leaves every sector half written per instruction, which halves the write
// bandwidth (measured 3.1 TB/s against 6.0 TB/s for whole sectors).
// Requires the 32 columns inside D and 16-byte aligned rows.
__device__ __forceinline__ void epi_store_chunk32_sectors(const EpiParams& e, void* D, int64_t m0, int64_t M,
                                                         int64_t n_base, const float (&x)[32], uint32_t stage) {
  const int lane = threadIdx.x & 31;
  __syncwarp();   // the previous chunk's reads of the buffer are done
  if (e.d_dtype == GEMM_F32) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stage + (uint32_t)(lane * 128 + ((q ^ (lane & 7)) << 4))),
                   "r"(__float_as_uint(x[4 * q])), "r"(__float_as_uint(x[4 * q + 1])),
                   "r"(__float_as_uint(x[4 * q + 2])), "r"(__float_as_uint(x[4 * q + 3]))
                   : "memory");
    __syncwarp();
    const int pl = lane & 7;
    float* dst = static_cast<float*>(D) + (m0 + (lane >> 3)) * e.ldd + n_base + pl * 4;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = 4 * i + (lane >> 3);
      uint4 v;
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                   : "r"(stage + (uint32_t)(r * 128 + ((pl ^ (r & 7)) << 4))) : "memory");
      if (m0 + r < M) *reinterpret_cast<uint4*>(dst + (int64_t)(4 * i) * e.ldd) = v;
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        if (e.d_dtype == GEMM_F16) {
          __half2 v = __floats2half2_rn(x[8 * q + 2 * h], x[8 * q + 2 * h + 1]);
          w[h] = *reinterpret_cast<uint32_t*>(&v);
        } else {
          __nv_bfloat162 v = __floats2bfloat162_rn(x[8 * q + 2 * h], x[8 * q + 2 * h + 1]);
          w[h] = *reinterpret_cast<uint32_t*>(&v);
        }
      }
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stage + (uint32_t)(lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4))),
                   "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                   : "memory");
    }
    __syncwarp();
    const int pl = lane & 3;
    uint16_t* dst = static_cast<uint16_t*>(D) + (m0 + (lane >> 2)) * e.ldd + n_base + pl * 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = 8 * i + (lane >> 2);
      uint4 v;
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                   : "r"(stage + (uint32_t)(r * 64 + ((pl ^ ((r >> 1) & 3)) << 4))) : "memory");
      if (m0 + r < M) *reinterpret_cast<uint4*>(dst + (int64_t)(8 * i) * e.ldd) = v;
    }
  }
}

// beta * C added into a warp's 32 x 32 chunk (lane r: row m0 + r, x = its 32
// values), with C read through the warp's shared buffer `stage`: each load
// instruction reads whole rows of the chunk (4 rows x 128 bytes of fp32 C, 8 rows
// x 64 bytes of 16-bit C) and the rows are turned around in the buffer (the
// same XOR swizzle as the D stores), where a load of 16 bytes from each of 32
// rows would touch 32 sectors per instruction.  ReLU on C if asked.  Rows at or
// past M are not read.  Requires the 32 columns inside C and 16-byte aligned rows.
__device__ __forceinline__ void epi_add_c_chunk32_turned(const EpiParams& e, const void* C, int64_t m0, int64_t M,
                                                         int64_t n_base, float (&x)[32], uint32_t stage) {
  const int lane = threadIdx.x & 31;
  __syncwarp();   // the previous chunk's use of the buffer is done
  if (e.c_dtype == GEMM_F32) {
    const int pl = lane & 7;
    const float* src = static_cast<const float*>(C) + (m0 + (lane >> 3)) * e.ldc + n_base + pl * 4;
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] = make_uint4(0u, 0u, 0u, 0u);
      if (m0 + 4 * i + (lane >> 3) < M) v[i] = *reinterpret_cast<const uint4*>(src + (int64_t)(4 * i) * e.ldc);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = 4 * i + (lane >> 3);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stage + (uint32_t)(r * 128 + ((pl ^ (r & 7)) << 4))),
                   "r"(v[i].x), "r"(v[i].y), "r"(v[i].z), "r"(v[i].w)
                   : "memory");
    }
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float4 c;
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(c.x), "=f"(c.y), "=f"(c.z), "=f"(c.w)
                   : "r"(stage + (uint32_t)(lane * 128 + ((q ^ (lane & 7)) << 4))) : "memory");
      if (e.c_relu) {
        c.x = fmaxf(c.x, 0.0f); c.y = fmaxf(c.y, 0.0f); c.z = fmaxf(c.z, 0.0f); c.w = fmaxf(c.w, 0.0f);
      }
      x[4 * q + 0] = fmaf(e.beta, c.x, x[4 * q + 0]);
      x[4 * q + 1] = fmaf(e.beta, c.y, x[4 * q + 1]);
      x[4 * q + 2] = fmaf(e.beta, c.z, x[4 * q + 2]);
      x[4 * q + 3] = fmaf(e.beta, c.w, x[4 * q + 3]);
    }
  } else {
    const int pl = lane & 3;
    const uint16_t* src = static_cast<const uint16_t*>(C) + (m0 + (lane >> 2)) * e.ldc + n_base + pl * 8;
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[i] = make_uint4(0u, 0u, 0u, 0u);
      if (m0 + 8 * i + (lane >> 2) < M) v[i] = *reinterpret_cast<const uint4*>(src + (int64_t)(8 * i) * e.ldc);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = 8 * i + (lane >> 2);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stage + (uint32_t)(r * 64 + ((pl ^ ((r >> 1) & 3)) << 4))),
                   "r"(v[i].x), "r"(v[i].y), "r"(v[i].z), "r"(v[i].w)
                   : "memory");
    }
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t w[4];
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                   : "r"(stage + (uint32_t)(lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4))) : "memory");
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float lo, hi;
        if (e.c_dtype == GEMM_F16) {
          __half2 hv = *reinterpret_cast<__half2*>(&w[h]);
          lo = __low2float(hv); hi = __high2float(hv);
        } else {
          __nv_bfloat162 bv = *reinterpret_cast<__nv_bfloat162*>(&w[h]);
          lo = __low2float(bv); hi = __high2float(bv);
        }
        if (e.c_relu) {
          lo = fmaxf(lo, 0.0f);
          hi = fmaxf(hi, 0.0f);
        }
        x[8 * q + 2 * h + 0] = fmaf(e.beta, lo, x[8 * q + 2 * h + 0]);
        x[8 * q + 2 * h + 1] = fmaf(e.beta, hi, x[8 * q + 2 * h + 1]);
      }
    }
  }
}

// x[j] holds alpha*acc for columns n_base..n_base+31 of row m.  Called by all
// 32 lanes of a warp together (the bias is shared by shuffles); lanes whose row
// is outside D (row_ok false) take part but neither read C nor store.
// stage != 0: the warp's 4 KiB shared buffer for row-contiguous stores of D and
// loads of C (each used when the 32 columns are inside the matrix and its rows
// are 16-byte aligned); M is then D's (and C's) row count.
__device__ __forceinline__ void epi_finish_row32_float(const EpiParams& e, const EpiPtrs& ptr, int64_t m,
                                                       bool row_ok, int64_t n_base, int64_t N, float (&x)[32],
                                                       uint32_t stage = 0, int64_t M = 0) {
  const bool full = n_base + 32 <= N;
  if (e.read_c && stage != 0 && full && e.vec_c) {
    // All 32 lanes take part; rows outside C are not read.
    epi_add_c_chunk32_turned(e, ptr.C, m - (threadIdx.x & 31), M, n_base, x, stage);
  } else if (e.read_c && row_ok) {
    const int64_t off = m * e.ldc + n_base;
    if (full && e.vec_c) {
      if (e.c_dtype == GEMM_F32) {
        const float4* c4 = reinterpret_cast<const float4*>(static_cast<const float*>(ptr.C) + off);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4 c = c4[q];
          if (e.c_relu) {
            c.x = fmaxf(c.x, 0.0f); c.y = fmaxf(c.y, 0.0f); c.z = fmaxf(c.z, 0.0f); c.w = fmaxf(c.w, 0.0f);
          }
          x[4 * q + 0] = fmaf(e.beta, c.x, x[4 * q + 0]);
          x[4 * q + 1] = fmaf(e.beta, c.y, x[4 * q + 1]);
          x[4 * q + 2] = fmaf(e.beta, c.z, x[4 * q + 2]);
          x[4 * q + 3] = fmaf(e.beta, c.w, x[4 * q + 3]);
        }
      } else {
        const uint4* c4 = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(ptr.C) + off);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 c = c4[q];
          uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            float lo, hi;
            if (e.c_dtype == GEMM_F16) {
              __half2 v = *reinterpret_cast<__half2*>(&w[h]);
              lo = __low2float(v); hi = __high2float(v);
            } else {
              __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&w[h]);
              lo = __low2float(v); hi = __high2float(v);
            }
            if (e.c_relu) {
              lo = fmaxf(lo, 0.0f);
              hi = fmaxf(hi, 0.0f);
            }
            x[8 * q + 2 * h + 0] = fmaf(e.beta, lo, x[8 * q + 2 * h + 0]);
            x[8 * q + 2 * h + 1] = fmaf(e.beta, hi, x[8 * q + 2 * h + 1]);
          }
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n_base + j < N) {
          float c = load_as_float(ptr.C, e.c_dtype, off + j);
          if (e.c_relu) c = fmaxf(c, 0.0f);
          x[j] = fmaf(e.beta, c, x[j]);
        }
    }
  }
  if (e.bias_mode == GEMM_BIAS_COL) {
    // Every lane needs the same 32 bias values: lane j loads bias[n_base + j]
    // once (coalesced) and the warp shares them by shuffles.
    const int lane = threadIdx.x & 31;
    const float bl = (n_base + lane < N) ? load_as_float(ptr.bias, e.bias_dtype, n_base + lane) : 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] += __shfl_sync(0xffffffffu, bl, j);
  } else if (e.bias_mode == GEMM_BIAS_ROW && row_ok) {
    const float b = load_as_float(ptr.bias, e.bias_dtype, m);
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] += b;
  }
  if (e.relu) {
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = fmaxf(x[j], 0.0f);
  }
  if (stage != 0 && full && e.vec_d) {
    // All 32 lanes take part; rows outside D are not stored.
    epi_store_chunk32_sectors(e, ptr.D, m - (threadIdx.x & 31), M, n_base, x, stage);
    return;
  }
  if (!row_ok) return;
  const int64_t doff = m * e.ldd + n_base;
  if (full && e.vec_d) {
    if (e.d_dtype == GEMM_F32) {
      float4* d4 = reinterpret_cast<float4*>(static_cast<float*>(ptr.D) + doff);
#pragma unroll
      for (int q = 0; q < 8; ++q) d4[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    } else {
      uint4* d4 = reinterpret_cast<uint4*>(static_cast<uint16_t*>(ptr.D) + doff);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          if (e.d_dtype == GEMM_F16) {
            __half2 v = __floats2half2_rn(x[8 * q + 2 * h], x[8 * q + 2 * h + 1]);
            w[h] = *reinterpret_cast<uint32_t*>(&v);
          } else {
            __nv_bfloat162 v = __floats2bfloat162_rn(x[8 * q + 2 * h], x[8 * q + 2 * h + 1]);
            w[h] = *reinterpret_cast<uint32_t*>(&v);
          }
        }
        d4[q] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (n_base + j < N) store_float_as(ptr.D, e.d_dtype, doff + j, x[j]);
  }
}

// 32 bytes of one row from one thread: a single 32-byte store where the address
// allows it (each lane of the warp then writes whole 32-byte sectors; two
// 16-byte stores per lane half-write every sector per request), else two.
__device__ __forceinline__ void st_row_32b(void* p, const uint32_t* w) {
  if ((reinterpret_cast<uintptr_t>(p) & 31) == 0) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
  } else {
    reinterpret_cast<uint4*>(p)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(p)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// epi_store_chunk32_sectors with D's type fixed at compile time.
template <int DT>
__device__ __forceinline__ void epi_store_chunk32_t(void* D, int64_t ldd, int64_t m0, int64_t M, int64_t n_base,
                                                    const float (&x)[32], uint32_t stage) {
  const int lane = threadIdx.x & 31;
  __syncwarp();   // the previous chunk's reads of the buffer are done
  if constexpr (DT == GEMM_F32) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stage + (uint32_t)(lane * 128 + ((q ^ (lane & 7)) << 4))),
                   "r"(__float_as_uint(x[4 * q])), "r"(__float_as_uint(x[4 * q + 1])),
                   "r"(__float_as_uint(x[4 * q + 2])), "r"(__float_as_uint(x[4 * q + 3]))
                   : "memory");
    __syncwarp();
    const int pl = lane & 7;
    float* dst = static_cast<float*>(D) + (m0 + (lane >> 3)) * ldd + n_base + pl * 4;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = 4 * i + (lane >> 3);
      uint4 v;
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                   : "r"(stage + (uint32_t)(r * 128 + ((pl ^ (r & 7)) << 4))) : "memory");
      if (m0 + r < M) *reinterpret_cast<uint4*>(dst + (int64_t)(4 * i) * ldd) = v;
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        if constexpr (DT == GEMM_F16) {
          __half2 v = __floats2half2_rn(x[8 * q + 2 * h], x[8 * q + 2 * h + 1]);
          w[h] = *reinterpret_cast<uint32_t*>(&v);
        } else {
          __nv_bfloat162 v = __floats2bfloat162_rn(x[8 * q + 2 * h], x[8 * q + 2 * h + 1]);
          w[h] = *reinterpret_cast<uint32_t*>(&v);
        }
      }
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stage + (uint32_t)(lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4))),
                   "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                   : "memory");
    }
    __syncwarp();
    const int pl = lane & 3;
    uint16_t* dst = static_cast<uint16_t*>(D) + (m0 + (lane >> 2)) * ldd + n_base + pl * 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = 8 * i + (lane >> 2);
      uint4 v;
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                   : "r"(stage + (uint32_t)(r * 64 + ((pl ^ ((r >> 1) & 3)) << 4))) : "memory");
      if (m0 + r < M) *reinterpret_cast<uint4*>(dst + (int64_t)(8 * i) * ldd) = v;
    }
  }
}

// The plain floating epilogue of one warp -- no beta*C, bias or ReLU, every
// chunk inside D, D taking vector stores -- over chunks [c_begin, c_end) of its
// rows (columns n0 + 32c ... n0 + 32c + 31; m0 = the warp's first row), with
// D's type fixed at compile time, so that no chunk tests the epilogue's
// parameters.  acc(c, x) fills x with alpha times chunk c's accumulator.
template <int DT, typename Acc>
__device__ __forceinline__ void epi_chunks_plain(void* D, int64_t ldd, int64_t m0, int64_t n0, int64_t M,
                                                 uint32_t stage, int c_begin, int c_end, Acc& acc) {
#pragma unroll 1
  for (int c = c_begin; c < c_end; ++c) {
    float x[32];
    acc(c, x);
    epi_store_chunk32_t<DT>(D, ldd, m0, M, n0 + c * 32, x, stage);
  }
}

// D = alpha * acc + beta * C with fp32 C and D and no bias or ReLU (the same
// conditions on the chunks as the plain loop, and C read as whole rows).
template <typename Acc>
__device__ __forceinline__ void epi_chunks_c32(const EpiParams& e, const EpiPtrs& ptr, int64_t m0, int64_t n0,
                                               int64_t M, uint32_t stage, int c_begin, int c_end, Acc& acc) {
#pragma unroll 1
  for (int c = c_begin; c < c_end; ++c) {
    float x[32];
    acc(c, x);
    epi_add_c_chunk32_turned(e, ptr.C, m0, M, n0 + c * 32, x, stage);
    epi_store_chunk32_t<GEMM_F32>(ptr.D, e.ldd, m0, M, n0 + c * 32, x, stage);
  }
}

// D = act(alpha * acc + bias[column]) with an fp32 column bias, no C, ReLU or
// not (the fully connected layer's epilogue), D's type fixed at compile time.
template <int DT, bool RELU, typename Acc>
__device__ __forceinline__ void epi_chunks_bias(const EpiParams& e, const EpiPtrs& ptr, int64_t m0, int64_t n0,
                                                int64_t M, uint32_t stage, int c_begin, int c_end, Acc& acc) {
  const int lane = threadIdx.x & 31;
  const float* bias = static_cast<const float*>(ptr.bias) + n0 + lane;
#pragma unroll 1
  for (int c = c_begin; c < c_end; ++c) {
    const float bl = bias[c * 32];   // lane j holds bias[n0 + 32c + j]; shared by shuffles
    float x[32];
    acc(c, x);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      x[j] += __shfl_sync(0xffffffffu, bl, j);
      if constexpr (RELU) x[j] = fmaxf(x[j], 0.0f);
    }
    epi_store_chunk32_t<DT>(ptr.D, e.ldd, m0, M, n0 + c * 32, x, stage);
  }
}

// The common epilogues of a warp's chunks [c_begin, c_end) (columns n0 + 32c ...,
// m0 = the warp's first row) in loops specialised on D's type:
//   - fp32 C and D, no bias or ReLU;
//   - plain: no C, bias or ReLU;
//   - an fp32 column bias with or without ReLU, no C.
// Each applies only when every chunk lies inside D (and C) and D's (and C's) rows
// take 16-byte vector accesses.  Returns false, having done nothing, for every
// other epilogue, which then takes the general per-chunk path.
template <typename Acc>
__device__ __forceinline__ bool epi_chunks_typed(const EpiParams& e, const EpiPtrs& ptr, int64_t m0, int64_t n0,
                                                 int64_t N, int64_t M, uint32_t stage, int c_begin, int c_end,
                                                 Acc&& acc) {
  if (!e.vec_d || n0 + 32 * (int64_t)c_end > N) return false;
  if (e.read_c) {
    if (e.vec_c && !e.c_relu && e.c_dtype == GEMM_F32 && e.d_dtype == GEMM_F32 && e.bias_mode == GEMM_BIAS_NONE &&
        !e.relu) {
      epi_chunks_c32(e, ptr, m0, n0, M, stage, c_begin, c_end, acc);
      return true;
    }
    return false;
  }
  if (e.bias_mode == GEMM_BIAS_NONE && !e.relu) {
    if (e.d_dtype == GEMM_F32) epi_chunks_plain<GEMM_F32>(ptr.D, e.ldd, m0, n0, M, stage, c_begin, c_end, acc);
    else if (e.d_dtype == GEMM_F16) epi_chunks_plain<GEMM_F16>(ptr.D, e.ldd, m0, n0, M, stage, c_begin, c_end, acc);
    else if (e.d_dtype == GEMM_BF16) epi_chunks_plain<GEMM_BF16>(ptr.D, e.ldd, m0, n0, M, stage, c_begin, c_end, acc);
    else return false;
    return true;
  }
  if (e.bias_mode != GEMM_BIAS_COL || e.bias_dtype != GEMM_F32) return false;
  if (e.d_dtype == GEMM_BF16) {
    if (e.relu) epi_chunks_bias<GEMM_BF16, true>(e, ptr, m0, n0, M, stage, c_begin, c_end, acc);
    else epi_chunks_bias<GEMM_BF16, false>(e, ptr, m0, n0, M, stage, c_begin, c_end, acc);
  } else if (e.d_dtype == GEMM_F16) {
    if (e.relu) epi_chunks_bias<GEMM_F16, true>(e, ptr, m0, n0, M, stage, c_begin, c_end, acc);
    else epi_chunks_bias<GEMM_F16, false>(e, ptr, m0, n0, M, stage, c_begin, c_end, acc);
  } else if (e.d_dtype == GEMM_F32) {
    if (e.relu) epi_chunks_bias<GEMM_F32, true>(e, ptr, m0, n0, M, stage, c_begin, c_end, acc);
    else epi_chunks_bias<GEMM_F32, false>(e, ptr, m0, n0, M, stage, c_begin, c_end, acc);
  } else {
    return false;
  }
  return true;
}

// x[j] holds the exact int32 product sums of columns n_base..n_base+31 of row m;
// it is finished in place (alpha, beta*C, bias, ReLU) and stored.  Called by all
// 32 lanes of a warp together, as the floating version.
__device__ __forceinline__ void epi_finish_row32_int(const EpiParams& e, const EpiPtrs& ptr, int64_t m,
                                                     bool row_ok, int64_t n_base, int64_t N, int32_t* x) {
  const bool full = n_base + 32 <= N;
#pragma unroll
  for (int j = 0; j < 32; ++j) x[j] = wrap_madd(e.alpha_i, x[j], 0);
  if (e.read_c && row_ok) {
    const int64_t off = m * e.ldc + n_base;
    if (full && e.vec_c) {
      const int4* c4 = reinterpret_cast<const int4*>(static_cast<const int32_t*>(ptr.C) + off);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        int4 c = c4[q];
        if (e.c_relu) {
          c.x = c.x > 0 ? c.x : 0; c.y = c.y > 0 ? c.y : 0; c.z = c.z > 0 ? c.z : 0; c.w = c.w > 0 ? c.w : 0;
        }
        x[4 * q + 0] = wrap_madd(e.beta_i, c.x, x[4 * q + 0]);
        x[4 * q + 1] = wrap_madd(e.beta_i, c.y, x[4 * q + 1]);
        x[4 * q + 2] = wrap_madd(e.beta_i, c.z, x[4 * q + 2]);
        x[4 * q + 3] = wrap_madd(e.beta_i, c.w, x[4 * q + 3]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n_base + j < N) {
          int32_t c = load_as_int(ptr.C, GEMM_S32, off + j);
          if (e.c_relu) c = c > 0 ? c : 0;
          x[j] = wrap_madd(e.beta_i, c, x[j]);
        }
    }
  }
  if (e.bias_mode == GEMM_BIAS_COL) {
    const int lane = threadIdx.x & 31;
    const int32_t bl = (n_base + lane < N) ? load_as_int(ptr.bias, GEMM_S32, n_base + lane) : 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = wrap_madd(1, __shfl_sync(0xffffffffu, bl, j), x[j]);
  } else if (e.bias_mode == GEMM_BIAS_ROW && row_ok) {
    const int32_t b = load_as_int(ptr.bias, GEMM_S32, m);
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = wrap_madd(1, b, x[j]);
  }
  if (!row_ok) return;
  if (e.relu) {
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = x[j] > 0 ? x[j] : 0;
  }
  if (e.d_dtype == GEMM_S8) {
    int8_t* d8 = static_cast<int8_t*>(ptr.D) + m * e.ldd + n_base;
    int8_t q[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) q[j] = requant_s8(x[j], e.out_scale);
    if (full && e.vec_d) {
      uint32_t w[8];
      memcpy(w, q, 32);
      st_row_32b(d8, w);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n_base + j < N) d8[j] = q[j];
    }
    return;
  }
  int32_t* d = static_cast<int32_t*>(ptr.D) + m * e.ldd + n_base;
  if (full && e.vec_d) {
#pragma unroll
    for (int q = 0; q < 4; ++q) st_row_32b(d + 8 * q, reinterpret_cast<const uint32_t*>(x + 8 * q));
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (n_base + j < N) d[j] = x[j];
  }
}

// ------------------------------- PTX wrappers -------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with acquire semantics at cluster scope: for barriers that threads of
// the other CTA of a pair arrive on (release.cluster) after writing shared
// memory that this thread's later tensor-core operations read.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Programmatic dependent launch.  launch_dependents lets the next kernel of the
// stream (if it was launched as a programmatic dependent) start its prologue on
// free SMs; wait blocks until every prerequisite grid has completed and its
// memory is visible -- it comes before this kernel's first access to data that
// an earlier kernel may write (operands, C, D, the error word).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Shared state of a CTA's bounded waits.
struct WaitCtx {
  volatile int32_t* abort;   // shared: set once any role of the CTA gave up
  int32_t* err;              // global error word (first failure wins)
  uint64_t timeout_ns;
};

// Wait for the phase of `bar` with the given parity to complete.  Gives up after
// ctx.timeout_ns (recording GEMM_ERR_TIMEOUT) or as soon as another role of the
// CTA has given up.  Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtx& ctx) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;   // try_wait itself suspends for a while
    if (*ctx.abort) return false;
    if (globaltimer_ns() - t0 > ctx.timeout_ns) {
      atomicCAS(ctx.err, 0, (int32_t)GEMM_ERR_TIMEOUT);
      *ctx.abort = 1;
      __threadfence_block();
      return false;
    }
  }
}

// mbar_wait with the cluster-scope acquire of mbar_try_wait_cluster.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, const WaitCtx& ctx) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*ctx.abort) return false;
    if (globaltimer_ns() - t0 > ctx.timeout_ns) {
      atomicCAS(ctx.err, 0, (int32_t)GEMM_ERR_TIMEOUT);
      *ctx.abort = 1;
      __threadfence_block();
      return false;
    }
  }
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int32_t x, int32_t y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 1-D tiled TMA load (a box of a vector; zero fill past its end).
__device__ __forceinline__ void tma_load_1d(uint32_t dst, const CUtensorMap* tm, int32_t x, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.1d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2}], [%3];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(bar)
      : "memory");
}

// 3-D tiled TMA load (x innermost, z = problem of a batch).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D(tmem) (+)= A(smem desc) * B(smem desc), kind::f16 (fp16/bf16 in, fp32 accumulate).
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp gets TMEM lane (base lane + t).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// ------------------------- CTA-pair (cluster of 2) helpers -----------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Full cluster barrier (every thread of both CTAs).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on an mbarrier of another CTA of the cluster (shared::cluster address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// TMA load whose completion may be signalled on the mbarrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* tm, int32_t x, int32_t y,
                                                 uint32_t bar_cluster_addr) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar_cluster_addr)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* tm, int32_t x, int32_t y,
                                                 int32_t z, uint32_t bar_cluster_addr) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar_cluster_addr)
      : "memory");
}

// The same with an L2 cache policy for the loaded lines (from createpolicy).
__device__ __forceinline__ void tma_load_3d_pair_hint(uint32_t dst, const CUtensorMap* tm, int32_t x, int32_t y,
                                                      int32_t z, uint32_t bar_cluster_addr, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar_cluster_addr), "l"(policy)
      : "memory");
}

// D(tmem, both CTAs) (+)= A(smem, both CTAs) * B(smem, N split over both CTAs).
__device__ __forceinline__ void tc_mma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at this offset in every CTA of `cta_mask` (bit r:
// CTA r of the pair) when the pair MMAs issued so far by this thread have
// completed.  This signals barriers only; it moves no operand data.
__device__ __forceinline__ void tc_commit_pair_mask(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Collective over the CTA pair: one warp of each CTA executes these.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// --------------------------- stream-K work division ---------------------------
// Tiles [0, t_dp) run whole: tile t on cluster t mod G.  The K blocks of tiles
// [t_dp, T) form one linear sequence (tile-major) of W = (T - t_dp) * KB blocks;
// cluster c takes the contiguous range [c*W/G, (c+1)*W/G).  A segment is one
// tile's share of a range: K blocks [kb0, kb1).
struct SegmentIter {
  int G, T, t_dp, KB, t_half;
  int t;                 // next whole tile of this cluster
  int u;                 // next half unit of this cluster
  int64_t L, L1;         // remaining linear range of this cluster
  // Tiles t_half ... T-1 (only without a stream-K tail, t_dp == T) run as two
  // units of half their columns each, unit 2(t - t_half) + h being half h of
  // tile t; with 2 (T - t_half) <= G each cluster runs at most one of them.
  __device__ __forceinline__ SegmentIter(int cid, int G_, int T_, int t_dp_, int KB_, int t_half_)
      : G(G_), T(T_), t_dp(t_dp_), KB(KB_), t_half(t_half_), t(cid), u(cid) {
    const int64_t W = (int64_t)(T - t_dp) * KB;
    L = (int64_t)cid * W / G;
    L1 = (int64_t)(cid + 1) * W / G;
  }
  // half: -1 for a whole tile (or a stream-K segment), else the column half.
  __device__ __forceinline__ bool next(int& tile, int& kb0, int& kb1, int& half) {
    half = -1;
    if (t < t_dp && t < t_half) {
      tile = t;
      kb0 = 0;
      kb1 = KB;
      t += G;
      return true;
    }
    if (u < 2 * (T - t_half)) {
      tile = t_half + u / 2;
      half = u & 1;
      kb0 = 0;
      kb1 = KB;
      u += G;
      return true;
    }
    if (L < L1) {
      const int64_t tl = L / KB;
      kb0 = (int)(L - tl * KB);
      const int64_t rest = L1 - L;
      kb1 = (int)(rest < (int64_t)(KB - kb0) ? kb0 + rest : KB);
      tile = t_dp + (int)tl;
      L += kb1 - kb0;
      return true;
    }
    return false;
  }
};

// Cluster whose stream-K range holds linear K-block index L (W blocks over G clusters).
__device__ __forceinline__ int sk_cluster_of(int64_t L, int64_t W, int G) {
  return (int)(((L + 1) * (int64_t)G + W - 1) / W) - 1;
}

__device__ __forceinline__ int32_t ld_acquire_gpu(const int32_t* p) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(int32_t* p, int32_t v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format) for a 128-byte-swizzled
// operand tile whose swizzle atoms (8 rows of 128 bytes) start on 1024-byte
// boundaries:
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-47  descriptor version (1)
//   bits 49-51  base offset (0: atoms are 1024-byte aligned)
//   bits 61-63  swizzle mode (2 = 128-byte swizzle)
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

#endif  // __CUDACC__

}  // namespace gemmlib

// kernels.h -- host-side launch interface of the library's kernels (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "common.cuh"

namespace gemmlib {

// Tensor-core kernel (tcgen05 + TMA), one CTA per SM, persistent over tiles.
struct TcParams {
  CUtensorMap tmA;        // A tiles (see tc_kernel.cu for the box shapes)
  CUtensorMap tmB;        // B tiles
  CUtensorMap tmBh;       // CTA-pair kernel: B boxes of half the columns, for half-tile units
  int32_t M, N, K;
  int32_t num_kb;         // K blocks of 64 elements
  int32_t tiles_m, tiles_n, num_tiles;
  int32_t tiles_per_batch;  // tiles_m * tiles_n; num_tiles = batch * tiles_per_batch
  int32_t a_batched;      // A's tensor map has one slice per problem (else slice 0 for all)
  int32_t b_batched;
  int32_t raster;         // tile rows per raster group
  int32_t a_mn_major;     // A stored M-contiguous (layout N) rather than K-contiguous
  int32_t b_mn_major;     // B stored N-contiguous (layout T) rather than K-contiguous
  uint32_t idesc;         // tcgen05 instruction descriptor
  uint32_t idesc_half;    // CTA-pair kernel: the same for half-tile units (N = 128)
  int32_t half_first_tile;  // CTA-pair kernel: tiles from here on run as two column halves (num_tiles: none)
  int32_t chunk_kb;       // > 0: exact integer mode, K blocks per fp32 chunk
  int32_t k_rotate;       // single-CTA kernel, one tile column: rotate each tile's K start (see tc_kernel.cu)
  LoadXf xf;              // transforms of the staged A / B tiles (launched as a separate kernel instance)
  EpiParams epi;
  int32_t* err;
  uint64_t timeout_ns;
  // Stream-K (floating mode, both tensor-core kernels): tiles below sk_first_tile
  // run whole, one per cluster (CTA) in turn; the K blocks of the remaining tiles
  // are split into equal contiguous ranges, one per cluster (CTA).
  // sk_first_tile == num_tiles turns it off.
  int32_t sk_first_tile;
  int32_t sk_epoch;       // value published in sk_flags by this launch
  // CTA-pair kernel: per cluster and CTA one 128 x 256 fp32 partial accumulator,
  // and the epoch of its last published partial.  Single-CTA kernel: per CTA two
  // 128 x BN fp32 partials (the tile its K range starts in, and the other), and
  // per tile an arrival counter (0 between launches).
  float* sk_partials;
  int32_t* sk_flags;
};

constexpr int TC_BM = 128;
constexpr int TC_BK = 64;   // 16-bit elements: one 128-byte swizzle row

int tc_stages(int bn);
int tc_k_per_stage(int bn);             // K depth of one pipeline stage of the single-CTA kernel
size_t tc_smem_bytes(int bn);
cudaError_t launch_tc(const TcParams& p, int bn, int grid, cudaStream_t stream);

// CTA-pair tensor-core kernel (cta_group::2): 256 x 256 tiles per cluster of two CTAs.
// Tensor-map boxes: A as for 128-row tiles, B as for 128-column tiles.
int tc_pair_stages();
int tc_pair_k_per_stage();              // K depth of one pipeline stage (64-deep slabs per stage x 64)
size_t tc_pair_smem_bytes();
int tc_pair_max_clusters(int device);   // co-resident clusters of two (0 if unknown)
cudaError_t launch_tc_pair(const TcParams& p, int clusters, cudaStream_t stream);

// FFMA SGEMM (fp32, CUDA cores): 128 x 128 tiles, one per CTA of 128 threads.
struct FfmaParams {
  const float* A;
  const float* B;
  int64_t lda, ldb;
  int64_t stride_a, stride_b;   // batched problems (elements); one problem per grid row
  int32_t M, N, K;
  // Split tail wave (single problems): tiles [full_tiles, tiles) run as `split`
  // CTAs each over kb_per_part K slices, writing raw fp32 sums to ws (128 x 128
  // row-major per tile and part); ffma tail reduction then finishes them.
  // full_tiles == tiles (split 1): no tail split.
  int32_t full_tiles;
  int32_t split;
  int32_t kb_per_part;
  float* ws;
  LoadXf xf;                    // transforms of A / B elements as they are loaded
  EpiParams epi;
};
constexpr int FFMA_BM = 128, FFMA_BN = 128, FFMA_BK = 16;
constexpr int FFMA_CTAS_PER_SM = 2;   // 128 threads x <= 256 registers, 33 KiB shared memory each
// Tail split for a single problem of `tiles` tiles and K of `K` on `sm_count` SMs:
// when the last wave of CTAs is at most half full, its tiles are split over K
// into *split parts (0: no split).  Returns the number of tail tiles.
int64_t ffma_tail_split(int64_t tiles, int64_t K, int sm_count, int* split);
cudaError_t launch_ffma(const FfmaParams& p, int a_row_major, int b_row_major, int batch, cudaStream_t stream);

// Generic CUDA-core kernel: any dtype, layout, alignment; K may be 0.
struct SimtParams {
  const void* A;
  const void* B;
  int64_t lda, ldb;
  int32_t ab_dtype;
  int32_t a_row_major, b_row_major;
  int64_t M, N, K;
  int64_t stride_a, stride_b;   // batched problems (elements); one problem per grid row
  LoadXf xf;                    // transforms of A / B elements as they are loaded
  EpiParams epi;
};
cudaError_t launch_simt(const SimtParams& p, int batch, cudaStream_t stream);
inline cudaError_t launch_simt(const SimtParams& p, cudaStream_t stream) { return launch_simt(p, 1, stream); }

// GEMM with one diagonal operand: D = epilogue(alpha * diag(d) * x + beta * C)
// (left) or epilogue(alpha * x * diag(d) + beta * C) (right), x the dense
// operand seen as an M x N matrix.  One product per output, no tensor cores.
struct DiagParams {
  // TMA-staged kernel (use_tma): 64 x 64 boxes of x (128-byte swizzle; 16-bit x)
  // and of C (two 32-column boxes for fp32 C), loaded into a ring of stages.
  CUtensorMap tmX;
  CUtensorMap tmC;
  CUtensorMap tmDiag;     // TMA-staged kernel: 64-entry boxes of the diagonal
  CUtensorMap tmBias;     // TMA-staged kernel: 64-entry boxes of the bias vector (when there is one)
  int32_t use_tma;
  int32_t* err;           // TMA-staged kernel: error word (first expired wait)
  uint64_t timeout_ns;    // TMA-staged kernel: bound of every wait
  const void* X;          // dense operand, ab_dtype, row-major (layout T) or column-major (N)
  const void* diag;       // the diagonal: M entries (left) or N entries (right), ab_dtype
  int64_t ldx;
  int64_t M, N;
  int64_t tiles_n, num_tiles;   // DIAG_TM x DIAG_TN tiles of D
  int32_t ab_dtype;
  int32_t left;           // 1: d[i] scales row i (A = diag(d)); 0: d[j] scales column j (B = diag(d))
  int32_t vec_x;          // x may be read as aligned 8-element vectors along its contiguous dimension
  int32_t vec_diag;       // the diagonal may be read as aligned 8-element vectors
  EpiParams epi;
};
constexpr int DIAG_TM = 64, DIAG_TN = 64;
constexpr int DIAG_TMA_STAGES = 6;   // ring depth of the TMA-staged kernel
// Persistent launch: min(tiles, sm_count x resident CTAs per SM) CTAs; the grid used goes to *grid_out.
cudaError_t launch_diag(const DiagParams& p, int x_row_major, int sm_count, int* grid_out, cudaStream_t stream);

// Complex / dual-number GEMM staging (pair_kernel.cu): B -> the 2K x 2N real
// matrix whose column pairs give the real and unit parts of each product; A ->
// an M x 2K real matrix (row-major copy, or split columns for column-major A).
// elem_bytes: 2 (f16/bf16) or 4 (f32); out is 256-byte aligned, ldo/lds even.
cudaError_t launch_pair_stage_b(const void* B, int64_t ldb, int b_row_major, int64_t K, int64_t N, int elem_bytes,
                                int dual, void* out, int64_t ldo, cudaStream_t stream);
cudaError_t launch_pair_stage_a(const void* A, int64_t lda, int a_row_major, int64_t M, int64_t K, int elem_bytes,
                                void* out, int64_t lds, cudaStream_t stream);

// Transform staging of a 16-bit operand: dst[r*ld + c] = t(src[r*ld + c]) for
// r < outer, c < inner, with the operand transform of op (0: A, 1: B) of x.
cudaError_t launch_xf_stage(const void* src, void* dst, int64_t outer, int64_t inner, int64_t ld, const LoadXf& x,
                            int op, cudaStream_t stream);

// int8 -> fp16 staging copy of a strided matrix: dst[r*ld + c] = src[r*ld + c]
// for r < outer, c < inner; relu != 0 stages max(src, 0) (the operand transform
// of an int8 problem).
cudaError_t launch_s8_to_f16(const int8_t* src, __half* dst, int64_t outer, int64_t inner, int64_t ld,
                             cudaStream_t stream, int relu = 0);

}  // namespace gemmlib

// tc_kernel.cu -- tcgen05 tensor-core GEMM with a fused epilogue (sm_103a).
//
// D = epilogue(alpha * op(A) * op(B) + beta * C) for fp16/bf16 operands with
// fp32 accumulation in tensor memory, and (exact integer mode) for int8
// operands staged as fp16.
//
// The structure follows the recursive blocking of "Flexible Performant GEMM
// Kernels on GPUs" (section 3: global -> shared -> MMA -> epilogue) and the
// software pipelining of the CUTLASS page ("Software Pipelining": loads, shared
// memory and math in flight at once), mapped onto Blackwell hardware:
//   - one persistent CTA per SM walks a list of 128 x BN output tiles;
//   - warp 0 (one thread) streams 128x64 A and BNx64 B tiles with TMA into an
//     S-stage ring of 128-byte-swizzled shared-memory buffers (full/empty
//     mbarriers) -- the swizzle removes the bank conflicts that section 5.1 of
//     the paper names as its main gap;
//   - warp 1 (one thread) issues tcgen05.mma (M=128, N=BN, K=16) into a
//     tensor-memory accumulator and commits stage releases to the empty
//     barriers; it owns the tensor-memory allocation (all 512 columns: two
//     128x256 or four 128x128 fp32 accumulators);
//   - warps 2-5 drain a finished accumulator with tcgen05.ld (one row per
//     thread), apply alpha, beta*C, bias, ReLU and the output cast in registers
//     and store with 16-byte vector writes, while warp 1 already accumulates the
//     next tile into the other accumulator buffer.
// Exact integer mode (int8 inputs): every product of two int8 values is exact
// in fp32 and so is any sum of up to 1024 of them (|sum| <= 2^24), so the MMA
// accumulates K in chunks of chunk_kb*64 <= 1024 into a fresh fp32 accumulator;
// the epilogue warps convert each finished chunk to int32 and add it into
// registers, giving the exact int32 result for any K.
//
// Operand transforms (a separate instance, XF): eight more warps wait for each
// stage's copies, apply t(x) = act(scale * x) in place to the staged A and/or B
// tiles, fence the async proxy and arrive on a stage-transformed barrier, which
// the MMA thread waits for instead of the full barrier.
//
// Every wait is bounded (see mbar_wait): on expiry the CTA records
// GEMM_ERR_TIMEOUT, drains its own copies and MMAs in flight (again bounded)
// and releases tensor memory before it exits.
#include "kernels.h"

namespace gemmlib {
namespace {

// A pipeline stage holds SLABS consecutive 64-deep K blocks: one stage-full wait
// and one tcgen05.commit per SLABS * 4 MMAs (each of those holds the tensor pipe
// for a while; see the CTA-pair kernel).
// 128-wide tiles: two slabs in each of 3 stages.  256-wide tiles: one slab in
// each of 4 stages (two slabs would leave a 2-stage ring, one stage of lookahead:
// measured 14 % slower at 8192^3).
template <int BN>
struct TcCfg {
  static constexpr int SLABS = (BN == 256) ? 1 : 2;
  static constexpr int STAGES = ((BN == 256) ? 4 : (BN == 128) ? 6 : 8) / SLABS;
  static constexpr int A_BYTES = TC_BM * TC_BK * 2;   // 16 KiB per slab
  static constexpr int B_BYTES = BN * TC_BK * 2;      // 32 / 16 / 8 KiB per slab (BN = 256 / 128 / 64)
  static constexpr int STAGE_BYTES = SLABS * (A_BYTES + B_BYTES);   // [A slabs][B slabs]
  static constexpr int ACC_BUFS = 512 / BN;           // accumulators in the 512 TMEM columns
  static constexpr int NUM_BARS = 3 * STAGES + 2 * ACC_BUFS + 1;
  static constexpr int OUT_STAGE_BYTES = 8 * 4096;   // a 32 x 32 output turn-around buffer per epilogue warp
  static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE_BYTES + OUT_STAGE_BYTES + NUM_BARS * 8 + 16;
};

// Producer warp, MMA warp, then the epilogue warps: 8 in floating mode (two per
// tensor-memory lane quarter, each finishing half of the tile's columns), 4 in
// exact integer mode (a thread keeps a whole row of int32 sums); then, with
// operand transforms, 8 transform warps (an in-place pass over a staged tile is
// bound by shared-memory latency and bandwidth: 8 warps took a 16384 x 64 x
// 16384 GEMM with A transformed from 183 to 140 us, against 95 us untransformed).
template <bool INT_MODE, bool XF = false>
struct TcThreads {
  static constexpr int EPI_WARPS = INT_MODE ? 4 : 8;
  static constexpr int XF_WARPS = XF ? 8 : 0;
  static constexpr int THREADS = 64 + 32 * (EPI_WARPS + XF_WARPS);
};
constexpr uint32_t TMEM_COLS = 512;
constexpr int MN_BOX = 64;            // MN extent of one TMA box for MN-major operands
constexpr uint32_t MN_BOX_BYTES = MN_BOX * TC_BK * 2;   // 8 KiB

// Tile t -> (tile row, tile column), in groups of `raster` tile rows so that
// CTAs running at the same time share A row panels and B column panels in L2
// (the block rasterisation of the CUTLASS page's policy).
__device__ __forceinline__ void tile_coords(int t, const TcParams& p, int& bz, int& tm, int& tn) {
  bz = t / p.tiles_per_batch;                     // problem of the batch
  const int tl = t - bz * p.tiles_per_batch;
  const int group_tiles = p.raster * p.tiles_n;
  const int g = tl / group_tiles;
  const int first_m = g * p.raster;
  const int gsize = min(p.tiles_m - first_m, p.raster);
  const int r = tl - g * group_tiles;
  tm = first_m + r % gsize;
  tn = r / gsize;
}

// Bounded wait that ignores the abort flag: used while winding down, so that no
// copy or MMA of this CTA is still in flight when it releases tensor memory and
// exits.  Its bound is at least one second whatever the user's wait bound is.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t user_timeout_ns) {
  const uint64_t timeout_ns = user_timeout_ns > 1000000000ull ? user_timeout_ns : 1000000000ull;
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) return;
  }
}

// All lanes of a warp wait; the warp gives up together if any lane gave up.
// CTA barrier of the four epilogue warps (named barrier 1; barrier 0 is __syncthreads).
template <int THREADS>
__device__ __forceinline__ void epi_warps_sync() { asm volatile("bar.sync 1, %0;" ::"n"(THREADS) : "memory"); }

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtx& wc) {
  const bool ok = mbar_wait(bar, parity, wc);
  return __all_sync(0xffffffffu, ok) != 0;
}

// The work of one CTA: whole tiles in turn (blockIdx.x, + gridDim.x, ...), or
// with stream-K (SK) whole tiles below sk_first_tile and then its contiguous
// share of the remaining tiles' K blocks, as (tile, K block range) segments.
template <bool SK>
struct TcWork {
  int t, G, T, KB;
  __device__ __forceinline__ TcWork(int cid, int G_, int T_, int KB_, int) : t(cid), G(G_), T(T_), KB(KB_) {}
  __device__ __forceinline__ bool next(int& tile, int& kb0, int& kb1) {
    if (t >= T) return false;
    tile = t;
    kb0 = 0;
    kb1 = KB;
    t += G;
    return true;
  }
};
template <>
struct TcWork<true> {
  SegmentIter it;
  __device__ __forceinline__ TcWork(int cid, int G, int T, int KB, int t_dp) : it(cid, G, T, t_dp, KB, T) {}
  __device__ __forceinline__ bool next(int& tile, int& kb0, int& kb1) {
    int half;
    return it.next(tile, kb0, kb1, half);
  }
};

template <int BN, bool INT_MODE, bool SK, bool XF>
__global__ void __launch_bounds__(TcThreads<INT_MODE, XF>::THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ TcParams p) {
  static_assert(!(XF && (INT_MODE || SK)), "operand transforms run whole floating tiles");
  constexpr int EPI_WARPS = TcThreads<INT_MODE, XF>::EPI_WARPS;
  constexpr int XF_WARPS = TcThreads<INT_MODE, XF>::XF_WARPS;
  constexpr int CHUNKS = BN / 32 / (EPI_WARPS / 4);   // 32-column chunks per epilogue warp
  static_assert(!INT_MODE || BN == 128, "exact integer mode keeps 128 int32 accumulators per thread");
  using Cfg = TcCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;       // swizzle atoms need 1024-byte alignment
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t out_stage0 = base + (uint32_t)(Cfg::STAGES * Cfg::STAGE_BYTES);
  const uint32_t bar0 = out_stage0 + (uint32_t)Cfg::OUT_STAGE_BYTES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + Cfg::STAGES * Cfg::STAGE_BYTES +
                                                    Cfg::OUT_STAGE_BYTES + Cfg::NUM_BARS * 8);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);

  auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(Cfg::STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (uint32_t)(2 * Cfg::STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (uint32_t)(2 * Cfg::STAGES + Cfg::ACC_BUFS + b); };
  const uint32_t teardown_bar = bar0 + 8u * (uint32_t)(2 * Cfg::STAGES + 2 * Cfg::ACC_BUFS);
  // Operand transforms: the stage's tiles have been transformed.
  auto xf_bar = [&](int s) { return teardown_bar + 8u * (uint32_t)(1 + s); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(full_bar(s), 1);    // producer's expect_tx arrival + TMA bytes
      mbar_init(empty_bar(s), 1);   // tcgen05.commit after the stage's MMAs
    }
    for (int b = 0; b < Cfg::ACC_BUFS; ++b) {
      mbar_init(tfull_bar(b), 1);   // tcgen05.commit after a unit's last MMA
      mbar_init(tempty_bar(b), EPI_WARPS);  // one arrival per epilogue warp
    }
    mbar_init(teardown_bar, 1);
    if constexpr (XF)
      for (int s = 0; s < Cfg::STAGES; ++s) mbar_init(xf_bar(s), XF_WARPS);   // one arrival per transform warp
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The prologue above touches no global data: overlap it with the previous kernel.
  pdl_launch_dependents();
  pdl_wait();
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};

  const int units_per_tile = p.chunk_kb > 0 ? (p.num_kb + p.chunk_kb - 1) / p.chunk_kb : 1;
  const int kb_per_unit = p.chunk_kb > 0 ? p.chunk_kb : p.num_kb;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      tma_prefetch_desc(&p.tmA);
      tma_prefetch_desc(&p.tmB);
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_parity = 0;
      bool ok = true;
      TcWork<SK> it(blockIdx.x, gridDim.x, p.num_tiles, p.num_kb, p.sk_first_tile);
      int t, kb_lo, kb_hi;
      while (ok && it.next(t, kb_lo, kb_hi)) {
        int bz, tm, tn;
        tile_coords(t, p, bz, tm, tn);
        const int m0 = tm * TC_BM, n0 = tn * BN;
        const int za = p.a_batched ? bz : 0, zb = p.b_batched ? bz : 0;
        // One tile column (every tile streams its own rows of A once, all share B):
        // tile t loads its K blocks starting at one of 8 evenly spaced blocks and
        // wraps around, so the CTAs' concurrent reads of A spread over DRAM instead
        // of all reading the same K columns at once.  The MMAs consume the stages in
        // order; only the summation order of K changes.
        const int rot = p.k_rotate ? (int)(((int64_t)(t & 7) * p.num_kb) >> 3) : 0;
        for (int kb0 = kb_lo; kb0 < kb_hi; kb0 += Cfg::SLABS) {
          // A unit of the exact integer mode spans an even number of K blocks, so
          // stages never straddle two units.
          const int nsl = kb_hi - kb0 < Cfg::SLABS ? kb_hi - kb0 : Cfg::SLABS;
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, wc)) { ok = false; break; }
          const uint32_t fb = full_bar(stage);
          mbar_expect_tx(fb, (uint32_t)(nsl * (Cfg::A_BYTES + Cfg::B_BYTES)));
          const uint32_t st = base + (uint32_t)(stage * Cfg::STAGE_BYTES);
          for (int sl = 0; sl < nsl; ++sl) {
          const uint32_t sa = st + (uint32_t)(sl * Cfg::A_BYTES);
          const uint32_t sb = st + (uint32_t)(Cfg::SLABS * Cfg::A_BYTES + sl * Cfg::B_BYTES);
          int kp = kb0 + sl + rot;
          if (kp >= p.num_kb) kp -= p.num_kb;
          const int k0 = kp * TC_BK;
          if (p.a_mn_major) {
#pragma unroll
            for (int h = 0; h < TC_BM / MN_BOX; ++h)
              tma_load_3d(sa + h * MN_BOX_BYTES, &p.tmA, m0 + h * MN_BOX, k0, za, fb);
          } else {
            tma_load_3d(sa, &p.tmA, k0, m0, za, fb);
          }
          if (p.b_mn_major) {
#pragma unroll
            for (int h = 0; h < BN / MN_BOX; ++h)
              tma_load_3d(sb + h * MN_BOX_BYTES, &p.tmB, n0 + h * MN_BOX, k0, zb, fb);
          } else {
            tma_load_3d(sb, &p.tmB, k0, n0, zb, fb);
          }
          }
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == Cfg::STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // Every copy this thread started must have landed before the CTA exits.
      for (int s = 0; s < Cfg::STAGES; ++s)
        if (issued & (1u << s)) drain_wait(full_bar(s), (last_parity >> s) & 1u, p.timeout_ns);
    }
  } else if (warp == 1) {
    // ------------------------------- MMA issuer -------------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_it = 0;
      bool ok = true;
      TcWork<SK> it(blockIdx.x, gridDim.x, p.num_tiles, p.num_kb, p.sk_first_tile);
      int t, kb_lo, kb_hi;
      while (ok && it.next(t, kb_lo, kb_hi)) {
        // Integer mode: whole tiles in fp32 chunks of kb_per_unit K blocks.  Floating
        // mode: one unit, the segment's K blocks (all of them unless stream-K split the tile).
        const int units = INT_MODE ? units_per_tile : 1;
        for (int u = 0; ok && u < units; ++u) {
          const int buf = (int)(acc_it % Cfg::ACC_BUFS);
          const uint32_t apar = (acc_it / Cfg::ACC_BUFS) & 1u;
          if (!mbar_wait(tempty_bar(buf), apar ^ 1u, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
          const int kb_begin = INT_MODE ? u * kb_per_unit : kb_lo;
          const int kb_end = INT_MODE ? min(p.num_kb, kb_begin + kb_per_unit) : kb_hi;
          for (int kb = kb_begin; kb < kb_end; kb += Cfg::SLABS) {
            const int nsl = kb_end - kb < Cfg::SLABS ? kb_end - kb : Cfg::SLABS;
            if (!mbar_wait(XF ? xf_bar(stage) : full_bar(stage), phase, wc)) { ok = false; break; }
            tc_fence_after();
            const uint32_t st = base + (uint32_t)(stage * Cfg::STAGE_BYTES);
#pragma unroll
            for (int sl = 0; sl < Cfg::SLABS; ++sl) {
              if (sl >= nsl) break;
              const uint32_t sa = st + (uint32_t)(sl * Cfg::A_BYTES);
              const uint32_t sb = st + (uint32_t)(Cfg::SLABS * Cfg::A_BYTES + sl * Cfg::B_BYTES);
#pragma unroll
              for (int kk = 0; kk < TC_BK / 16; ++kk) {
                // K-major: the 16-element K step is 32 bytes inside each 128-byte row.
                // MN-major: it is 16 rows of 128 bytes; LBO steps between 64-wide MN boxes.
                const uint64_t ad = p.a_mn_major ? smem_desc_sw128(sa + kk * 2048u, MN_BOX_BYTES, 1024)
                                                 : smem_desc_sw128(sa + kk * 32u, 16, 1024);
                const uint64_t bd = p.b_mn_major ? smem_desc_sw128(sb + kk * 2048u, MN_BOX_BYTES, 1024)
                                                 : smem_desc_sw128(sb + kk * 32u, 16, 1024);
                tc_mma_f16(d_tmem, ad, bd, p.idesc, (kb > kb_begin || sl > 0 || kk > 0) ? 1u : 0u);
              }
            }
            tc_commit(empty_bar(stage));
            if (++stage == Cfg::STAGES) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          tc_commit(tfull_bar(buf));
          ++acc_it;
        }
      }
      // Every MMA this thread issued must be complete before tensor memory is freed.
      tc_commit(teardown_bar);
      drain_wait(teardown_bar, 0, p.timeout_ns);
    }
  } else if (XF && warp >= 2 + EPI_WARPS) {
    // ---------------------------- operand transforms ----------------------------
    // Wait for a stage's copies, transform the loaded A and/or B bytes in place,
    // make the writes visible to the tensor cores (async proxy), count the warp in.
    constexpr int NT = 32 * XF_WARPS;
    const int xt = (int)threadIdx.x - 32 * (2 + EPI_WARPS);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    TcWork<SK> it(blockIdx.x, gridDim.x, p.num_tiles, p.num_kb, p.sk_first_tile);
    int t, kb_lo, kb_hi;
    while (ok && it.next(t, kb_lo, kb_hi)) {
      for (int kb0 = kb_lo; kb0 < kb_hi; kb0 += Cfg::SLABS) {
        const int nsl = kb_hi - kb0 < Cfg::SLABS ? kb_hi - kb0 : Cfg::SLABS;
        if (!warp_wait(full_bar(stage), phase, wc)) { ok = false; break; }
        const uint32_t st = base + (uint32_t)(stage * Cfg::STAGE_BYTES);
        if (p.xf.a_on)
          xf_smem(st, (uint32_t)(nsl * Cfg::A_BYTES), p.xf, 0, xt, NT);
        if (p.xf.b_on)
          xf_smem(st + (uint32_t)(Cfg::SLABS * Cfg::A_BYTES), (uint32_t)(nsl * Cfg::B_BYTES), p.xf, 1, xt, NT);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(xf_bar(stage));
        if (++stage == Cfg::STAGES) { stage = 0; phase ^= 1u; }
      }
    }
  } else {
    // -------------------------------- epilogue --------------------------------
    const int q = warp & 3;                          // TMEM lane quarter this warp may access
    const int c0 = ((warp - 2) >> 2) * CHUNKS;       // this warp's first 32-column chunk
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    volatile int32_t* sk_role = abort_flag + 1;   // stream-K: this CTA finishes the tile (1), aborted (2)
    uint32_t acc_it = 0;
    bool ok = true;
    TcWork<SK> it(blockIdx.x, gridDim.x, p.num_tiles, p.num_kb, p.sk_first_tile);
    int t, kb_lo, kb_hi;
    while (ok && it.next(t, kb_lo, kb_hi)) {
      int bz, tm, tn;
      tile_coords(t, p, bz, tm, tn);
      const int64_t m = (int64_t)tm * TC_BM + q * 32 + lane;
      const int64_t n0 = (int64_t)tn * BN;
      const bool row_ok = m < p.M;
      const EpiPtrs ptr = epi_ptrs(p.epi, bz);
      if constexpr (INT_MODE) {
        int32_t acc[BN];
#pragma unroll
        for (int j = 0; j < BN; ++j) acc[j] = 0;
        for (int u = 0; u < units_per_tile; ++u) {
          const int buf = (int)(acc_it % Cfg::ACC_BUFS);
          const uint32_t apar = (acc_it / Cfg::ACC_BUFS) & 1u;
          if (!warp_wait(tfull_bar(buf), apar, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t tb = tmem_base + lane_base + (uint32_t)(buf * BN);
#pragma unroll
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tb + (uint32_t)(c * 32), r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[c * 32 + j] += __float2int_rn(__uint_as_float(r[j]));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(buf));
          ++acc_it;
        }
        if (!ok) break;
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) epi_finish_row32_int(p.epi, ptr, m, row_ok, n0 + c * 32, p.N, &acc[c * 32]);
      } else if (SK && (kb_lo > 0 || kb_hi < p.num_kb)) {
        // Stream-K: this CTA holds K blocks [kb_lo, kb_hi) of tile t, which several
        // CTAs share.  It publishes its raw fp32 partial, then counts itself in on
        // the tile; the CTA that arrives last adds every part, in the order of the
        // K blocks, and runs the epilogue.  No CTA waits for another.  Every
        // epilogue warp reaches both CTA barriers below, whatever happened before.
        const int buf = (int)(acc_it % Cfg::ACC_BUFS);
        const uint32_t apar = (acc_it / Cfg::ACC_BUFS) & 1u;
        const bool w_ok = warp_wait(tfull_bar(buf), apar, wc);
        constexpr int SLOT_FLOATS = TC_BM * BN;
        const int G = (int)gridDim.x;
        const int64_t W = (int64_t)(p.num_tiles - p.sk_first_tile) * p.num_kb;
        const int64_t tl = t - p.sk_first_tile;
        const int row_in_cta = q * 32 + lane;
        // Slot 0 of a CTA holds the part of the tile its K range starts in, slot 1 the other.
        auto slot_of = [&](int cta) {
          const int64_t start = (int64_t)cta * W / G;
          return p.sk_partials + (size_t)(cta * 2 + (start / p.num_kb == tl ? 0 : 1)) * SLOT_FLOATS;
        };
        if (w_ok) {
          tc_fence_after();
          const uint32_t tb = tmem_base + lane_base + (uint32_t)(buf * BN);
          float4* slot = reinterpret_cast<float4*>(slot_of((int)blockIdx.x));
#pragma unroll 1
          for (int c = c0; c < c0 + CHUNKS; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tb + (uint32_t)(c * 32), r);
            tmem_wait_ld();
#pragma unroll
            for (int v = 0; v < 8; ++v)
              __stcg(&slot[(c * 8 + v) * TC_BM + row_in_cta],
                     make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                 __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3])));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(buf));
        }
        __threadfence();
        epi_warps_sync<32 * EPI_WARPS>();
        const int c_first = sk_cluster_of(tl * p.num_kb, W, G);
        const int c_last = sk_cluster_of(tl * p.num_kb + p.num_kb - 1, W, G);
        if (warp == 2 && lane == 0) {
          if (*wc.abort) {
            *sk_role = 2;
          } else {
            const int old = atomicAdd(&p.sk_flags[t], 1);
            *sk_role = old == c_last - c_first ? 1 : 0;
          }
        }
        epi_warps_sync<32 * EPI_WARPS>();
        const int role = *sk_role;
        if (role == 2) { ok = false; break; }
        if (role == 1) {
          __threadfence();
#pragma unroll 1
          for (int c = c0; c < c0 + CHUNKS; ++c) {
            float x[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = 0.0f;
            // Two parts' loads in flight per round trip (the sum keeps the parts' order).
#pragma unroll 1
            for (int cc = c_first; cc <= c_last; cc += 2) {
              const bool two = cc + 1 <= c_last;
              const float4* s4a = reinterpret_cast<const float4*>(slot_of(cc));
              const float4* s4b = reinterpret_cast<const float4*>(slot_of(two ? cc + 1 : cc));
              float4 ya[8], yb[8];
#pragma unroll
              for (int v = 0; v < 8; ++v) ya[v] = __ldcg(&s4a[(c * 8 + v) * TC_BM + row_in_cta]);
              if (two) {
#pragma unroll
                for (int v = 0; v < 8; ++v) yb[v] = __ldcg(&s4b[(c * 8 + v) * TC_BM + row_in_cta]);
              }
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                x[4 * v] += ya[v].x;
                x[4 * v + 1] += ya[v].y;
                x[4 * v + 2] += ya[v].z;
                x[4 * v + 3] += ya[v].w;
              }
              if (two) {
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                  x[4 * v] += yb[v].x;
                  x[4 * v + 1] += yb[v].y;
                  x[4 * v + 2] += yb[v].z;
                  x[4 * v + 3] += yb[v].w;
                }
              }
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] *= p.epi.alpha;
            epi_finish_row32_float(p.epi, ptr, m, row_ok, n0 + c * 32, p.N, x,
                                   out_stage0 + (uint32_t)((warp - 2) * 4096), p.M);
          }
          // Every part has been counted and read: the counter is ready for the next launch.
          if (warp == 2 && lane == 0) p.sk_flags[t] = 0;
        }
        ++acc_it;
      } else {
        const int buf = (int)(acc_it % Cfg::ACC_BUFS);
        const uint32_t apar = (acc_it / Cfg::ACC_BUFS) & 1u;
        if (!warp_wait(tfull_bar(buf), apar, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tb = tmem_base + lane_base + (uint32_t)(buf * BN);
        const uint32_t stage_buf = out_stage0 + (uint32_t)((warp - 2) * 4096);
        // The common epilogues in loops specialised on D's type, the others on the
        // general per-chunk path.
        auto acc = [&](int c, float (&x)[32]) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tb + (uint32_t)(c * 32), r);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]) * p.epi.alpha;
        };
        if (!epi_chunks_typed(p.epi, ptr, m - lane, n0, p.N, p.M, stage_buf, c0, c0 + CHUNKS, acc)) {
#pragma unroll 1
          for (int c = c0; c < c0 + CHUNKS; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tb + (uint32_t)(c * 32), r);
            tmem_wait_ld();
            float x[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]) * p.epi.alpha;
            epi_finish_row32_float(p.epi, ptr, m, row_ok, n0 + c * 32, p.N, x, stage_buf, p.M);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(buf));
        ++acc_it;
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

template <int BN, bool INT_MODE, bool SK, bool XF = false>
cudaError_t launch_bn(const TcParams& p, int grid, cudaStream_t stream) {
  using Cfg = TcCfg<BN>;
  static_assert(Cfg::SMEM <= 232448, "shared memory budget");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool configured[64] = {};
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(tc_gemm_kernel<BN, INT_MODE, SK, XF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Cfg::SMEM);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  // A programmatic dependent of the previous kernel: one CTA per SM, none waits
  // for another, so starting early on free SMs is safe (see pdl_wait).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(TcThreads<INT_MODE, XF>::THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<BN, INT_MODE, SK, XF>, p);
}

}  // namespace

int tc_stages(int bn) { return bn == 256 ? TcCfg<256>::STAGES : bn == 128 ? TcCfg<128>::STAGES : TcCfg<64>::STAGES; }
int tc_k_per_stage(int bn) {
  return (bn == 256 ? TcCfg<256>::SLABS : bn == 128 ? TcCfg<128>::SLABS : TcCfg<64>::SLABS) * TC_BK;
}
size_t tc_smem_bytes(int bn) { return bn == 256 ? TcCfg<256>::SMEM : bn == 128 ? TcCfg<128>::SMEM : TcCfg<64>::SMEM; }

cudaError_t launch_tc(const TcParams& p, int bn, int grid, cudaStream_t stream) {
  if (p.chunk_kb > 0) {
    // exact integer mode keeps 128 int32 accumulators per thread: BN = 128 only
    if (p.xf.a_on || p.xf.b_on) return cudaErrorInvalidValue;   // int8 transforms run in the staging pass
    return bn == 128 ? launch_bn<128, true, false>(p, grid, stream) : cudaErrorInvalidValue;
  }
  const bool sk = p.sk_first_tile < p.num_tiles;   // stream-K: a separate instance, so whole tiles lose nothing
  if (p.xf.a_on || p.xf.b_on) {
    // Operand transforms: their own instance, whole tiles (the host turns stream-K off).
    if (sk) return cudaErrorInvalidValue;
    if (bn == 256) return launch_bn<256, false, false, true>(p, grid, stream);
    if (bn == 128) return launch_bn<128, false, false, true>(p, grid, stream);
    if (bn == 64) return launch_bn<64, false, false, true>(p, grid, stream);
    return cudaErrorInvalidValue;
  }
  if (bn == 256) return sk ? launch_bn<256, false, true>(p, grid, stream) : launch_bn<256, false, false>(p, grid, stream);
  if (bn == 128) return sk ? launch_bn<128, false, true>(p, grid, stream) : launch_bn<128, false, false>(p, grid, stream);
  if (bn == 64) return sk ? launch_bn<64, false, true>(p, grid, stream) : launch_bn<64, false, false>(p, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gemmlib

// tc2_kernel.cu -- tcgen05 GEMM on CTA pairs (cta_group::2), 256 x 256 tiles.
//
// Same computation and epilogue as tc_kernel.cu, with one output tile of
// 256 (M) x 256 (N) per cluster of two CTAs on two SMs:
//   - CTA r of the pair stages, per 64-deep K block, its own 128 rows of A
//     (rows m0 + 128r ...) and its own half of B (columns n0 + 128r ...) --
//     32 KiB per K block; a pipeline stage holds two K blocks (64 KiB) and the
//     ring has three stages -- so each SM moves 2/3 of the operand bytes of a
//     128 x 256 single-CTA tile for the same MMA work;
//   - both CTAs' TMA loads complete on the leader CTA's (rank 0) full barrier;
//   - one thread of the leader issues tcgen05.mma.cta_group::2 (M = 256,
//     N = 256, K = 16): the hardware takes A's rows from both CTAs and B's halves
//     from both CTAs, and writes each CTA's 128 rows of D into that CTA's tensor
//     memory (two 256-column fp32 accumulators per CTA, double buffered);
//   - its commits arrive on both CTAs' barriers (the commit's CTA mask): the
//     stage-free barriers that the two producers wait on and the
//     accumulator-full barriers the two epilogues wait on;
//   - the epilogue warps of both CTAs finish their 128 rows (alpha, beta*C,
//     bias, ReLU, cast, 16-byte stores) and release the accumulator on the
//     leader's barrier (the peer's four warps arrive remotely).
// Exact integer mode (int8 operands staged as fp16): the MMA accumulates each
// 1024-deep K chunk into a fresh fp32 accumulator (exact, |sum| <= 2^24); eight
// epilogue warps per CTA -- two per tensor-memory lane quarter, one per half of
// the 256 columns -- convert each finished chunk to int32 and add it into 128
// registers per thread, then apply the integer epilogue after the last chunk.
// Operand transforms (a separate instance, XF): four more warps per CTA apply
// t(x) = act(scale * x) in place to the CTA's staged A and/or B tiles of each
// stage.  Then each CTA's TMA loads complete on its own full barrier, the
// transform warps of both CTAs wait there, transform, fence the async proxy and
// arrive on the leader's stage-transformed barrier, which is what the MMA
// thread waits for instead of the full barrier.
// Every TMA load brings one CTA's own operand data into that CTA's shared
// memory; no load is delivered to more than one CTA.
// Every mbarrier wait is bounded, as in tc_kernel.cu.
#include "kernels.h"

namespace gemmlib {
namespace {

constexpr int PAIR_BN = 256;                            // tile columns (both CTAs)
constexpr int PAIR_A_BYTES = TC_BM * TC_BK * 2;          // 16 KiB: this CTA's 128 rows of A
constexpr int PAIR_B_BYTES = (PAIR_BN / 2) * TC_BK * 2;  // 16 KiB: this CTA's half of B
// One stage holds PAIR_SLABS consecutive 64-deep K blocks (slabs).  Every stage
// costs one stage-full wait and one tcgen05.commit in the MMA thread, and each of
// those holds the tensor pipe for a while; two slabs per stage (eight MMAs per
// commit) keep it busy ~91 % of the time where one slab per stage managed ~83 %
// (measured at 8192^3).
#ifndef GEMM_PAIR_SLABS
#define GEMM_PAIR_SLABS 2
#endif
constexpr int PAIR_SLABS = GEMM_PAIR_SLABS;
constexpr int PAIR_SLAB_BYTES = PAIR_A_BYTES + PAIR_B_BYTES;   // 32 KiB
constexpr int PAIR_STAGE_BYTES = PAIR_SLABS * PAIR_SLAB_BYTES;  // [A slabs][B slabs]
constexpr int PAIR_ACC_BUFS = 2;                        // 2 x 256 fp32 columns of TMEM
#ifndef GEMM_PAIR_STAGES
#define GEMM_PAIR_STAGES (6 / GEMM_PAIR_SLABS)
#endif
constexpr int PAIR_STAGES = GEMM_PAIR_STAGES;
constexpr int PAIR_NUM_BARS = 3 * PAIR_STAGES + 2 * PAIR_ACC_BUFS + 2;
constexpr int PAIR_OUT_STAGE_BYTES = 4 * 4096;   // a 32 x 32 output turn-around buffer per floating epilogue warp
constexpr size_t PAIR_SMEM =
    1024 + (size_t)PAIR_STAGES * PAIR_STAGE_BYTES + PAIR_OUT_STAGE_BYTES + PAIR_NUM_BARS * 8 + 16;

// Producer warp, MMA warp, then 4 epilogue warps (floating) or 8 (exact integer),
// then (operand transforms) 4 transform warps.
template <bool INT_MODE, bool XF>
struct PairThreads {
  static constexpr int EPI_WARPS = INT_MODE ? 8 : 4;
  static constexpr int XF_WARPS = XF ? 4 : 0;
  static constexpr int THREADS = 64 + 32 * (EPI_WARPS + XF_WARPS);
};
constexpr uint32_t PAIR_TMEM_COLS = 512;
constexpr int MN_BOX = 64;   // MN extent of one TMA box of an MN-major operand (128 bytes)
// An MN-major operand is loaded in boxes of 64 (MN) x PAIR_SLABS * 64 (K): one
// box per 64-wide MN group per stage (fewer, larger copies than one per K block).
constexpr uint32_t MN_STAGE_BYTES = MN_BOX * 2 * PAIR_SLABS * TC_BK;

__device__ __forceinline__ void pair_tile_coords(int t, const TcParams& p, int& bz, int& tm, int& tn) {
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

__device__ __forceinline__ void drain_wait_pair(uint32_t bar, uint32_t parity, uint64_t user_timeout_ns) {
  const uint64_t timeout_ns = user_timeout_ns > 1000000000ull ? user_timeout_ns : 1000000000ull;
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) return;
  }
}

__device__ __forceinline__ bool warp_wait_pair(uint32_t bar, uint32_t parity, const WaitCtx& wc) {
  const bool ok = mbar_wait(bar, parity, wc);
  return __all_sync(0xffffffffu, ok) != 0;
}

// One CTA pair per cluster of two.  A_MN / B_MN: the operand is stored
// MN-contiguous (A column-major, B row-major) rather than K-contiguous.
template <bool INT_MODE, bool A_MN, bool B_MN, bool XF>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairThreads<INT_MODE, XF>::THREADS, 1)
    tc_pair_gemm_kernel(const __grid_constant__ TcParams p) {
  static_assert(!(XF && INT_MODE), "int8 operands are transformed in their staging pass");
  constexpr int EPI_WARPS = PairThreads<INT_MODE, XF>::EPI_WARPS;
  constexpr int XF_WARPS = PairThreads<INT_MODE, XF>::XF_WARPS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;   // same offset in both CTAs
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t out_stage0 = base + (uint32_t)(PAIR_STAGES * PAIR_STAGE_BYTES);
  const uint32_t bar0 = out_stage0 + (uint32_t)PAIR_OUT_STAGE_BYTES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + PAIR_STAGES * PAIR_STAGE_BYTES +
                                                    PAIR_OUT_STAGE_BYTES + PAIR_NUM_BARS * 8);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);

  auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(PAIR_STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (uint32_t)(2 * PAIR_STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (uint32_t)(2 * PAIR_STAGES + PAIR_ACC_BUFS + b); };
  const uint32_t teardown_bar = bar0 + 8u * (uint32_t)(2 * PAIR_STAGES + 2 * PAIR_ACC_BUFS);
  const uint32_t sk_bar = teardown_bar + 8u;   // epilogue warps: stream-K partial written
  // Operand transforms: stage transformed in both CTAs (the leader's barrier counts).
  auto xf_bar = [&](int s) { return sk_bar + 8u * (uint32_t)(1 + s); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank() & 1u;    // position in the CTA pair
  const uint32_t pair_leader = 0;                  // cluster rank of the pair's leader
  const bool leader = rank == 0;
  const int cluster_id = (int)(blockIdx.x / 2);
  const int num_clusters = (int)(gridDim.x / 2);

  if (threadIdx.x == 0) {
    for (int s = 0; s < PAIR_STAGES; ++s) {
      mbar_init(full_bar(s), 1);    // leader: its expect_tx arrival + both CTAs' TMA bytes
      mbar_init(empty_bar(s), 1);   // the leader's commit (CTA mask: both CTAs)
    }
    for (int b = 0; b < PAIR_ACC_BUFS; ++b) {
      mbar_init(tfull_bar(b), 1);   // the leader's commit (CTA mask: both CTAs)
      mbar_init(tempty_bar(b), 2 * EPI_WARPS);  // leader: every epilogue warp of both CTAs
    }
    mbar_init(teardown_bar, 1);
    mbar_init(sk_bar, EPI_WARPS);
    if constexpr (XF)
      for (int s = 0; s < PAIR_STAGES; ++s) mbar_init(xf_bar(s), 2 * XF_WARPS);   // transform warps of both CTAs
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  cluster_sync();                                   // both CTAs' barriers exist
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), PAIR_TMEM_COLS);
  tc_fence_before();
  cluster_sync();                                   // tensor memory allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The prologue above touches no global data: overlap it with the previous kernel.
  pdl_launch_dependents();
  pdl_wait();
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};
  // Integer mode runs whole tiles (the host turns the stream-K tail off for it).
  const int kb_per_unit = INT_MODE ? p.chunk_kb : p.num_kb;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      tma_prefetch_desc(&p.tmA);
      tma_prefetch_desc(&p.tmB);
      if (p.half_first_tile < p.num_tiles) tma_prefetch_desc(&p.tmBh);
      // A's row panels serve every wave of tiles in a raster group, B's column
      // panels one wave: half of A's lines are kept in L2 ahead of other lines,
      // which cuts the DRAM reads of an 8192^3 launch by 11 % (measured).
      uint64_t a_policy;
      asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 0.5;" : "=l"(a_policy));
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_parity = 0;
      bool ok = true;
      SegmentIter it(cluster_id, num_clusters, p.num_tiles, p.sk_first_tile, p.num_kb, p.half_first_tile);
      int tile, kb0, kb1, half;
      while (ok && it.next(tile, kb0, kb1, half)) {
        int bz, tm, tn;
        pair_tile_coords(tile, p, bz, tm, tn);
        const int m0 = tm * (2 * TC_BM) + (int)rank * TC_BM;        // this CTA's rows of A
        // This CTA's half of B's columns: 128 of a whole tile, 64 of a half-tile unit.
        const int n0 = half < 0 ? tn * PAIR_BN + (int)rank * (PAIR_BN / 2)
                                : tn * PAIR_BN + half * (PAIR_BN / 2) + (int)rank * (PAIR_BN / 4);
        const int za = p.a_batched ? bz : 0, zb = p.b_batched ? bz : 0;
        // B bytes of one K block for this CTA: 128 columns of a whole tile, 64 of a half-tile unit.
        const uint32_t b_slab_bytes = half < 0 ? (uint32_t)PAIR_B_BYTES : (uint32_t)(PAIR_B_BYTES / 2);
        for (int kb = kb0; kb < kb1; kb += PAIR_SLABS) {
          const int nsl = kb1 - kb < PAIR_SLABS ? kb1 - kb : PAIR_SLABS;   // K blocks in this stage
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, wc)) { ok = false; break; }
          const uint32_t fb_local = full_bar(stage);
          // An MN-major operand arrives in stage-deep boxes, which always carry the
          // whole stage (zero-filled past K); a K-major one in one box per K block.
          const uint32_t a_bytes = (uint32_t)(A_MN ? PAIR_SLABS : nsl) * (uint32_t)PAIR_A_BYTES;
          const uint32_t b_bytes = (uint32_t)(B_MN ? PAIR_SLABS : nsl) * b_slab_bytes;
          // With operand transforms each CTA's copies complete on its own full
          // barrier (its transform warps wait there); otherwise both CTAs' copies
          // complete on the leader's.
          if (XF) mbar_expect_tx(fb_local, a_bytes + b_bytes);
          else if (leader) mbar_expect_tx(fb_local, 2u * (a_bytes + b_bytes));
          const uint32_t fb = (XF || leader) ? fb_local : mapa_shared(fb_local, pair_leader);
          const uint32_t sa = base + (uint32_t)(stage * PAIR_STAGE_BYTES);
          const uint32_t sb = sa + (uint32_t)(PAIR_SLABS * PAIR_A_BYTES);
          const int k0 = kb * TC_BK;
          if constexpr (A_MN) {
#pragma unroll
            for (int h = 0; h < TC_BM / MN_BOX; ++h)
              tma_load_3d_pair_hint(sa + h * MN_STAGE_BYTES, &p.tmA, m0 + h * MN_BOX, k0, za, fb, a_policy);
          } else {
            for (int sl = 0; sl < nsl; ++sl)
              tma_load_3d_pair_hint(sa + sl * PAIR_A_BYTES, &p.tmA, k0 + sl * TC_BK, m0, za, fb, a_policy);
          }
          if constexpr (B_MN) {
            // 128 columns: two stage-deep boxes of 64; a half-tile unit's 64 columns: one.
            const int nh = half < 0 ? (PAIR_BN / 2) / MN_BOX : 1;
            for (int h = 0; h < nh; ++h)
              tma_load_3d_pair(sb + h * MN_STAGE_BYTES, &p.tmB, n0 + h * MN_BOX, k0, zb, fb);
          } else {
            // One box per K block: 128 rows (tmB), or 64 rows for a half-tile unit (tmBh).
            const CUtensorMap* tb = half < 0 ? &p.tmB : &p.tmBh;
            for (int sl = 0; sl < nsl; ++sl) tma_load_3d_pair(sb + sl * PAIR_B_BYTES, tb, k0 + sl * TC_BK, n0, zb, fb);
          }
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == PAIR_STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // The leader's full barriers count both CTAs' bytes: once its drains pass,
      // every copy of the pair has landed (the peer waits at the final cluster barrier).
      // With operand transforms every CTA's barriers count its own copies.
      if (leader || XF) {
        for (int s = 0; s < PAIR_STAGES; ++s)
          if (issued & (1u << s)) drain_wait_pair(full_bar(s), (last_parity >> s) & 1u, p.timeout_ns);
      } else if (!ok) {
        // Wind-down after a failure: give this CTA's own copies time to land
        // before it can leave (they complete on the leader's barrier).
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------- MMA issuer (leader CTA only) ----------------------
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_it = 0;
      bool ok = true;
      SegmentIter it(cluster_id, num_clusters, p.num_tiles, p.sk_first_tile, p.num_kb, p.half_first_tile);
      int tile, kb0, kb1, half;
      while (ok && it.next(tile, kb0, kb1, half)) {
        const int units = INT_MODE ? (kb1 - kb0 + kb_per_unit - 1) / kb_per_unit : 1;
        const uint32_t idesc = half < 0 ? p.idesc : p.idesc_half;   // N = 256, or 128 for a half-tile unit
        for (int u = 0; ok && u < units; ++u) {
          const int buf = (int)(acc_it % PAIR_ACC_BUFS);
          const uint32_t apar = (acc_it / PAIR_ACC_BUFS) & 1u;
          if (!mbar_wait(tempty_bar(buf), apar ^ 1u, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(buf * PAIR_BN);
          const int kb_begin = INT_MODE ? kb0 + u * kb_per_unit : kb0;
          const int kb_end = INT_MODE ? min(kb1, kb_begin + kb_per_unit) : kb1;
          for (int kb = kb_begin; kb < kb_end; kb += PAIR_SLABS) {
            const int nsl = kb_end - kb < PAIR_SLABS ? kb_end - kb : PAIR_SLABS;
            const bool landed = XF ? mbar_wait_cluster(xf_bar(stage), phase, wc) : mbar_wait(full_bar(stage), phase, wc);
            if (!landed) { ok = false; break; }
            tc_fence_after();
            const uint32_t sa = base + (uint32_t)(stage * PAIR_STAGE_BYTES);
            const uint32_t sb = sa + (uint32_t)(PAIR_SLABS * PAIR_A_BYTES);
#pragma unroll
            for (int sl = 0; sl < PAIR_SLABS; ++sl) {
              if (sl >= nsl) break;
#pragma unroll
              for (int kk = 0; kk < TC_BK / 16; ++kk) {
                // K-major: one 128-byte-wide box per K block; the 16-element K step is
                // 32 bytes inside each row.  MN-major: stage-deep boxes of 64 MN; the K
                // step is 16 rows of 128 bytes, LBO steps from one 64-wide box to the next.
                const uint64_t ad = A_MN ? smem_desc_sw128(sa + sl * (TC_BK * 128u) + kk * 2048u, MN_STAGE_BYTES, 1024)
                                         : smem_desc_sw128(sa + sl * PAIR_A_BYTES + kk * 32u, 16, 1024);
                const uint64_t bd = B_MN ? smem_desc_sw128(sb + sl * (TC_BK * 128u) + kk * 2048u, MN_STAGE_BYTES, 1024)
                                         : smem_desc_sw128(sb + sl * PAIR_B_BYTES + kk * 32u, 16, 1024);
                tc_mma_f16_pair(d_tmem, ad, bd, idesc, (kb > kb_begin || sl > 0 || kk > 0) ? 1u : 0u);
              }
            }
            tc_commit_pair_mask(empty_bar(stage), 0x3);   // both CTAs' producers
            if (++stage == PAIR_STAGES) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          tc_commit_pair_mask(tfull_bar(buf), (uint16_t)(0x3u << pair_leader));
          ++acc_it;
        }
      }
      tc_commit_pair(teardown_bar);
      drain_wait_pair(teardown_bar, 0, p.timeout_ns);
    }
  } else if (XF && warp >= 2 + EPI_WARPS) {
    // ------------------------ operand transforms (both CTAs) ------------------------
    // Wait for this CTA's copies of a stage, transform the loaded bytes of A and/or
    // B in place, make the writes visible to the tensor cores (async proxy) and
    // count the warp in on the leader's stage-transformed barrier.
    constexpr int NT = 32 * XF_WARPS;
    const int xt = (int)threadIdx.x - 32 * (2 + EPI_WARPS);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    SegmentIter it(cluster_id, num_clusters, p.num_tiles, p.sk_first_tile, p.num_kb, p.half_first_tile);
    int tile, kb0, kb1, half;
    while (ok && it.next(tile, kb0, kb1, half)) {
      for (int kb = kb0; kb < kb1; kb += PAIR_SLABS) {
        const int nsl = kb1 - kb < PAIR_SLABS ? kb1 - kb : PAIR_SLABS;
        if (!warp_wait_pair(full_bar(stage), phase, wc)) { ok = false; break; }
        const uint32_t sa = base + (uint32_t)(stage * PAIR_STAGE_BYTES);
        const uint32_t sb = sa + (uint32_t)(PAIR_SLABS * PAIR_A_BYTES);
        if (p.xf.a_on)
          xf_smem(sa, (uint32_t)(A_MN ? PAIR_SLABS : nsl) * (uint32_t)PAIR_A_BYTES, p.xf, 0, xt, NT);
        if (p.xf.b_on) {
          if (B_MN) {
            xf_smem(sb, (half < 0 ? 2u : 1u) * MN_STAGE_BYTES, p.xf, 1, xt, NT);
          } else if (half < 0) {
            xf_smem(sb, (uint32_t)nsl * (uint32_t)PAIR_B_BYTES, p.xf, 1, xt, NT);
          } else {
            for (int sl = 0; sl < nsl; ++sl)
              xf_smem(sb + (uint32_t)(sl * PAIR_B_BYTES), (uint32_t)(PAIR_B_BYTES / 2), p.xf, 1, xt, NT);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(xf_bar(stage));
          else mbar_arrive_cluster(mapa_shared(xf_bar(stage), pair_leader));
        }
        if (++stage == PAIR_STAGES) { stage = 0; phase ^= 1u; }
      }
    }
  } else {
    // ---------------------------- epilogue (both CTAs) ----------------------------
    const int q = warp & 3;                                   // TMEM lane quarter of this warp
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t acc_it = 0;
    bool ok = true;
    SegmentIter it(cluster_id, num_clusters, p.num_tiles, p.sk_first_tile, p.num_kb, p.half_first_tile);
    int tile, kb0, kb1, half;
    while (ok && it.next(tile, kb0, kb1, half)) {
      int bz, tm, tn;
      pair_tile_coords(tile, p, bz, tm, tn);
      const int row_in_cta = q * 32 + lane;
      const int64_t m = (int64_t)tm * (2 * TC_BM) + (int64_t)rank * TC_BM + row_in_cta;
      // A half-tile unit's columns start half a tile further and fill half the accumulator.
      const int64_t n0 = (int64_t)tn * PAIR_BN + (half > 0 ? PAIR_BN / 2 : 0);
      const int chunks = half < 0 ? PAIR_BN / 32 : PAIR_BN / 64;
      const bool row_ok = m < p.M;
      const EpiPtrs ptr = epi_ptrs(p.epi, bz);
      if constexpr (INT_MODE) {
        const int colh = (warp - 2) >> 2;                     // columns 128*colh ... 128*colh + 127
        const int units = (kb1 - kb0 + kb_per_unit - 1) / kb_per_unit;
        int32_t acc[128];
#pragma unroll
        for (int j = 0; j < 128; ++j) acc[j] = 0;
        for (int u = 0; u < units; ++u) {
          const int buf = (int)(acc_it % PAIR_ACC_BUFS);
          const uint32_t apar = (acc_it / PAIR_ACC_BUFS) & 1u;
          if (!warp_wait_pair(tfull_bar(buf), apar, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t tb = tmem_base + lane_base + (uint32_t)(buf * PAIR_BN + colh * 128);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tb + (uint32_t)(c * 32), r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[c * 32 + j] += __float2int_rn(__uint_as_float(r[j]));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (leader) mbar_arrive(tempty_bar(buf));
            else mbar_arrive_cluster(mapa_shared(tempty_bar(buf), pair_leader));
          }
          ++acc_it;
        }
        if (!ok) break;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          epi_finish_row32_int(p.epi, ptr, m, row_ok, n0 + colh * 128 + c * 32, p.N, &acc[c * 32]);
      } else {
        const int buf = (int)(acc_it % PAIR_ACC_BUFS);
        const uint32_t apar = (acc_it / PAIR_ACC_BUFS) & 1u;
        if (!warp_wait_pair(tfull_bar(buf), apar, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tb = tmem_base + lane_base + (uint32_t)(buf * PAIR_BN);
        // Stream-K slots hold raw accumulators (before alpha), 128 x 256 fp32 per CTA,
        // laid out so that each 16-byte column group of a warp's 32 rows is contiguous.
        constexpr int SLOT_FLOATS = TC_BM * PAIR_BN;
        if (kb0 > 0) {
          // A later part of a tile whose first part another cluster owns: publish it.
          float* slot = p.sk_partials + (size_t)(cluster_id * 2 + (int)rank) * SLOT_FLOATS;
#pragma unroll 1
          for (int c = 0; c < PAIR_BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tb + (uint32_t)(c * 32), r);
            tmem_wait_ld();
#pragma unroll
            for (int v = 0; v < 8; ++v)
              reinterpret_cast<float4*>(slot)[(c * 8 + v) * TC_BM + row_in_cta] =
                  make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                              __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (leader) mbar_arrive(tempty_bar(buf));
            else mbar_arrive_cluster(mapa_shared(tempty_bar(buf), pair_leader));
            __threadfence();
            mbar_arrive(sk_bar);
          }
          if (warp == 2 && lane == 0) {
            // Every epilogue warp of this CTA has written its rows: release the partial.
            if (mbar_wait(sk_bar, 0, wc)) {
              __threadfence();
              st_release_gpu(&p.sk_flags[cluster_id * 2 + (int)rank], p.sk_epoch);
            }
          }
        } else {
          // A whole tile, or the first part of a tile (then add the later parts).
          int cp_first = 0, cp_last = -1;
          if (kb1 < p.num_kb) {
            const int64_t W = (int64_t)(p.num_tiles - p.sk_first_tile) * p.num_kb;
            const int64_t tl = tile - p.sk_first_tile;
            cp_first = cluster_id + 1;
            cp_last = sk_cluster_of(tl * p.num_kb + p.num_kb - 1, W, num_clusters);
            int good = 1;
            if (lane == 0) {
              for (int cp = cp_first; cp <= cp_last && good; ++cp) {
                const int32_t* f = &p.sk_flags[cp * 2 + (int)rank];
                if (ld_acquire_gpu(f) == p.sk_epoch) continue;
                const uint64_t t0 = globaltimer_ns();
                while (ld_acquire_gpu(f) != p.sk_epoch) {
                  if (*wc.abort) { good = 0; break; }
                  if (globaltimer_ns() - t0 > wc.timeout_ns) {
                    atomicCAS(wc.err, 0, (int32_t)GEMM_ERR_TIMEOUT);
                    *wc.abort = 1;
                    good = 0;
                    break;
                  }
                  __nanosleep(256);
                }
              }
            }
            good = __shfl_sync(0xffffffffu, good, 0);
            __syncwarp();
            if (!good) cp_last = cp_first - 1;   // results are void; the error word says why
          }
          const uint32_t stage_buf = out_stage0 + (uint32_t)((warp - 2) * 4096);
          // A whole tile (no later parts to add): the common epilogues run in loops
          // specialised on D's type, the others on the general per-chunk path.
          auto acc = [&](int c, float (&x)[32]) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tb + (uint32_t)(c * 32), r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]) * p.epi.alpha;
          };
          if (cp_last >= cp_first ||
              !epi_chunks_typed(p.epi, ptr, m - lane, n0, p.N, p.M, stage_buf, 0, chunks, acc)) {
#pragma unroll 1
            for (int c = 0; c < chunks; ++c) {
              uint32_t r[32];
              tmem_ld_32x32b_x32(tb + (uint32_t)(c * 32), r);
              tmem_wait_ld();
              float x[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]);
              for (int cp = cp_first; cp <= cp_last; ++cp) {
                const float4* slot = reinterpret_cast<const float4*>(
                    p.sk_partials + (size_t)(cp * 2 + (int)rank) * SLOT_FLOATS);
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                  const float4 y = __ldcg(&slot[(c * 8 + v) * TC_BM + row_in_cta]);
                  x[4 * v] += y.x;
                  x[4 * v + 1] += y.y;
                  x[4 * v + 2] += y.z;
                  x[4 * v + 3] += y.w;
                }
              }
#pragma unroll
              for (int j = 0; j < 32; ++j) x[j] *= p.epi.alpha;
              epi_finish_row32_float(p.epi, ptr, m, row_ok, n0 + c * 32, p.N, x, stage_buf, p.M);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (leader) mbar_arrive(tempty_bar(buf));
            else mbar_arrive_cluster(mapa_shared(tempty_bar(buf), pair_leader));
          }
        }
        ++acc_it;
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  cluster_sync();       // neither CTA leaves while the other may still signal it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, PAIR_TMEM_COLS);
}

template <bool INT_MODE, bool A_MN, bool B_MN, bool XF>
int max_clusters_for(int device) {
  static int cached[64] = {};
  if (device < 0 || device >= 64) return 0;
  if (cached[device] > 0) return cached[device];
  if (cudaFuncSetAttribute(tc_pair_gemm_kernel<INT_MODE, A_MN, B_MN, XF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)PAIR_SMEM) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 256, 1, 1);
  cfg.blockDim = dim3(PairThreads<INT_MODE, XF>::THREADS, 1, 1);
  cfg.dynamicSmemBytes = PAIR_SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc_pair_gemm_kernel<INT_MODE, A_MN, B_MN, XF>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cached[device] = n;
  return n;
}

template <bool INT_MODE, bool A_MN, bool B_MN, bool XF>
cudaError_t launch_mode(const TcParams& p, int clusters, cudaStream_t stream) {
  static_assert(PAIR_SMEM <= 232448, "shared memory budget");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool configured[64] = {};
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(tc_pair_gemm_kernel<INT_MODE, A_MN, B_MN, XF>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PAIR_SMEM);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  if (clusters <= 0) return cudaErrorInvalidValue;
  // A programmatic dependent of the previous kernel (its prologue overlaps that
  // kernel's end) -- unless the stream-K tail is on: its CTA pairs wait for each
  // other, so they must all start together on an otherwise free GPU.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(PairThreads<INT_MODE, XF>::THREADS, 1, 1);
  cfg.dynamicSmemBytes = PAIR_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = p.sk_first_tile == p.num_tiles ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_pair_gemm_kernel<INT_MODE, A_MN, B_MN, XF>, p);
}

}  // namespace

int tc_pair_stages() { return PAIR_STAGES; }
int tc_pair_k_per_stage() { return PAIR_SLABS * TC_BK; }
size_t tc_pair_smem_bytes() { return PAIR_SMEM; }

int tc_pair_max_clusters(int device) {
  // Every instantiation has the same shared memory; the thread counts differ by mode.
  const int a = max_clusters_for<false, false, false, false>(device);
  const int b = max_clusters_for<true, false, false, false>(device);
  const int c = max_clusters_for<false, false, false, true>(device);
  return std::min(a, std::min(b, c));
}

template <bool INT_MODE, bool XF>
cudaError_t launch_layouts(const TcParams& p, int clusters, cudaStream_t stream) {
  if (p.a_mn_major)
    return p.b_mn_major ? launch_mode<INT_MODE, true, true, XF>(p, clusters, stream)
                        : launch_mode<INT_MODE, true, false, XF>(p, clusters, stream);
  return p.b_mn_major ? launch_mode<INT_MODE, false, true, XF>(p, clusters, stream)
                      : launch_mode<INT_MODE, false, false, XF>(p, clusters, stream);
}

cudaError_t launch_tc_pair(const TcParams& p, int clusters, cudaStream_t stream) {
  if (p.chunk_kb > 0) return p.xf.a_on || p.xf.b_on ? cudaErrorInvalidValue : launch_layouts<true, false>(p, clusters, stream);
  // Operand transforms run in their own instance (four more warps), and without
  // the stream-K tail (the host turns it off for them).
  if (p.xf.a_on || p.xf.b_on)
    return p.sk_first_tile < p.num_tiles ? cudaErrorInvalidValue : launch_layouts<false, true>(p, clusters, stream);
  return launch_layouts<false, false>(p, clusters, stream);
}

}  // namespace gemmlib

// gemm_api.cu -- the C ABI of libgemm.so (declared in include/gemm.h):
// argument validation, the tile-shape selector, TMA tensor-map encoding, plan
// state and kernel launches.  Host code only; the kernels live in
// tc_kernel.cu and simt_kernels.cu.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <cstdio>
#include <mutex>
#include <new>

#include <nvtx3/nvToolsExt.h>

#include "kernels.h"

using namespace gemmlib;

struct gemm_plan {
  int device = 0;
  gemm_dtype_t ab = GEMM_F16;
  gemm_dtype_t c = GEMM_F32;
  int sm_count = 0;
  int32_t* d_err = nullptr;          // device error word
  void* ws = nullptr;                // int8 staging: fp16 copies of A and B
  size_t ws_bytes = 0;
  void* stage = nullptr;             // gemm_run_host device buffers
  size_t stage_bytes = 0;
  gemm_kernel_t forced = GEMM_KERNEL_AUTO;
  int pair_clusters = 0;             // co-resident CTA-pair clusters (0: pair kernel unavailable)
  void* sk_ws = nullptr;             // stream-K partial accumulators and flags (per cluster and CTA)
  size_t sk_ws_bytes = 0;
  int32_t sk_epoch = 0;
  // Stream-K of the single-CTA kernel: two fp32 partial slots per CTA, then one
  // arrival counter per tile (zero between launches; each tile's last arriver
  // resets its counter).
  void* sk1_ws = nullptr;
  size_t sk1_ws_bytes = 0;
  gemm_config_t last{};
  uint64_t timeout_ns = 4000000000ull;
  // gemm_run_host's row-panel pipeline: copy-in and copy-out streams and the
  // events that order them with the caller's stream (created on first use).
  cudaStream_t host_in = nullptr, host_out = nullptr;
  cudaEvent_t host_ev[36] = {};
  bool host_pipe = false;
};

namespace {

constexpr int64_t kMaxDim = 0x7fffffffLL;   // tile indices and TMA coordinates are 32-bit
constexpr int kHostMaxPanels = 16;           // gemm_run_host: most row panels of its copy pipeline

// NVTX range around a public entry point (a profiler's timeline shows each call;
// without a tool attached a push or pop costs a predictable branch).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// GEMM_LOG=1: every launch prints the configuration it runs to stderr.
bool log_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("GEMM_LOG");
    return v != nullptr && std::atoi(v) != 0;
  }();
  return on;
}

const char* kernel_label(int k) {
  switch (k) {
    case GEMM_KERNEL_NONE: return "none";
    case GEMM_KERNEL_TC: return "tc";
    case GEMM_KERNEL_TC_INT8: return "tc_int8";
    case GEMM_KERNEL_FFMA: return "ffma";
    case GEMM_KERNEL_SIMT: return "simt";
    case GEMM_KERNEL_TC_PAIR: return "tc_pair";
    case GEMM_KERNEL_DIAG: return "diag";
    default: return "?";
  }
}

void log_config(const char* entry, int64_t M, int64_t N, int64_t K, int64_t batch, const gemm_config_t& c) {
  if (!log_enabled()) return;
  std::fprintf(stderr,
               "gemm: %s M=%lld N=%lld K=%lld batch=%lld kernel=%s tile=%dx%dx%d stages=%d cta_group=%d grid=%d "
               "tiles=%d split_k=%d sk_tiles=%d half_tiles=%d k_chunk=%d xf_staged=%d\n",
               entry, (long long)M, (long long)N, (long long)K, (long long)batch, kernel_label(c.kernel), c.bm, c.bn,
               c.bk, c.stages, c.cta_group, c.grid, c.tiles, c.split_k, c.sk_tiles, c.half_tiles, c.k_chunk,
               c.xf_staged);
}

bool is_f16ish(int t) { return t == GEMM_F16 || t == GEMM_BF16; }
bool is_float_out(int t) { return t == GEMM_F32 || t == GEMM_F16 || t == GEMM_BF16; }

gemm_status_t check_types(gemm_dtype_t ab, gemm_dtype_t c) {
  switch (ab) {
    case GEMM_F16:
    case GEMM_BF16: return is_float_out(c) ? GEMM_OK : GEMM_ERR_INVALID_ARG;
    case GEMM_S8: return c == GEMM_S32 ? GEMM_OK : GEMM_ERR_INVALID_ARG;
    case GEMM_F32: return c == GEMM_F32 ? GEMM_OK : GEMM_ERR_INVALID_ARG;
    default: return GEMM_ERR_INVALID_ARG;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Can TMA describe this operand (16-byte aligned base, 16-byte multiple row pitch)?
bool tma_ok(const void* p, int64_t ld, int esize) {
  return aligned16(p) && ((ld * esize) % 16) == 0 && ld * esize < (int64_t(1) << 40);
}

// Storage extent (elements) of a rows x cols logical matrix in a layout.
int64_t storage_elems(gemm_layout_t layout, int64_t rows, int64_t cols, int64_t ld) {
  if (rows == 0 || cols == 0) return 0;
  return layout == GEMM_OP_T ? (rows - 1) * ld + cols : (cols - 1) * ld + rows;
}

bool integral_int32(double v) {
  return std::isfinite(v) && v == std::floor(v) && v >= -2147483648.0 && v <= 2147483647.0;
}

gemm_dtype_t out_dtype_of(gemm_dtype_t c, const gemm_epilogue_t* epi) {
  return epi ? epi->out_dtype : c;
}

gemm_status_t validate(gemm_dtype_t ab, gemm_dtype_t c, gemm_layout_t la, gemm_layout_t lb, int64_t M,
                       int64_t N, int64_t K, double alpha, const void* A, int64_t lda, const void* B,
                       int64_t ldb, double beta, const void* C, int64_t ldc, const void* D, int64_t ldd,
                       const gemm_epilogue_t* epi) {
  gemm_status_t s = check_types(ab, c);
  if (s != GEMM_OK) return s;
  if ((la != GEMM_OP_N && la != GEMM_OP_T) || (lb != GEMM_OP_N && lb != GEMM_OP_T)) return GEMM_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return GEMM_ERR_UNSUPPORTED;
  const gemm_dtype_t out = out_dtype_of(c, epi);
  if (ab == GEMM_S8 ? (out != GEMM_S32 && out != GEMM_S8) : !is_float_out(out)) return GEMM_ERR_INVALID_ARG;
  if (out == GEMM_S8 && !std::isfinite(epi->out_scale)) return GEMM_ERR_INVALID_ARG;
  if (epi) {
    if (epi->act != GEMM_ACT_NONE && epi->act != GEMM_ACT_RELU) return GEMM_ERR_INVALID_ARG;
    if (epi->c_act != GEMM_ACT_NONE && epi->c_act != GEMM_ACT_RELU) return GEMM_ERR_INVALID_ARG;
    if (epi->bias_mode != GEMM_BIAS_NONE && epi->bias_mode != GEMM_BIAS_COL &&
        epi->bias_mode != GEMM_BIAS_ROW)
      return GEMM_ERR_INVALID_ARG;
    if (epi->bias_mode != GEMM_BIAS_NONE) {
      if (!epi->bias) return GEMM_ERR_INVALID_ARG;
      if (ab == GEMM_S8 ? epi->bias_dtype != GEMM_S32 : !is_float_out(epi->bias_dtype))
        return GEMM_ERR_INVALID_ARG;
    }
    // Operand transforms: only the two operand bits, known activations, finite
    // scales; int8 operands take the activation alone.
    if (epi->load_xf & ~(GEMM_XF_A | GEMM_XF_B)) return GEMM_ERR_INVALID_ARG;
    const struct { uint32_t bit; gemm_act_t act; float scale; } ops[2] = {
        {GEMM_XF_A, epi->a_act, epi->a_scale}, {GEMM_XF_B, epi->b_act, epi->b_scale}};
    for (const auto& o : ops) {
      if (!(epi->load_xf & o.bit)) continue;
      if (o.act != GEMM_ACT_NONE && o.act != GEMM_ACT_RELU) return GEMM_ERR_INVALID_ARG;
      if (!std::isfinite(o.scale)) return GEMM_ERR_INVALID_ARG;
      if (ab == GEMM_S8 && o.scale != 1.0f) return GEMM_ERR_UNSUPPORTED;
    }
  }
  if (ab == GEMM_S8 && (!integral_int32(alpha) || !integral_int32(beta))) return GEMM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return GEMM_OK;
  if (!D || ldd < N) return GEMM_ERR_INVALID_ARG;
  if (K > 0) {
    if (!A || !B) return GEMM_ERR_INVALID_ARG;
    if (lda < std::max<int64_t>(1, la == GEMM_OP_N ? M : K)) return GEMM_ERR_INVALID_ARG;
    if (ldb < std::max<int64_t>(1, lb == GEMM_OP_N ? K : N)) return GEMM_ERR_INVALID_ARG;
  }
  if (beta != 0.0) {
    if (!C || ldc < N) return GEMM_ERR_INVALID_ARG;
    if (C == D && (ldc != ldd || c != out)) return GEMM_ERR_INVALID_ARG;
  }
  return GEMM_OK;
}

// Relative cost of one 128 x BN tile of the tensor-core kernel (a 128x128 tile
// does half the MMA work of a 128x256 tile but keeps the fixed per-tile costs).
// Relative time per K block of a 128 x bn single-CTA tile (measured: 4096^3 and
// 1024^3 fp16 for 256 and 128; 64 from 1024^3 and the skinny 16384 x 64 x 16384).
double tc_tile_cost(int bn) { return bn == 256 ? 1.0 : bn == 128 ? 0.77 : 0.6; }

// Run a tensor-core problem on CTA pairs?  Both dimensions must exceed one
// 128-wide tile.  Then the choice is the smaller estimated time:
//   waves x max(mainloop of a tile, its epilogue) + fixed cost per launch,
// with a tile's mainloop = K/64 blocks x a per-block time.  Fitted to fp16 runs
// from 256^3 to 8192^3 and two batches: per 64-deep block 0.323 us for a
// 256 x 256 pair tile and 0.397 us for a 128 x 256 single-CTA tile (0.77 of that
// for 128 x 128); epilogues of ~4.4 us (pair tile) and ~3.3 us (single-CTA
// tile) bound tiles of small K; fixed costs ~8.3 us and ~5.0 us (the single-CTA
// kernel's eight-warp epilogue finishes its last tile sooner).  The stream-K
// tail, when requested, spreads pair tiles over all pairs.
// GEMM_TC_CTA_GROUP=1 never uses pairs; =2 uses them whenever both dimensions allow.
// Tail halves of the CTA-pair kernel: T tiles over G pairs leave a last wave of
// r = T mod G tiles.  When 2r <= G those r tiles run as 2r units of 256 x 128
// (half the columns, half the MMA work each), one per pair, so the last wave
// takes half a tile's time.  Returns the number of tiles so split (0: none).
// GEMM_TC_TAIL_HALVES=0 turns it off.
int64_t pair_tail_halves(int64_t T, int64_t G) {
  if (G <= 0) return 0;
  if (const char* env = std::getenv("GEMM_TC_TAIL_HALVES"))
    if (std::atoi(env) == 0) return 0;
  const int64_t r = T % G;
  return (r > 0 && 2 * r <= G) ? r : 0;
}

// Single-CTA stream-K (floating mode) for T tiles of KB K blocks on sm_count
// SMs: publishing a partial, the fence and the last arrival's reads cost ~4 us,
// about 20 K blocks of a 128 x 128 tile, so it is taken when the idle SMs of a
// single partial wave would save at least 48 K blocks per CTA, and every CTA gets
// at least 4.
bool single_stream_k_pays(int64_t T, int64_t KB, int sm_count) {
  return T < sm_count && (double)KB * (1.0 - (double)T / sm_count) >= 48.0 && T * KB >= 4 * (int64_t)sm_count;
}

bool use_pairs(int64_t M, int64_t N, int64_t K, int64_t batch, int pair_clusters, int sm_count) {
  if (pair_clusters <= 0 || M <= 128 || N <= 128) return false;
  if (const char* env = std::getenv("GEMM_TC_CTA_GROUP")) {
    const int v = std::atoi(env);
    if (v == 1) return false;
    if (v == 2) return true;
  }
  if (const char* sk = std::getenv("GEMM_STREAM_K"))
    if (std::atoi(sk) != 0) return true;
  const double kb = (double)((K + 63) / 64);
  const int64_t pair_tiles = batch * ((M + 255) / 256) * ((N + 255) / 256);
  // A split tail wave costs about half a tile; the estimate counts it only behind
  // at least one whole wave (single partial waves are where the time model's
  // fixed costs were calibrated, and the kernel's own choice between halves and
  // whole tiles does not change which kernel is faster there).
  const double tail = pair_tiles % pair_clusters == 0 ? 0.0
                      : (pair_tiles >= pair_clusters && pair_tail_halves(pair_tiles, pair_clusters) > 0) ? 0.5
                                                                                                          : 1.0;
  const double t_pair =
      ((double)(pair_tiles / pair_clusters) + tail) * std::max(kb * 0.323, 4.4) + 8.3;
  double t_one = 1e300;
  for (int bn : {256, 128, 64}) {
    const int64_t tiles = batch * ((M + 127) / 128) * ((N + bn - 1) / bn);
    const double per_tile = std::max(kb * 0.397 * tc_tile_cost(bn), 3.3 * (bn / 256.0));
    t_one = std::min(t_one, (double)((tiles + sm_count - 1) / sm_count) * per_tile + 5.0);
  }
  return t_pair < t_one;
}

// pair_clusters: co-resident clusters of two CTAs for the CTA-pair kernel on the
// target device (0: that kernel is not considered unless forced).
gemm_status_t select_config(gemm_dtype_t ab, gemm_dtype_t c, gemm_layout_t la, gemm_layout_t lb, int64_t M,
                            int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                            int sm_count, gemm_kernel_t forced, gemm_config_t* out, int pair_clusters = 0,
                            int64_t batch = 1, bool xf = false) {
  // xf: operand transforms are requested; their kernel instances run whole tiles
  // (no stream-K).
  (void)c;
  gemm_config_t cfg{};
  cfg.split_k = 1;
  cfg.cta_group = 1;
  cfg.cluster = 1;
  if (sm_count <= 0) sm_count = 1;
  if (M == 0 || N == 0) {
    cfg.kernel = GEMM_KERNEL_NONE;
    *out = cfg;
    return GEMM_OK;
  }
  // Which kernels could serve this request?
  const bool tc_ok = K > 0 && is_f16ish(ab) && tma_ok(A, lda, 2) && tma_ok(B, ldb, 2);
  const bool int8_ok = K > 0 && ab == GEMM_S8 && (lda % 8) == 0 && (ldb % 8) == 0;
  const bool ffma_ok = K > 0 && ab == GEMM_F32 && aligned16(A) && aligned16(B) && (lda % 4) == 0 &&
                       (ldb % 4) == 0;
  gemm_kernel_t k;
  if (forced != GEMM_KERNEL_AUTO) {
    k = forced;
    bool type_ok = true, feasible = true;
    switch (forced) {
      case GEMM_KERNEL_TC: type_ok = is_f16ish(ab); feasible = tc_ok; break;
      case GEMM_KERNEL_TC_PAIR: type_ok = is_f16ish(ab); feasible = tc_ok && pair_clusters > 0; break;
      case GEMM_KERNEL_TC_INT8: type_ok = ab == GEMM_S8; feasible = int8_ok; break;
      case GEMM_KERNEL_FFMA: type_ok = ab == GEMM_F32; feasible = ffma_ok; break;
      case GEMM_KERNEL_SIMT: break;
      default: return GEMM_ERR_INVALID_ARG;
    }
    if (!type_ok) return GEMM_ERR_UNSUPPORTED;
    if (!feasible) return K == 0 ? GEMM_ERR_UNSUPPORTED : GEMM_ERR_ALIGNMENT;
  } else {
    k = tc_ok ? GEMM_KERNEL_TC
              : int8_ok ? GEMM_KERNEL_TC_INT8 : ffma_ok ? GEMM_KERNEL_FFMA : GEMM_KERNEL_SIMT;
    // 256 x 256 tiles on CTA pairs move a third fewer operand bytes per SM for the
    // same MMA work, but a pair's fixed cost per launch is higher (~9 us against
    // ~5 us measured) and its tiles are four times larger: below one full wave of
    // pairs the single-CTA kernel's finer grid finishes first.
    if (k == GEMM_KERNEL_TC && use_pairs(M, N, K, batch, pair_clusters, sm_count)) k = GEMM_KERNEL_TC_PAIR;
  }
  (void)la;
  (void)lb;
  cfg.kernel = k;
  switch (k) {
    case GEMM_KERNEL_TC_PAIR: {
      cfg.bm = 2 * TC_BM;
      cfg.bn = 256;
      cfg.bk = tc_pair_k_per_stage();
      cfg.stages = tc_pair_stages();
      cfg.cta_group = 2;
      const int64_t tiles_m = (M + 255) / 256, tiles_n = (N + 255) / 256;
      cfg.tiles = (int32_t)std::min<int64_t>(batch * tiles_m * tiles_n, kMaxDim);
      int raster = 8;
      if (const char* env = std::getenv("GEMM_TC_RASTER")) raster = std::max(1, std::atoi(env));
      cfg.raster = (int32_t)std::min<int64_t>(raster, tiles_m);
      cfg.grid = 2 * (int32_t)std::min<int64_t>(cfg.tiles, pair_clusters);
      // Stream-K tail (opt-in, GEMM_STREAM_K=1): when the tiles leave the last
      // wave of CTA pairs partly idle, the K blocks of the last (G + T mod G)
      // tiles -- or of all tiles when there are fewer than G -- are shared out
      // evenly over all G pairs.  Off by default: on GB300 the fixup of split
      // tiles cost more than the idle tail it recovers in every measured shape
      // (the chip runs power-capped under load, so idle SMs in a tail wave let
      // the busy ones clock higher).
      const int64_t T = cfg.tiles, G = pair_clusters, KB = (K + TC_BK - 1) / TC_BK;
      const int64_t q = T / G, r = T % G;
      bool sk = r != 0 && (double)r / (double)G < 0.9;
      int64_t sk_tiles = q >= 1 ? G + r : T;
      if (sk_tiles * KB < 8 * G) sk = false;          // too little K work per pair
      const char* sk_env = std::getenv("GEMM_STREAM_K");
      sk = sk && sk_env != nullptr && std::atoi(sk_env) != 0 && !xf;
      if (sk) {
        cfg.sk_tiles = (int32_t)sk_tiles;
        cfg.grid = 2 * (int32_t)G;
        const int64_t per = std::max<int64_t>(1, sk_tiles * KB / G);
        cfg.split_k = (int32_t)std::min<int64_t>((KB + per - 1) / per + 1, KB);
      }
      cfg.cluster = 2;
      if (!sk) {
        cfg.half_tiles = (int32_t)pair_tail_halves(T, G);
        if (cfg.half_tiles > 0) cfg.grid = 2 * (int32_t)std::min<int64_t>(T + cfg.half_tiles, G);
      }
      break;
    }
    case GEMM_KERNEL_TC:
    case GEMM_KERNEL_TC_INT8: {
      int bn = 128;
      if (k == GEMM_KERNEL_TC) {
        // Pick the tile width with the smaller estimated makespan over the SMs
        // (the largest tile that fits, unless it leaves SMs idle).
        double best = 1e300;
        for (int cand : {256, 128, 64}) {
          const int64_t tiles = batch * ((M + 127) / 128) * ((N + cand - 1) / cand);
          const int64_t waves = (tiles + sm_count - 1) / sm_count;
          const double cost = (double)waves * tc_tile_cost(cand);
          if (cost < best - 1e-9) { best = cost; bn = cand; }
        }
        // A narrower tile fills more SMs, but a wider one that qualifies for stream-K
        // (deep K on few tiles) keeps every SM busy with less operand traffic.
        const int64_t KB = (K + TC_BK - 1) / TC_BK;
        auto tiles_of = [&](int w) { return batch * ((M + 127) / 128) * ((N + w - 1) / w); };
        if (!xf && !single_stream_k_pays(tiles_of(bn), KB, sm_count)) {
          for (int cand : {128, 256})
            if (cand > bn && single_stream_k_pays(tiles_of(cand), KB, sm_count)) {
              bn = cand;
              break;
            }
        }
        // Tuning override: GEMM_TC_BN=64, 128 or 256 fixes the tile width.
        if (const char* env = std::getenv("GEMM_TC_BN")) {
          const int v = std::atoi(env);
          if (v == 64 || v == 128 || v == 256) bn = v;
        }
      }
      cfg.bm = TC_BM;
      cfg.bn = bn;
      cfg.bk = tc_k_per_stage(bn);
      cfg.stages = tc_stages(bn);
      const int64_t tiles_m = (M + 127) / 128, tiles_n = (N + bn - 1) / bn;
      cfg.tiles = (int32_t)std::min<int64_t>(batch * tiles_m * tiles_n, kMaxDim);
      cfg.raster = (int32_t)std::min<int64_t>(16, tiles_m);
      cfg.grid = (int32_t)std::min<int64_t>(cfg.tiles, sm_count);
      // Exact int8 chunk: |sum of 1024 products| <= 1024 * 2^14 = 2^24, and every
      // integer of that size is exact in fp32.  (GEMM_INT8_CHUNK=512 halves it.)
      int chunk = 1024;
      if (const char* env = std::getenv("GEMM_INT8_CHUNK")) {
        if (std::atoi(env) == 512) chunk = 512;
      }
      cfg.k_chunk = k == GEMM_KERNEL_TC_INT8 ? chunk : 0;
      // Stream-K for a wave that leaves SMs idle (floating mode): all CTAs share
      // the tiles' K blocks evenly and the last arrival on a tile finishes it
      // (single_stream_k_pays); GEMM_TC_SPLITK=0 turns it off, =1 forces it when
      // every CTA gets a K block.
      if (k == GEMM_KERNEL_TC) {
        const int64_t T = cfg.tiles, KB = (K + TC_BK - 1) / TC_BK;
        bool sk1 = single_stream_k_pays(T, KB, sm_count);
        if (const char* env = std::getenv("GEMM_TC_SPLITK")) {
          const int v = std::atoi(env);
          if (v == 0) sk1 = false;
          else if (v == 1) sk1 = T * KB >= sm_count;
        }
        if (xf) sk1 = false;
        if (sk1) {
          cfg.sk_tiles = (int32_t)T;
          cfg.grid = sm_count;
          const int64_t per = std::max<int64_t>(1, T * KB / sm_count);
          cfg.split_k = (int32_t)std::min<int64_t>((KB + per - 1) / per + 1, KB);
        }
      }
      const bool pair_int = k == GEMM_KERNEL_TC_INT8 && use_pairs(M, N, K, batch, pair_clusters, sm_count);
      if (pair_int) {   // exact integer mode on CTA pairs: 256 x 256 tiles
        cfg.bm = 2 * TC_BM;
        cfg.bn = 256;
        cfg.bk = tc_pair_k_per_stage();
        cfg.stages = tc_pair_stages();
        cfg.cta_group = 2;
        const int64_t ptm = (M + 255) / 256, ptn = (N + 255) / 256;
        cfg.tiles = (int32_t)std::min<int64_t>(batch * ptm * ptn, kMaxDim);
        cfg.raster = (int32_t)std::min<int64_t>(8, ptm);
        cfg.grid = 2 * (int32_t)std::min<int64_t>(cfg.tiles, pair_clusters);
        cfg.cluster = 2;
      }
      break;
    }
    case GEMM_KERNEL_FFMA: {
      cfg.bm = FFMA_BM;
      cfg.bn = FFMA_BN;
      cfg.bk = FFMA_BK;
      cfg.stages = 2;
      const int64_t tiles = batch * ((M + FFMA_BM - 1) / FFMA_BM) * ((N + FFMA_BN - 1) / FFMA_BN);
      cfg.tiles = (int32_t)std::min<int64_t>(tiles, kMaxDim);
      cfg.grid = cfg.tiles;
      cfg.raster = 1;
      // A last wave of CTAs at most half full (single problems): its tiles are
      // split over K, and a reduction pass finishes them (GEMM_FFMA_TAIL=0: off).
      int split = 0;
      int64_t tail = batch == 1 ? ffma_tail_split(tiles, K, sm_count, &split) : 0;
      if (const char* env = std::getenv("GEMM_FFMA_TAIL"))
        if (std::atoi(env) == 0) tail = 0;
      if (tail > 0) {
        cfg.sk_tiles = (int32_t)tail;
        cfg.split_k = split;
        cfg.grid = (int32_t)(tiles - tail + tail * split);
      }
      break;
    }
    default: {  // SIMT
      cfg.bm = 16;
      cfg.bn = 16;
      cfg.bk = 16;
      cfg.stages = 1;
      const int64_t tiles = batch * ((M + 15) / 16) * ((N + 15) / 16);
      cfg.tiles = (int32_t)std::min<int64_t>(tiles, kMaxDim);
      cfg.grid = cfg.tiles;
      cfg.raster = 1;
      break;
    }
  }
  *out = cfg;
  return GEMM_OK;
}

// --------------------------- TMA tensor maps -------------------------------

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// A row-pitched tensor of 16-bit elements (inner elements contiguous, `ld`
// elements between rows of the outer dimension) with a third, outermost
// dimension: `nbatch` problems `bstride` elements apart (one problem when
// nbatch == 1).  128-byte swizzle; out-of-bounds elements read as zero.
bool encode_3d(CUtensorMap* tm, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t outer,
               uint64_t ld, uint64_t nbatch, uint64_t bstride, uint32_t box_inner, uint32_t box_outer) {
  if (!encode_fn()) return false;
  if (nbatch <= 1) {
    nbatch = 1;
    bstride = (ld * outer + 7) / 8 * 8;   // unused; any 16-byte multiple past the problem
  }
  cuuint64_t dims[3] = {inner, outer, nbatch};
  cuuint64_t strides[2] = {ld * 2, bstride * 2};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(tm, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A strided batch of independent problems (count 1: one problem).
struct Batch {
  int64_t count = 1;
  int64_t sa = 0, sb = 0, sc = 0, sd = 0, sbias = 0;   // element strides (0: shared by all)
};

// tcgen05 instruction descriptor, kind::f16 with fp32 accumulation:
//   bits 4-5 D format (1 = f32), 7-9 A format, 10-12 B format (0 = f16, 1 = bf16),
//   15 / 16 A / B MN-major, 17-22 N >> 3, 24-28 M >> 4.
uint32_t make_idesc(bool bf16, int bn, bool a_mn_major, bool b_mn_major, int bm = TC_BM) {
  const uint32_t f = bf16 ? 1u : 0u;
  return (1u << 4) | (f << 7) | (f << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(bm >> 4) << 24);
}

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

EpiParams make_epi(const gemm_plan* plan, double alpha, double beta, const void* C, int64_t ldc, void* D,
                   int64_t ldd, const gemm_epilogue_t* epi) {
  EpiParams e{};
  const gemm_dtype_t out = out_dtype_of(plan->c, epi);
  e.alpha = (float)alpha;
  e.beta = (float)beta;
  if (plan->ab == GEMM_S8) {
    e.alpha_i = (int32_t)alpha;
    e.beta_i = (int32_t)beta;
  }
  e.read_c = beta != 0.0 ? 1 : 0;
  e.C = e.read_c ? C : nullptr;
  e.ldc = ldc;
  e.c_dtype = plan->c;
  e.D = D;
  e.ldd = ldd;
  e.d_dtype = out;
  e.bias = (epi && epi->bias_mode != GEMM_BIAS_NONE) ? epi->bias : nullptr;
  e.bias_dtype = epi ? epi->bias_dtype : GEMM_F32;
  e.bias_mode = epi ? epi->bias_mode : GEMM_BIAS_NONE;
  e.relu = (epi && epi->act == GEMM_ACT_RELU) ? 1 : 0;
  e.c_relu = (epi && epi->c_act == GEMM_ACT_RELU) ? 1 : 0;
  e.out_scale = epi ? epi->out_scale : 1.0f;
  e.vec_c = (e.read_c && aligned16(C) && (ldc * dtype_bytes(plan->c)) % 16 == 0) ? 1 : 0;
  e.vec_d = (aligned16(D) && (ldd * dtype_bytes(out)) % 16 == 0) ? 1 : 0;
  return e;
}

// The kernels' view of the operand transforms; an identity transform (no
// activation, scale 1) is dropped, so it costs nothing.
// How the tensor-core kernels transform a pair of 16-bit elements: bf16 through
// fp32; fp16 with a scale that fp16 holds exactly in fp16 arithmetic (the
// product of two fp16 values is exact in fp32, so one fp16 rounding equals the
// fp32 product rounded to fp16); any other fp16 scale through fp32.
int xf_kind(gemm_dtype_t ab, float scale, uint32_t* scale2) {
  *scale2 = 0;
  if (ab == GEMM_BF16) return XF_BF16;
  const __half h = __float2half_rn(scale);
  if (__half2float(h) != scale) return XF_F16_F32;
  const uint16_t bits = *reinterpret_cast<const uint16_t*>(&h);
  *scale2 = (uint32_t)bits | ((uint32_t)bits << 16);
  return XF_F16_PACKED;
}

LoadXf make_xf(gemm_dtype_t ab, const gemm_epilogue_t* epi) {
  LoadXf x{};
  x.a_scale = x.b_scale = 1.0f;
  if (!epi) return x;
  if ((epi->load_xf & GEMM_XF_A) && (epi->a_act == GEMM_ACT_RELU || epi->a_scale != 1.0f)) {
    x.a_on = 1;
    x.a_relu = epi->a_act == GEMM_ACT_RELU ? 1 : 0;
    x.a_scale = epi->a_scale;
  }
  if ((epi->load_xf & GEMM_XF_B) && (epi->b_act == GEMM_ACT_RELU || epi->b_scale != 1.0f)) {
    x.b_on = 1;
    x.b_relu = epi->b_act == GEMM_ACT_RELU ? 1 : 0;
    x.b_scale = epi->b_scale;
  }
  x.a_kind = xf_kind(ab, x.a_scale, &x.a_scale2);
  x.b_kind = xf_kind(ab, x.b_scale, &x.b_scale2);
  return x;
}

bool xf_any(const gemm_epilogue_t* epi) {
  const LoadXf x = make_xf(GEMM_F16, epi);
  return x.a_on || x.b_on;
}

gemm_status_t ensure_ws(gemm_plan* plan, size_t bytes, cudaStream_t stream) {
  if (plan->ws_bytes >= bytes) return GEMM_OK;
  if (plan->ws) {
    cudaFreeAsync(plan->ws, stream);
    plan->ws = nullptr;
    plan->ws_bytes = 0;
  }
  void* p = nullptr;
  if (cudaMallocAsync(&p, bytes, stream) != cudaSuccess) return GEMM_ERR_CUDA;
  plan->ws = p;
  plan->ws_bytes = bytes;
  return GEMM_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

gemm_status_t launch_tc_problem(gemm_plan* plan, const gemm_config_t& cfg, gemm_layout_t la, gemm_layout_t lb,
                                int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                                int64_t ldb, CUtensorMapDataType dt, bool bf16, const EpiParams& epi,
                                int chunk_kb, cudaStream_t stream, const Batch& bt = Batch(),
                                const LoadXf& xf = LoadXf{}) {
  TcParams tp;
  std::memset(&tp, 0, sizeof(tp));
  const int bn = cfg.bn;
  const bool a_mn = la == GEMM_OP_N, b_mn = lb == GEMM_OP_T;
  const uint64_t na = (bt.count > 1 && bt.sa != 0) ? (uint64_t)bt.count : 1;
  const uint64_t nb = (bt.count > 1 && bt.sb != 0) ? (uint64_t)bt.count : 1;
  bool ok;
  // A: K-major (row-major A) boxes 64(K) x 128(M); M-major boxes 64(M) x 64(K).
  if (!a_mn) ok = encode_3d(&tp.tmA, dt, A, (uint64_t)K, (uint64_t)M, (uint64_t)lda, na, bt.sa, TC_BK, TC_BM);
  else ok = encode_3d(&tp.tmA, dt, A, (uint64_t)M, (uint64_t)K, (uint64_t)lda, na, bt.sa, 64, TC_BK);
  if (!ok) return GEMM_ERR_CUDA;
  // B: K-major (column-major B) boxes 64(K) x BN(N); N-major boxes 64(N) x 64(K).
  if (!b_mn) ok = encode_3d(&tp.tmB, dt, B, (uint64_t)K, (uint64_t)N, (uint64_t)ldb, nb, bt.sb, TC_BK, (uint32_t)bn);
  else ok = encode_3d(&tp.tmB, dt, B, (uint64_t)N, (uint64_t)K, (uint64_t)ldb, nb, bt.sb, 64, TC_BK);
  if (!ok) return GEMM_ERR_CUDA;
  tp.M = (int32_t)M;
  tp.N = (int32_t)N;
  tp.K = (int32_t)K;
  tp.num_kb = (int32_t)((K + TC_BK - 1) / TC_BK);
  tp.tiles_m = (int32_t)((M + TC_BM - 1) / TC_BM);
  tp.tiles_n = (int32_t)((N + bn - 1) / bn);
  tp.tiles_per_batch = tp.tiles_m * tp.tiles_n;
  tp.num_tiles = tp.tiles_per_batch * (int32_t)bt.count;
  tp.a_batched = na > 1;
  tp.b_batched = nb > 1;
  tp.raster = cfg.raster > 0 ? cfg.raster : 1;
  tp.a_mn_major = a_mn ? 1 : 0;
  tp.b_mn_major = b_mn ? 1 : 0;
  tp.idesc = make_idesc(bf16, bn, a_mn, b_mn);
  tp.chunk_kb = chunk_kb;
  tp.xf = xf;
  tp.epi = epi;
  tp.err = plan->d_err;
  tp.timeout_ns = plan->timeout_ns;
  tp.sk_first_tile = tp.num_tiles;
  if (cfg.sk_tiles > 0 && chunk_kb == 0) {
    // Stream-K over the last sk_tiles tiles: two 128 x bn fp32 partial slots per
    // CTA, then one arrival counter per tile.
    const size_t part_bytes = (size_t)cfg.grid * 2 * TC_BM * (size_t)bn * sizeof(float);
    const size_t need = part_bytes + (size_t)tp.num_tiles * sizeof(int32_t);
    if (plan->sk1_ws_bytes < need) {
      if (plan->sk1_ws) cudaFreeAsync(plan->sk1_ws, stream);
      plan->sk1_ws = nullptr;
      plan->sk1_ws_bytes = 0;
      if (cudaMallocAsync(&plan->sk1_ws, need, stream) != cudaSuccess) return GEMM_ERR_CUDA;
      if (cudaMemsetAsync(plan->sk1_ws, 0, need, stream) != cudaSuccess) return GEMM_ERR_CUDA;
      plan->sk1_ws_bytes = need;
    }
    tp.sk_first_tile = tp.num_tiles - std::min<int32_t>(cfg.sk_tiles, tp.num_tiles);
    tp.sk_partials = static_cast<float*>(plan->sk1_ws);
    tp.sk_flags = reinterpret_cast<int32_t*>(static_cast<char*>(plan->sk1_ws) + part_bytes);
  }
  // K rotation for a single tile column (whole floating tiles only; GEMM_TC_KROT=0 off).
  tp.k_rotate = (tp.tiles_n == 1 && tp.tiles_m > 1 && chunk_kb == 0 && tp.sk_first_tile == tp.num_tiles) ? 1 : 0;
  if (const char* env = std::getenv("GEMM_TC_KROT"))
    if (std::atoi(env) == 0) tp.k_rotate = 0;
  return launch_tc(tp, bn, cfg.grid, stream) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

// A 2-D tensor map with elements of `es` bytes, 128-byte swizzle (the
// diagonal kernel's boxes: 128-byte inner extent).
bool encode_2d(CUtensorMap* tm, CUtensorMapDataType dt, int es, const void* ptr, uint64_t inner, uint64_t outer,
               uint64_t ld, uint32_t box_inner, uint32_t box_outer) {
  if (!encode_fn()) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * (uint64_t)es};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(tm, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A 1-D tensor map over a vector of n elements, boxes of `box` elements.
bool encode_1d(CUtensorMap* tm, CUtensorMapDataType dt, const void* ptr, uint64_t n, uint32_t box) {
  if (!encode_fn()) return false;
  cuuint64_t dims[1] = {n};
  cuuint64_t strides[1] = {0};   // unused for rank 1
  cuuint32_t boxd[1] = {box};
  cuuint32_t estr[1] = {1};
  CUresult r = g_encode(tm, dt, 1, const_cast<void*>(ptr), dims, strides, boxd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

CUtensorMapDataType tma_dtype(gemm_dtype_t t) {
  return t == GEMM_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                       : t == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// The CTA-pair kernel: each CTA of a pair loads 128 rows of A and 128 columns
// of B per K block, so both tensor maps use 128-row (K-major) or 64 x 64
// (MN-major) boxes; the MMA instruction covers M = 256, N = 256.
gemm_status_t launch_pair_problem(gemm_plan* plan, const gemm_config_t& cfg, gemm_layout_t la, gemm_layout_t lb,
                                  int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                                  int64_t ldb, bool bf16, const EpiParams& epi, cudaStream_t stream,
                                  int chunk_kb = 0, const Batch& bt = Batch(), const LoadXf& xf = LoadXf{}) {
  TcParams tp;
  std::memset(&tp, 0, sizeof(tp));
  const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const bool a_mn = la == GEMM_OP_N, b_mn = lb == GEMM_OP_T;
  const uint64_t na = (bt.count > 1 && bt.sa != 0) ? (uint64_t)bt.count : 1;
  const uint64_t nb = (bt.count > 1 && bt.sb != 0) ? (uint64_t)bt.count : 1;
  bool ok;
  // MN-major operands: boxes of 64 (MN) x one pipeline stage of K, one per stage.
  const uint32_t kstage = (uint32_t)tc_pair_k_per_stage();
  if (!a_mn) ok = encode_3d(&tp.tmA, dt, A, (uint64_t)K, (uint64_t)M, (uint64_t)lda, na, bt.sa, TC_BK, TC_BM);
  else ok = encode_3d(&tp.tmA, dt, A, (uint64_t)M, (uint64_t)K, (uint64_t)lda, na, bt.sa, 64, kstage);
  if (!ok) return GEMM_ERR_CUDA;
  if (!b_mn) ok = encode_3d(&tp.tmB, dt, B, (uint64_t)K, (uint64_t)N, (uint64_t)ldb, nb, bt.sb, TC_BK, 128);
  else ok = encode_3d(&tp.tmB, dt, B, (uint64_t)N, (uint64_t)K, (uint64_t)ldb, nb, bt.sb, 64, kstage);
  if (!ok) return GEMM_ERR_CUDA;
  // Half-tile units load 64 columns of B per CTA: K-major boxes of 64 rows (an
  // MN-major box is already 64 columns wide).
  const bool halves = cfg.half_tiles > 0 && chunk_kb == 0 && cfg.sk_tiles == 0;
  if (halves && !b_mn) {
    if (!encode_3d(&tp.tmBh, dt, B, (uint64_t)K, (uint64_t)N, (uint64_t)ldb, nb, bt.sb, TC_BK, 64))
      return GEMM_ERR_CUDA;
  } else {
    tp.tmBh = tp.tmB;
  }
  tp.M = (int32_t)M;
  tp.N = (int32_t)N;
  tp.K = (int32_t)K;
  tp.num_kb = (int32_t)((K + TC_BK - 1) / TC_BK);
  tp.tiles_m = (int32_t)((M + 255) / 256);
  tp.tiles_n = (int32_t)((N + 255) / 256);
  tp.tiles_per_batch = tp.tiles_m * tp.tiles_n;
  tp.num_tiles = tp.tiles_per_batch * (int32_t)bt.count;
  tp.a_batched = na > 1;
  tp.b_batched = nb > 1;
  tp.raster = cfg.raster > 0 ? cfg.raster : 1;
  tp.a_mn_major = a_mn ? 1 : 0;
  tp.b_mn_major = b_mn ? 1 : 0;
  tp.idesc = make_idesc(bf16, 256, a_mn, b_mn, 256);
  tp.idesc_half = make_idesc(bf16, 128, a_mn, b_mn, 256);
  tp.chunk_kb = chunk_kb;
  tp.xf = xf;
  tp.epi = epi;
  tp.err = plan->d_err;
  tp.timeout_ns = plan->timeout_ns;
  tp.sk_first_tile = tp.num_tiles;
  tp.half_first_tile = tp.num_tiles;
  if (halves && cfg.half_tiles <= tp.num_tiles) tp.half_first_tile = tp.num_tiles - cfg.half_tiles;
  if (cfg.sk_tiles > 0 && chunk_kb == 0) {
    const int clusters = cfg.grid / 2;
    const size_t part_bytes = (size_t)clusters * 2 * TC_BM * 256 * sizeof(float);
    const size_t need = part_bytes + (size_t)clusters * 2 * sizeof(int32_t);
    if (plan->sk_ws_bytes < need) {
      if (plan->sk_ws) cudaFreeAsync(plan->sk_ws, stream);
      plan->sk_ws = nullptr;
      plan->sk_ws_bytes = 0;
      if (cudaMallocAsync(&plan->sk_ws, need, stream) != cudaSuccess) return GEMM_ERR_CUDA;
      if (cudaMemsetAsync(plan->sk_ws, 0, need, stream) != cudaSuccess) return GEMM_ERR_CUDA;
      plan->sk_ws_bytes = need;
      plan->sk_epoch = 0;
    }
    tp.sk_first_tile = tp.num_tiles - cfg.sk_tiles;
    tp.sk_partials = static_cast<float*>(plan->sk_ws);
    tp.sk_flags = reinterpret_cast<int32_t*>(static_cast<char*>(plan->sk_ws) + part_bytes);
    if (++plan->sk_epoch <= 0) plan->sk_epoch = 1;
    tp.sk_epoch = plan->sk_epoch;
  }
  return launch_tc_pair(tp, cfg.grid / 2, stream) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

// Operand transforms of 16-bit operands on the tensor-core kernels: which
// operands are transformed by a staging pass into plan scratch before the GEMM
// (GEMM_XF_A / GEMM_XF_B bits) rather than in place on the staged tiles inside
// the kernel.  Inside the kernel every tile that reads an element transforms it
// again -- an A element once per tile column, a B element once per tile row --
// and each pass costs shared-memory bandwidth the MMAs need; measured on an
// 8192^3 fp16 GEMM it took the kernel from 0.63 ms to 1.3-1.6 ms, where a
// staging pass costs one read and one write of the operand at HBM speed (~40 us
// for 134 MB).  An operand that only one tile reads (a skinny GEMM's A) is
// transformed inside the kernel (once, and overlapped with its streaming), and
// so is one under 4 MiB, where the extra launch would dominate.
// GEMM_XF_STAGE=0 / 1: never / always stage.
uint32_t xf_stage_mask(gemm_dtype_t ab, const LoadXf& x, const gemm_config_t& cfg, gemm_layout_t la,
                       gemm_layout_t lb, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, const Batch& bt) {
  if (!is_f16ish(ab) || (cfg.kernel != GEMM_KERNEL_TC && cfg.kernel != GEMM_KERNEL_TC_PAIR)) return 0;
  const uint32_t want = (x.a_on ? GEMM_XF_A : 0u) | (x.b_on ? GEMM_XF_B : 0u);
  if (const char* env = std::getenv("GEMM_XF_STAGE")) {
    const int v = std::atoi(env);
    if (v == 0) return 0;
    if (v == 1) return want;
  }
  const int64_t tiles_m = (M + cfg.bm - 1) / cfg.bm, tiles_n = (N + cfg.bn - 1) / cfg.bn;
  const int64_t na = (bt.count > 1 && bt.sa != 0) ? bt.count : 1;
  const int64_t nb = (bt.count > 1 && bt.sb != 0) ? bt.count : 1;
  const int64_t a_bytes = ((na - 1) * bt.sa + storage_elems(la, M, K, lda)) * 2;
  const int64_t b_bytes = ((nb - 1) * bt.sb + storage_elems(lb, K, N, ldb)) * 2;
  constexpr int64_t kMinStage = 4ll << 20;
  uint32_t m = 0;
  if (x.a_on && tiles_n >= 2 && a_bytes >= kMinStage) m |= GEMM_XF_A;
  if (x.b_on && tiles_m >= 2 && b_bytes >= kMinStage) m |= GEMM_XF_B;
  return m;
}

// The selector's configuration for a request with operand transforms `x`: the
// kernel and tile first (as without transforms), then which operands are
// staged; if some transform stays inside the kernel the configuration is
// chosen again for the transform instances (whole tiles, no stream-K).
gemm_status_t select_with_transforms(gemm_dtype_t ab, gemm_dtype_t c, gemm_layout_t la, gemm_layout_t lb, int64_t M,
                                     int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                                     int sm_count, gemm_kernel_t forced, int pair_clusters, const Batch& bt,
                                     const LoadXf& x, gemm_config_t* cfg, LoadXf* in_kernel) {
  gemm_status_t s = select_config(ab, c, la, lb, M, N, K, A, lda, B, ldb, sm_count, forced, cfg, pair_clusters,
                                  bt.count, false);
  *in_kernel = x;
  if (s != GEMM_OK || !(x.a_on || x.b_on)) return s;
  const uint32_t staged = xf_stage_mask(ab, x, *cfg, la, lb, M, N, K, lda, ldb, bt);
  if (staged & GEMM_XF_A) in_kernel->a_on = 0;
  if (staged & GEMM_XF_B) in_kernel->b_on = 0;
  if (in_kernel->a_on || in_kernel->b_on) {
    s = select_config(ab, c, la, lb, M, N, K, A, lda, B, ldb, sm_count, forced, cfg, pair_clusters, bt.count, true);
    if (s != GEMM_OK) return s;
  }
  cfg->xf_staged = (int32_t)staged;
  return GEMM_OK;
}

}  // namespace

extern "C" {

int gemm_abi_version(void) { return 109; }

const char* gemm_status_string(gemm_status_t s) {
  switch (s) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG: invalid size, leading dimension, pointer or enum";
    case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED: request not implemented by this library";
    case GEMM_ERR_ALIGNMENT: return "GEMM_ERR_ALIGNMENT: forced kernel needs 16-byte aligned operands";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA: a CUDA call failed";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT: a bounded in-kernel wait expired";
    default: return "unknown gemm_status_t";
  }
}

gemm_status_t gemm_validate(gemm_dtype_t ab, gemm_dtype_t c, gemm_layout_t la, gemm_layout_t lb, int64_t M,
                            int64_t N, int64_t K, double alpha, const void* A, int64_t lda, const void* B,
                            int64_t ldb, double beta, const void* C, int64_t ldc, const void* D, int64_t ldd,
                            const gemm_epilogue_t* epi) {
  return validate(ab, c, la, lb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd, epi);
}

gemm_status_t gemm_select(gemm_dtype_t ab, gemm_dtype_t c, gemm_layout_t la, gemm_layout_t lb, int64_t M,
                          int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                          const void* C, int64_t ldc, const void* D, int64_t ldd, double beta,
                          const gemm_epilogue_t* epi, int sm_count, gemm_config_t* out) {
  if (!out) return GEMM_ERR_INVALID_ARG;
  const double alpha_probe = ab == GEMM_S8 ? 1.0 : 1.0;
  gemm_status_t s = validate(ab, c, la, lb, M, N, K, alpha_probe, A, lda, B, ldb, beta, C, ldc, D, ldd, epi);
  if (s != GEMM_OK) return s;
  // Host-only: a device whose SMs all pair up.
  LoadXf in_kernel{};
  return select_with_transforms(ab, c, la, lb, M, N, K, A, lda, B, ldb, sm_count, GEMM_KERNEL_AUTO, sm_count / 2,
                                Batch(), make_xf(ab, epi), out, &in_kernel);
}

gemm_status_t gemm_plan_create(gemm_plan_t* plan, gemm_dtype_t ab, gemm_dtype_t c, int device) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  *plan = nullptr;
  gemm_status_t s = check_types(ab, c);
  if (s != GEMM_OK) return s;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  DeviceGuard g(device);
  if (!g.ok) return GEMM_ERR_CUDA;
  gemm_plan* p = new (std::nothrow) gemm_plan();
  if (!p) return GEMM_ERR_CUDA;
  p->device = device;
  p->ab = ab;
  p->c = c;
  if (cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaMalloc(&p->d_err, sizeof(int32_t)) != cudaSuccess ||
      cudaMemset(p->d_err, 0, sizeof(int32_t)) != cudaSuccess) {
    if (p->d_err) cudaFree(p->d_err);
    delete p;
    return GEMM_ERR_CUDA;
  }
  p->pair_clusters = tc_pair_max_clusters(device);
  *plan = p;
  return GEMM_OK;
}

gemm_status_t gemm_plan_destroy(gemm_plan_t plan) {
  if (!plan) return GEMM_OK;
  DeviceGuard g(plan->device);
  cudaDeviceSynchronize();
  if (plan->ws) cudaFree(plan->ws);
  if (plan->stage) cudaFree(plan->stage);
  if (plan->sk_ws) cudaFree(plan->sk_ws);
  if (plan->sk1_ws) cudaFree(plan->sk1_ws);
  if (plan->d_err) cudaFree(plan->d_err);
  if (plan->host_pipe) {
    for (cudaEvent_t e : plan->host_ev) cudaEventDestroy(e);
    cudaStreamDestroy(plan->host_in);
    cudaStreamDestroy(plan->host_out);
  }
  delete plan;
  return GEMM_OK;
}

gemm_status_t gemm_plan_set_kernel(gemm_plan_t plan, gemm_kernel_t kernel) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  if (kernel != GEMM_KERNEL_AUTO && kernel != GEMM_KERNEL_TC && kernel != GEMM_KERNEL_TC_INT8 &&
      kernel != GEMM_KERNEL_FFMA && kernel != GEMM_KERNEL_SIMT && kernel != GEMM_KERNEL_TC_PAIR)
    return GEMM_ERR_INVALID_ARG;
  plan->forced = kernel;
  return GEMM_OK;
}

gemm_status_t gemm_plan_last_config(gemm_plan_t plan, gemm_config_t* out) {
  if (!plan || !out) return GEMM_ERR_INVALID_ARG;
  *out = plan->last;
  return GEMM_OK;
}

gemm_status_t gemm_plan_set_timeout(gemm_plan_t plan, uint64_t timeout_ns) {
  if (!plan || timeout_ns == 0) return GEMM_ERR_INVALID_ARG;
  plan->timeout_ns = timeout_ns;
  return GEMM_OK;
}

gemm_status_t gemm_plan_device_status(gemm_plan_t plan, gemm_stream_t stream, int32_t* code) {
  if (!plan || !code) return GEMM_ERR_INVALID_ARG;
  DeviceGuard g(plan->device);
  if (!g.ok) return GEMM_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GEMM_ERR_CUDA;
  if (cudaMemcpy(&v, plan->d_err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return GEMM_ERR_CUDA;
  if (cudaMemset(plan->d_err, 0, sizeof(int32_t)) != cudaSuccess) return GEMM_ERR_CUDA;
  // A launch that gave up may have left stream-K arrival counters counted in.
  if (v != 0 && plan->sk1_ws && cudaMemset(plan->sk1_ws, 0, plan->sk1_ws_bytes) != cudaSuccess) return GEMM_ERR_CUDA;
  *code = v;
  return GEMM_OK;
}

}  // extern "C"

namespace {

// One launch of a (strided) batch of problems whose arguments are already valid.
gemm_status_t run_impl(gemm_plan_t plan, gemm_layout_t la, gemm_layout_t lb, int64_t M, int64_t N, int64_t K,
                       double alpha, const void* A, int64_t lda, const void* B, int64_t ldb, double beta,
                       const void* C, int64_t ldc, void* D, int64_t ldd, const gemm_epilogue_t* epi,
                       gemm_stream_t stream_, const Batch& bt) {
  gemm_config_t cfg{};
  const LoadXf xf_req = make_xf(plan->ab, epi);
  LoadXf xf{};
  gemm_status_t s = select_with_transforms(plan->ab, plan->c, la, lb, M, N, K, A, lda, B, ldb, plan->sm_count,
                                           plan->forced, plan->pair_clusters, bt, xf_req, &cfg, &xf);
  if (s != GEMM_OK) return s;
  if (cfg.kernel == GEMM_KERNEL_NONE) {
    plan->last = cfg;
    return GEMM_OK;
  }
  DeviceGuard g(plan->device);
  if (!g.ok) return GEMM_ERR_CUDA;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  EpiParams e = make_epi(plan, alpha, beta, C, ldc, D, ldd, epi);
  e.stride_c = bt.sc;
  e.stride_d = bt.sd;
  e.stride_bias = bt.sbias;
  // The CTA-pair kernel's stream-K publishes partials under a per-launch epoch
  // chosen here on the host; a CUDA graph would replay the same epoch, so while
  // the stream is being captured the launch runs without stream-K.
  if (cfg.kernel == GEMM_KERNEL_TC_PAIR && cfg.sk_tiles > 0) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return GEMM_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone) {
      cfg.sk_tiles = 0;
      cfg.split_k = 1;
    }
  }

  // Staged operand transforms: each transformed operand (every problem of a
  // batch, a shared one once) is written to plan scratch with its own layout,
  // leading dimension and batch stride, and the GEMM reads the copy.
  if (cfg.xf_staged != 0) {
    const int64_t na = (bt.count > 1 && bt.sa != 0) ? bt.count : 1;
    const int64_t nb = (bt.count > 1 && bt.sb != 0) ? bt.count : 1;
    const int64_t a_el = (na - 1) * bt.sa + storage_elems(la, M, K, lda);
    const int64_t b_el = (nb - 1) * bt.sb + storage_elems(lb, K, N, ldb);
    const size_t a_bytes = (cfg.xf_staged & GEMM_XF_A) ? align_up((size_t)a_el * 2, 256) : 0;
    const size_t b_bytes = (cfg.xf_staged & GEMM_XF_B) ? (size_t)b_el * 2 : 0;
    s = ensure_ws(plan, a_bytes + b_bytes, stream);
    if (s != GEMM_OK) return s;
    cudaError_t ce = cudaSuccess;
    if (cfg.xf_staged & GEMM_XF_A) {
      uint16_t* As = static_cast<uint16_t*>(plan->ws);
      const uint16_t* Ao = static_cast<const uint16_t*>(A);
      for (int64_t z = 0; z < na && ce == cudaSuccess; ++z)
        ce = la == GEMM_OP_T ? launch_xf_stage(Ao + z * bt.sa, As + z * bt.sa, M, K, lda, xf_req, 0, stream)
                             : launch_xf_stage(Ao + z * bt.sa, As + z * bt.sa, K, M, lda, xf_req, 0, stream);
      A = As;
    }
    if (cfg.xf_staged & GEMM_XF_B) {
      uint16_t* Bs = reinterpret_cast<uint16_t*>(static_cast<char*>(plan->ws) + a_bytes);
      const uint16_t* Bo = static_cast<const uint16_t*>(B);
      for (int64_t z = 0; z < nb && ce == cudaSuccess; ++z)
        ce = lb == GEMM_OP_N ? launch_xf_stage(Bo + z * bt.sb, Bs + z * bt.sb, N, K, ldb, xf_req, 1, stream)
                             : launch_xf_stage(Bo + z * bt.sb, Bs + z * bt.sb, K, N, ldb, xf_req, 1, stream);
      B = Bs;
    }
    if (ce != cudaSuccess) return GEMM_ERR_CUDA;
  }

  switch (cfg.kernel) {
    case GEMM_KERNEL_TC_PAIR:
      s = launch_pair_problem(plan, cfg, la, lb, M, N, K, A, lda, B, ldb, plan->ab == GEMM_BF16, e, stream, 0, bt,
                              xf);
      break;
    case GEMM_KERNEL_TC: {
      const bool bf16 = plan->ab == GEMM_BF16;
      s = launch_tc_problem(plan, cfg, la, lb, M, N, K, A, lda, B, ldb,
                            bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, bf16,
                            e, 0, stream, bt, xf);
      break;
    }
    case GEMM_KERNEL_TC_INT8: {
      // Stage exact fp16 copies of A and B (same layouts, leading dimensions and
      // batch strides; a shared operand, stride 0, is staged once).
      const int64_t na = (bt.count > 1 && bt.sa != 0) ? bt.count : 1;
      const int64_t nb = (bt.count > 1 && bt.sb != 0) ? bt.count : 1;
      const int64_t a_el = (na - 1) * bt.sa + storage_elems(la, M, K, lda);
      const int64_t b_el = (nb - 1) * bt.sb + storage_elems(lb, K, N, ldb);
      const size_t a_bytes = align_up((size_t)a_el * 2, 256);
      s = ensure_ws(plan, a_bytes + (size_t)b_el * 2, stream);
      if (s != GEMM_OK) break;
      __half* A16 = static_cast<__half*>(plan->ws);
      __half* B16 = reinterpret_cast<__half*>(static_cast<char*>(plan->ws) + a_bytes);
      const int8_t* A8 = static_cast<const int8_t*>(A);
      const int8_t* B8 = static_cast<const int8_t*>(B);
      cudaError_t ce = cudaSuccess;
      // The int8 operand transform (ReLU) is applied as the operands are staged.
      for (int64_t z = 0; z < na && ce == cudaSuccess; ++z)
        ce = la == GEMM_OP_T ? launch_s8_to_f16(A8 + z * bt.sa, A16 + z * bt.sa, M, K, lda, stream, xf.a_relu)
                             : launch_s8_to_f16(A8 + z * bt.sa, A16 + z * bt.sa, K, M, lda, stream, xf.a_relu);
      for (int64_t z = 0; z < nb && ce == cudaSuccess; ++z)
        ce = lb == GEMM_OP_N ? launch_s8_to_f16(B8 + z * bt.sb, B16 + z * bt.sb, N, K, ldb, stream, xf.b_relu)
                             : launch_s8_to_f16(B8 + z * bt.sb, B16 + z * bt.sb, K, N, ldb, stream, xf.b_relu);
      if (ce != cudaSuccess) { s = GEMM_ERR_CUDA; break; }
      if (cfg.cta_group == 2)
        s = launch_pair_problem(plan, cfg, la, lb, M, N, K, A16, lda, B16, ldb, false, e, stream,
                                cfg.k_chunk / TC_BK, bt);
      else
        s = launch_tc_problem(plan, cfg, la, lb, M, N, K, A16, lda, B16, ldb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                              false, e, cfg.k_chunk / TC_BK, stream, bt);
      break;
    }
    case GEMM_KERNEL_FFMA: {
      FfmaParams fp{};
      fp.A = static_cast<const float*>(A);
      fp.B = static_cast<const float*>(B);
      fp.lda = lda;
      fp.ldb = ldb;
      fp.M = (int32_t)M;
      fp.N = (int32_t)N;
      fp.K = (int32_t)K;
      fp.stride_a = bt.sa;
      fp.stride_b = bt.sb;
      fp.full_tiles = cfg.tiles;
      fp.split = 1;
      if (cfg.sk_tiles > 0) {
        // Split tail wave: raw fp32 sums of each part of each tail tile in plan scratch.
        fp.full_tiles = cfg.tiles - cfg.sk_tiles;
        fp.split = cfg.split_k;
        const int64_t nkt = (K + FFMA_BK - 1) / FFMA_BK;
        fp.kb_per_part = (int32_t)((nkt + cfg.split_k - 1) / cfg.split_k);
        s = ensure_ws(plan, (size_t)cfg.sk_tiles * cfg.split_k * FFMA_BM * FFMA_BN * sizeof(float), stream);
        if (s != GEMM_OK) break;
        fp.ws = static_cast<float*>(plan->ws);
      }
      fp.xf = xf;
      fp.epi = e;
      s = launch_ffma(fp, la == GEMM_OP_T, lb == GEMM_OP_T, (int)bt.count, stream) == cudaSuccess ? GEMM_OK
                                                                                     : GEMM_ERR_CUDA;
      break;
    }
    default: {
      SimtParams sp{};
      sp.A = A;
      sp.B = B;
      sp.lda = lda;
      sp.ldb = ldb;
      sp.ab_dtype = plan->ab;
      sp.a_row_major = la == GEMM_OP_T;
      sp.b_row_major = lb == GEMM_OP_T;
      sp.M = M;
      sp.N = N;
      sp.K = K;
      sp.stride_a = bt.sa;
      sp.stride_b = bt.sb;
      sp.xf = xf;
      sp.epi = e;
      s = launch_simt(sp, (int)bt.count, stream) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
      break;
    }
  }
  if (s == GEMM_OK) {
    plan->last = cfg;
    log_config("run", M, N, K, bt.count, cfg);
  }
  return s;
}

// Can the tensor-core paths take this batch as one launch (TMA batch
// dimension, tile count within range, grid rows within range for CUDA cores)?
bool batch_fits_one_launch(gemm_dtype_t ab, int64_t M, int64_t N, const Batch& bt) {
  if (bt.count <= 1) return true;
  if (bt.count > 65535) return false;
  const int es = dtype_bytes(ab);
  const int64_t stage_es = ab == GEMM_S8 ? 2 : es;   // int8 operands are staged as fp16
  for (int64_t st : {bt.sa, bt.sb})
    if (st != 0 && ((st * stage_es) % 16 != 0 || st * stage_es >= (int64_t(1) << 40))) return false;
  const int64_t tiles = bt.count * ((M + 127) / 128) * ((N + 127) / 128);
  return tiles <= kMaxDim;
}

}  // namespace

extern "C" {

gemm_status_t gemm_run(gemm_plan_t plan, gemm_layout_t la, gemm_layout_t lb, int64_t M, int64_t N, int64_t K,
                       double alpha, const void* A, int64_t lda, const void* B, int64_t ldb, double beta,
                       const void* C, int64_t ldc, void* D, int64_t ldd, const gemm_epilogue_t* epi,
                       gemm_stream_t stream) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  NvtxRange range("gemm_run");
  gemm_status_t s = validate(plan->ab, plan->c, la, lb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd, epi);
  if (s != GEMM_OK) return s;
  return run_impl(plan, la, lb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd, epi, stream, Batch());
}

gemm_status_t gemm_run_strided_batched(gemm_plan_t plan, gemm_layout_t la, gemm_layout_t lb, int64_t M,
                                       int64_t N, int64_t K, double alpha, const void* A, int64_t lda,
                                       int64_t stride_a, const void* B, int64_t ldb, int64_t stride_b,
                                       double beta, const void* C, int64_t ldc, int64_t stride_c, void* D,
                                       int64_t ldd, int64_t stride_d, int64_t batch,
                                       const gemm_epilogue_t* epi, int64_t stride_bias, gemm_stream_t stream) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  NvtxRange range("gemm_run_strided_batched");
  gemm_status_t s = validate(plan->ab, plan->c, la, lb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd, epi);
  if (s != GEMM_OK) return s;
  if (batch < 0 || stride_a < 0 || stride_b < 0 || stride_c < 0 || stride_d < 0 || stride_bias < 0)
    return GEMM_ERR_INVALID_ARG;
  if (batch == 0 || M == 0 || N == 0) return GEMM_OK;
  // Outputs of different problems must not overlap; in-place C == D needs equal strides.
  if (batch > 1 && stride_d < (M - 1) * ldd + N) return GEMM_ERR_INVALID_ARG;
  if (beta != 0.0 && C == D && stride_c != stride_d) return GEMM_ERR_INVALID_ARG;
  Batch bt;
  bt.count = batch;
  bt.sa = K > 0 ? stride_a : 0;
  bt.sb = K > 0 ? stride_b : 0;
  bt.sc = beta != 0.0 ? stride_c : 0;
  bt.sd = stride_d;
  bt.sbias = (epi && epi->bias_mode != GEMM_BIAS_NONE) ? stride_bias : 0;
  if (batch_fits_one_launch(plan->ab, M, N, bt))
    return run_impl(plan, la, lb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd, epi, stream, bt);
  // Otherwise one launch per problem.
  const int es = dtype_bytes(plan->ab), cs = dtype_bytes(plan->c);
  const gemm_dtype_t out = out_dtype_of(plan->c, epi);
  for (int64_t z = 0; z < batch; ++z) {
    gemm_epilogue_t ez{};
    if (epi) {
      ez = *epi;
      if (ez.bias_mode != GEMM_BIAS_NONE)
        ez.bias = static_cast<const char*>(epi->bias) + z * bt.sbias * dtype_bytes(epi->bias_dtype);
    }
    s = run_impl(plan, la, lb, M, N, K, alpha, static_cast<const char*>(A) + z * bt.sa * es, lda,
                 static_cast<const char*>(B) + z * bt.sb * es, ldb, beta,
                 C ? static_cast<const char*>(C) + z * bt.sc * cs : nullptr, ldc,
                 static_cast<char*>(D) + z * bt.sd * dtype_bytes(out), ldd, epi ? &ez : nullptr, stream,
                 Batch());
    if (s != GEMM_OK) return s;
  }
  return GEMM_OK;
}

gemm_status_t gemm_run_diag(gemm_plan_t plan, gemm_side_t side, gemm_layout_t lx, int64_t M, int64_t N,
                            double alpha, const void* diag, const void* X, int64_t ldx, double beta,
                            const void* C, int64_t ldc, void* D, int64_t ldd, const gemm_epilogue_t* epi,
                            gemm_stream_t stream_) {
  if (!plan || (side != GEMM_SIDE_LEFT && side != GEMM_SIDE_RIGHT)) return GEMM_ERR_INVALID_ARG;
  NvtxRange range("gemm_run_diag");
  const bool left = side == GEMM_SIDE_LEFT;
  // The checks of the equivalent dense call (the diagonal as a square operand).
  gemm_status_t s =
      left ? validate(plan->ab, plan->c, GEMM_OP_N, lx, M, N, M, alpha, diag, std::max<int64_t>(1, M), X, ldx,
                      beta, C, ldc, D, ldd, epi)
           : validate(plan->ab, plan->c, lx, GEMM_OP_N, M, N, N, alpha, X, ldx, diag, std::max<int64_t>(1, N),
                      beta, C, ldc, D, ldd, epi);
  if (s != GEMM_OK) return s;
  if (epi && epi->load_xf != 0) return GEMM_ERR_UNSUPPORTED;   // no operand transforms on this path
  gemm_config_t cfg{};
  cfg.split_k = 1;
  cfg.cta_group = 1;
  cfg.cluster = 1;
  if (M == 0 || N == 0) {
    cfg.kernel = GEMM_KERNEL_NONE;
    plan->last = cfg;
    return GEMM_OK;
  }
  DeviceGuard g(plan->device);
  if (!g.ok) return GEMM_ERR_CUDA;
  DiagParams p{};
  p.X = X;
  p.diag = diag;
  p.ldx = ldx;
  p.M = M;
  p.N = N;
  p.tiles_n = (N + DIAG_TN - 1) / DIAG_TN;
  p.num_tiles = ((M + DIAG_TM - 1) / DIAG_TM) * p.tiles_n;
  p.ab_dtype = plan->ab;
  p.left = left ? 1 : 0;
  const int es = dtype_bytes(plan->ab);
  p.vec_x = (aligned16(X) && (ldx * es) % 16 == 0) ? 1 : 0;
  p.vec_diag = aligned16(diag) ? 1 : 0;
  p.epi = make_epi(plan, alpha, beta, C, ldc, D, ldd, epi);
  // 16-bit x with TMA-alignable x and C: the TMA-staged kernel (x and C stream
  // through a ring of shared-memory stages; GEMM_DIAG_TMA=0 keeps the register kernel).
  const int cs = dtype_bytes(plan->c);
  const bool has_bias = p.epi.bias_mode != GEMM_BIAS_NONE;
  bool tma = is_f16ish(plan->ab) && tma_ok(X, ldx, 2) && aligned16(diag) &&
             (!p.epi.read_c || (is_float_out(plan->c) && tma_ok(C, ldc, cs))) &&
             (!has_bias || (is_float_out((gemm_dtype_t)p.epi.bias_dtype) && aligned16(p.epi.bias)));
  if (const char* env = std::getenv("GEMM_DIAG_TMA"))
    if (std::atoi(env) == 0) tma = false;
  if (tma) {
    const CUtensorMapDataType xdt =
        plan->ab == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const bool x_rm = lx == GEMM_OP_T;
    bool ok = encode_2d(&p.tmX, xdt, 2, X, x_rm ? (uint64_t)N : (uint64_t)M, x_rm ? (uint64_t)M : (uint64_t)N,
                        (uint64_t)ldx, DIAG_TN, DIAG_TM);
    if (ok && p.epi.read_c)
      ok = encode_2d(&p.tmC, tma_dtype(plan->c), cs, C, (uint64_t)N, (uint64_t)M, (uint64_t)ldc,
                     plan->c == GEMM_F32 ? 32 : 64, DIAG_TM);
    if (ok) ok = encode_1d(&p.tmDiag, xdt, diag, (uint64_t)(left ? M : N), 64);
    if (ok && has_bias)
      ok = encode_1d(&p.tmBias, tma_dtype((gemm_dtype_t)p.epi.bias_dtype), p.epi.bias,
                     (uint64_t)(p.epi.bias_mode == GEMM_BIAS_ROW ? M : N), 64);
    if (!ok) return GEMM_ERR_CUDA;
    p.use_tma = 1;
    p.err = plan->d_err;
    p.timeout_ns = plan->timeout_ns;
  }
  int grid = 0;
  if (launch_diag(p, lx == GEMM_OP_T, plan->sm_count, &grid, reinterpret_cast<cudaStream_t>(stream_)) !=
      cudaSuccess)
    return GEMM_ERR_CUDA;
  cfg.kernel = GEMM_KERNEL_DIAG;
  cfg.bm = DIAG_TM;
  cfg.bn = DIAG_TN;
  cfg.stages = p.use_tma ? DIAG_TMA_STAGES : 1;
  cfg.grid = grid;
  cfg.tiles = (int32_t)std::min<int64_t>(p.num_tiles, kMaxDim);
  plan->last = cfg;
  log_config("diag", M, N, left ? M : N, 1, cfg);
  return GEMM_OK;
}

gemm_status_t gemm_run_complex(gemm_plan_t plan, gemm_unit_t unit, gemm_layout_t la, gemm_layout_t lb,
                               int64_t M, int64_t N, int64_t K, double alpha, const void* A, int64_t lda,
                               const void* B, int64_t ldb, double beta, const void* C, int64_t ldc, void* D,
                               int64_t ldd, const gemm_epilogue_t* epi, gemm_stream_t stream_) {
  if (!plan || (unit != GEMM_UNIT_IMAGINARY && unit != GEMM_UNIT_DUAL)) return GEMM_ERR_INVALID_ARG;
  NvtxRange range("gemm_run_complex");
  // The argument checks of gemm_run, in pairs.
  gemm_status_t s = validate(plan->ab, plan->c, la, lb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd, epi);
  if (s != GEMM_OK) return s;
  if (plan->ab == GEMM_S8) return GEMM_ERR_UNSUPPORTED;
  if (epi && epi->bias_mode == GEMM_BIAS_ROW) return GEMM_ERR_UNSUPPORTED;
  if (epi && epi->load_xf != 0) return GEMM_ERR_UNSUPPORTED;   // no operand transforms on this path
  if (2 * N > kMaxDim || 2 * K > kMaxDim) return GEMM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) {
    gemm_config_t none{};
    none.kernel = GEMM_KERNEL_NONE;
    plan->last = none;
    return GEMM_OK;
  }
  DeviceGuard g(plan->device);
  if (!g.ok) return GEMM_ERR_CUDA;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const int es = dtype_bytes(plan->ab);
  // The real problem: M x 2N x 2K; A as an M x 2K matrix, B as the staged 2K x 2N one.
  const void* Ar = A;
  int64_t lda_r = 2 * lda;
  gemm_layout_t la_r = la;
  const void* Br = B;
  int64_t ldb_r = 0;
  if (K > 0) {
    // A: row-major A is read in place when TMA can address it; otherwise staged.
    const bool stage_a = la == GEMM_OP_N || !tma_ok(A, 2 * lda, es);
    const int64_t lds = la == GEMM_OP_N ? (M + 7) / 8 * 8 : (2 * K + 7) / 8 * 8;
    const size_t a_bytes = stage_a ? align_up((size_t)lds * (la == GEMM_OP_N ? 2 * K : M) * es, 256) : 0;
    ldb_r = lb == GEMM_OP_N ? (2 * K + 7) / 8 * 8 : (2 * N + 7) / 8 * 8;
    const size_t b_bytes = (size_t)ldb_r * (lb == GEMM_OP_N ? 2 * N : 2 * K) * es;
    s = ensure_ws(plan, a_bytes + b_bytes, stream);
    if (s != GEMM_OK) return s;
    char* ws = static_cast<char*>(plan->ws);
    cudaError_t ce = cudaSuccess;
    if (stage_a) {
      ce = launch_pair_stage_a(A, lda, la == GEMM_OP_T, M, K, es, ws, lds, stream);
      Ar = ws;
      lda_r = lds;
    }
    if (ce == cudaSuccess)
      ce = launch_pair_stage_b(B, ldb, lb == GEMM_OP_T, K, N, es, unit == GEMM_UNIT_DUAL, ws + a_bytes, ldb_r,
                               stream);
    if (ce != cudaSuccess) return GEMM_ERR_CUDA;
    Br = ws + a_bytes;
    la_r = la;
  }
  return run_impl(plan, la_r, lb, M, 2 * N, 2 * K, alpha, Ar, lda_r, Br, ldb_r, beta, C, 2 * ldc, D, 2 * ldd, epi,
                  stream_, Batch());
}

gemm_status_t gemm_run_host(gemm_plan_t plan, gemm_layout_t la, gemm_layout_t lb, int64_t M, int64_t N,
                            int64_t K, double alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
                            double beta, const void* C, int64_t ldc, void* D, int64_t ldd,
                            const gemm_epilogue_t* epi, gemm_stream_t stream_) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  NvtxRange range("gemm_run_host");
  gemm_status_t s = validate(plan->ab, plan->c, la, lb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd, epi);
  if (s != GEMM_OK) return s;
  if (M == 0 || N == 0) return GEMM_OK;
  DeviceGuard g(plan->device);
  if (!g.ok) return GEMM_ERR_CUDA;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const gemm_dtype_t out = out_dtype_of(plan->c, epi);
  const int ab_b = dtype_bytes(plan->ab);
  const size_t a_bytes = K > 0 ? (size_t)storage_elems(la, M, K, lda) * ab_b : 0;
  const size_t b_bytes = K > 0 ? (size_t)storage_elems(lb, K, N, ldb) * ab_b : 0;
  const bool in_place = beta != 0.0 && C == D;
  const size_t c_bytes = (beta != 0.0 && !in_place) ? (size_t)((M - 1) * ldc + N) * dtype_bytes(plan->c) : 0;
  const bool has_bias = epi && epi->bias_mode != GEMM_BIAS_NONE;
  const size_t bias_bytes =
      has_bias ? (size_t)(epi->bias_mode == GEMM_BIAS_COL ? N : M) * dtype_bytes(epi->bias_dtype) : 0;
  const size_t d_bytes = (size_t)((M - 1) * ldd + N) * dtype_bytes(out);
  size_t off_a = 0, off_b = align_up(off_a + a_bytes, 256), off_c = align_up(off_b + b_bytes, 256);
  size_t off_bias = align_up(off_c + c_bytes, 256), off_d = align_up(off_bias + bias_bytes, 256);
  const size_t total = align_up(off_d + d_bytes, 256);
  if (plan->stage_bytes < total) {
    if (plan->stage) {
      cudaStreamSynchronize(stream);
      cudaFree(plan->stage);
      plan->stage = nullptr;
      plan->stage_bytes = 0;
    }
    if (cudaMalloc(&plan->stage, total) != cudaSuccess) return GEMM_ERR_CUDA;
    plan->stage_bytes = total;
  }
  char* base = static_cast<char*>(plan->stage);
  void* dA = base + off_a;
  void* dB = base + off_b;
  void* dD = base + off_d;
  void* dC = in_place ? dD : (beta != 0.0 ? base + off_c : nullptr);
  void* dbias = has_bias ? base + off_bias : nullptr;
  gemm_epilogue_t e2{};
  if (epi) {
    e2 = *epi;
    e2.bias = dbias;
  }
  const int cb = dtype_bytes(plan->c), db = dtype_bytes(out);

  // Row panels: rows [m0, m0 + mi) of A (layout T: whole rows; layout N: one strip
  // of every column), C and D.  Panel i's inputs are copied in on one stream while
  // panel i-1 runs on the caller's stream and panel i-2's D is copied out on a
  // third, so the host link carries both directions at once and the GEMM hides
  // behind the copies.  Small problems run as one panel.
  int64_t rows = M;
  if (K > 0 && M >= 2048 && a_bytes + c_bytes + d_bytes >= ((size_t)64 << 20)) {
    const int64_t panels = std::min<int64_t>(kHostMaxPanels, M / 1024);
    rows = ((M + panels - 1) / panels + 255) / 256 * 256;
  }
  const int P = (int)((M + rows - 1) / rows);
  if (P > 1 && !plan->host_pipe) {
    bool ok = cudaStreamCreateWithFlags(&plan->host_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&plan->host_out, cudaStreamNonBlocking) == cudaSuccess;
    for (cudaEvent_t& e : plan->host_ev) ok = ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) return GEMM_ERR_CUDA;
    plan->host_pipe = true;
  }
  cudaStream_t in = P > 1 ? plan->host_in : stream, outs = P > 1 ? plan->host_out : stream;
  cudaEvent_t* ev = plan->host_ev;   // [0] start, [1] end, [2 + i] panel i in, [2 + kHostMaxPanels + i] panel i done
  auto ck = [](cudaError_t e) { return e == cudaSuccess; };
  if (P > 1) {
    // Everything already queued on the caller's stream comes first.
    if (!ck(cudaEventRecord(ev[0], stream)) || !ck(cudaStreamWaitEvent(in, ev[0], 0)) ||
        !ck(cudaStreamWaitEvent(outs, ev[0], 0)))
      return GEMM_ERR_CUDA;
  }
  if (b_bytes && !ck(cudaMemcpyAsync(dB, B, b_bytes, cudaMemcpyHostToDevice, in))) return GEMM_ERR_CUDA;
  if (has_bias && !ck(cudaMemcpyAsync(dbias, epi->bias, bias_bytes, cudaMemcpyHostToDevice, in))) return GEMM_ERR_CUDA;
  for (int i = 0; i < P; ++i) {
    const int64_t m0 = (int64_t)i * rows, mi = std::min<int64_t>(rows, M - m0);
    const char* hA = static_cast<const char*>(A);
    char* pA = static_cast<char*>(dA);
    if (K > 0) {
      if (la == GEMM_OP_T) {
        if (!ck(cudaMemcpyAsync(pA + m0 * lda * ab_b, hA + m0 * lda * ab_b, (size_t)((mi - 1) * lda + K) * ab_b,
                                cudaMemcpyHostToDevice, in)))
          return GEMM_ERR_CUDA;
      } else if (!ck(cudaMemcpy2DAsync(pA + m0 * ab_b, (size_t)lda * ab_b, hA + m0 * ab_b, (size_t)lda * ab_b,
                                       (size_t)mi * ab_b, (size_t)K, cudaMemcpyHostToDevice, in))) {
        return GEMM_ERR_CUDA;
      }
    }
    if (beta != 0.0 && !ck(cudaMemcpyAsync(static_cast<char*>(dC) + m0 * ldc * cb,
                                           static_cast<const char*>(C) + m0 * ldc * cb,
                                           (size_t)((mi - 1) * ldc + N) * cb, cudaMemcpyHostToDevice, in)))
      return GEMM_ERR_CUDA;
    if (P > 1 && (!ck(cudaEventRecord(ev[2 + i], in)) || !ck(cudaStreamWaitEvent(stream, ev[2 + i], 0))))
      return GEMM_ERR_CUDA;
    gemm_epilogue_t ei = e2;
    if (has_bias && epi->bias_mode == GEMM_BIAS_ROW)
      ei.bias = static_cast<const char*>(dbias) + m0 * dtype_bytes(epi->bias_dtype);
    const void* pAi = la == GEMM_OP_T ? (const void*)(pA + m0 * lda * ab_b) : (const void*)(pA + m0 * ab_b);
    s = gemm_run(plan, la, lb, mi, N, K, alpha, pAi, lda, dB, ldb, beta,
                 beta != 0.0 ? static_cast<const char*>(dC) + m0 * ldc * cb : nullptr, ldc,
                 static_cast<char*>(dD) + m0 * ldd * db, ldd, epi ? &ei : nullptr, stream_);
    if (s != GEMM_OK) return s;
    if (P > 1 && (!ck(cudaEventRecord(ev[2 + kHostMaxPanels + i], stream)) ||
                  !ck(cudaStreamWaitEvent(outs, ev[2 + kHostMaxPanels + i], 0))))
      return GEMM_ERR_CUDA;
    // Only the N columns of each row: the caller's padding between rows stays untouched.
    char* hD = static_cast<char*>(D) + m0 * ldd * db;
    const char* sD = static_cast<const char*>(dD) + m0 * ldd * db;
    const cudaError_t ce = ldd == N ? cudaMemcpyAsync(hD, sD, (size_t)(mi * N) * db, cudaMemcpyDeviceToHost, outs)
                                    : cudaMemcpy2DAsync(hD, (size_t)ldd * db, sD, (size_t)ldd * db, (size_t)N * db,
                                                        (size_t)mi, cudaMemcpyDeviceToHost, outs);
    if (!ck(ce)) return GEMM_ERR_CUDA;
  }
  if (P > 1 && (!ck(cudaEventRecord(ev[1], outs)) || !ck(cudaStreamWaitEvent(stream, ev[1], 0))))
    return GEMM_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return GEMM_ERR_CUDA;
  return GEMM_OK;
}

}  // extern "C"

// ===========================================================================
// gemm_run_s8_noalloc: the int8 path with its fp16 staging in a fixed device
// array instead of plan-owned, allocated scratch (see include/gemm.h).
// ===========================================================================

// The staging array and the library's own error word.  In host code these
// names are host-side stand-ins, not device addresses: the host only ever
// passes the addresses cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GEMM_NOALLOC_SCRATCH_BYTES];
static __device__ __align__(16) int32_t g_noalloc_status;

namespace {

struct NoallocDevice {
  bool ready = false;
  void* scratch = nullptr;     // device address of g_noalloc_scratch on this device
  int32_t* status = nullptr;   // device address of g_noalloc_status on this device
  int sm_count = 0;
};

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mu;
NoallocDevice g_noalloc_dev[kNoallocMaxDevices];
// Bound of the in-kernel waits of gemm_run_s8_noalloc (gemm_noalloc_set_timeout).
std::atomic<uint64_t> g_noalloc_timeout_ns{4000000000ull};

// Once per device, with that device current: look up the arrays' device addresses.
gemm_status_t noalloc_device(int dev, NoallocDevice** out) {
  if (dev < 0 || dev >= kNoallocMaxDevices) return GEMM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocDevice& d = g_noalloc_dev[dev];
  if (!d.ready) {
    void* scratch = nullptr;
    void* status = nullptr;
    if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess) return GEMM_ERR_CUDA;
    if (cudaGetSymbolAddress(&status, g_noalloc_status) != cudaSuccess) return GEMM_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return GEMM_ERR_CUDA;
    d.scratch = scratch;
    d.status = static_cast<int32_t*>(status);
    d.ready = true;
  }
  *out = &d;
  return GEMM_OK;
}

}  // namespace

extern "C" gemm_status_t gemm_run_s8_noalloc(gemm_layout_t la, gemm_layout_t lb, int64_t M, int64_t N,
                                             int64_t K, double alpha, const void* A, int64_t lda,
                                             const void* B, int64_t ldb, double beta, const void* C,
                                             int64_t ldc, void* D, int64_t ldd, const gemm_epilogue_t* epi,
                                             int32_t* status, gemm_stream_t stream_) {
  gemm_status_t s = validate(GEMM_S8, GEMM_S32, la, lb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd, epi);
  if (s != GEMM_OK) return s;
  if (M == 0 || N == 0) return GEMM_OK;
  size_t a_bytes = 0, total = 0;
  if (K > 0) {
    if ((lda % 8) != 0 || (ldb % 8) != 0) return GEMM_ERR_ALIGNMENT;
    a_bytes = align_up((size_t)storage_elems(la, M, K, lda) * 2, 256);
    total = a_bytes + (size_t)storage_elems(lb, K, N, ldb) * 2;
    if (total > (size_t)GEMM_NOALLOC_SCRATCH_BYTES) return GEMM_ERR_UNSUPPORTED;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
  NoallocDevice* nd = nullptr;
  s = noalloc_device(dev, &nd);
  if (s != GEMM_OK) return s;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  // The library's word keeps the first failure until gemm_noalloc_device_status reads it.
  int32_t* err = status ? status : nd->status;

  // A plan-shaped record on the stack (no device memory behind it) so that the
  // launch helpers of gemm_run serve this entry point unchanged.
  gemm_plan local;
  local.device = dev;
  local.ab = GEMM_S8;
  local.c = GEMM_S32;
  local.sm_count = nd->sm_count;
  local.d_err = err;
  local.timeout_ns = g_noalloc_timeout_ns.load();
  gemm_config_t cfg{};
  s = select_config(GEMM_S8, GEMM_S32, la, lb, M, N, K, A, lda, B, ldb, local.sm_count, GEMM_KERNEL_AUTO, &cfg);
  if (s != GEMM_OK) return s;
  const EpiParams e = make_epi(&local, alpha, beta, C, ldc, D, ldd, epi);
  // With K > 0 the leading dimensions were checked above, so the selector picks
  // the single-CTA int8 kernel (no CTA-pair plan data exists here); K == 0 leaves
  // the epilogue of beta*C alone, which the generic kernel runs without staging.
  if (cfg.kernel != GEMM_KERNEL_TC_INT8) {
    if (K != 0) return GEMM_ERR_UNSUPPORTED;
    SimtParams sp{};
    sp.A = A;
    sp.B = B;
    sp.lda = lda;
    sp.ldb = ldb;
    sp.ab_dtype = GEMM_S8;
    sp.a_row_major = la == GEMM_OP_T;
    sp.b_row_major = lb == GEMM_OP_T;
    sp.M = M;
    sp.N = N;
    sp.K = K;
    sp.epi = e;
    return launch_simt(sp, stream) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
  }
  __half* A16 = static_cast<__half*>(nd->scratch);
  __half* B16 = reinterpret_cast<__half*>(static_cast<char*>(nd->scratch) + a_bytes);
  const int8_t* A8 = static_cast<const int8_t*>(A);
  const int8_t* B8 = static_cast<const int8_t*>(B);
  // The int8 operand transform (ReLU), if any, is applied as the operands are staged.
  const LoadXf xf = make_xf(GEMM_S8, epi);
  cudaError_t ce = la == GEMM_OP_T ? launch_s8_to_f16(A8, A16, M, K, lda, stream, xf.a_relu)
                                   : launch_s8_to_f16(A8, A16, K, M, lda, stream, xf.a_relu);
  if (ce == cudaSuccess)
    ce = lb == GEMM_OP_N ? launch_s8_to_f16(B8, B16, N, K, ldb, stream, xf.b_relu)
                         : launch_s8_to_f16(B8, B16, K, N, ldb, stream, xf.b_relu);
  if (ce != cudaSuccess) return GEMM_ERR_CUDA;
  return launch_tc_problem(&local, cfg, la, lb, M, N, K, A16, lda, B16, ldb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                           false, e, cfg.k_chunk / TC_BK, stream);
}

extern "C" gemm_status_t gemm_noalloc_device_status(int32_t* code, gemm_stream_t stream_) {
  if (!code) return GEMM_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
  NoallocDevice* nd = nullptr;
  gemm_status_t s = noalloc_device(dev, &nd);
  if (s != GEMM_OK) return s;
  int32_t v = 0;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream_)) != cudaSuccess) return GEMM_ERR_CUDA;
  if (cudaMemcpy(&v, nd->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return GEMM_ERR_CUDA;
  if (cudaMemset(nd->status, 0, sizeof(int32_t)) != cudaSuccess) return GEMM_ERR_CUDA;
  *code = v;
  return GEMM_OK;
}

extern "C" gemm_status_t gemm_noalloc_set_timeout(uint64_t timeout_ns) {
  if (timeout_ns == 0) return GEMM_ERR_INVALID_ARG;
  g_noalloc_timeout_ns.store(timeout_ns);
  return GEMM_OK;
}


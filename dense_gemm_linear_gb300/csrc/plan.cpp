// Host-side planner: path selection, the tile ladder, the padding screen and
// a cost model built on tile- and wave-quantisation efficiency.  Pure host
// code (no CUDA calls), so it runs and is tested without a GPU.
//
//  * Tile/wave quantisation: "GEMM analysis in TraceLens", section "GEMM
//    dimension efficiency" (tile_eff, wq_eff, dim_eff; "Split-K or Stream-K
//    are not yet modeled" there, and are not here either).
//  * Padding screen: FlyDSL pull request 1303 (autotuner): reject a tile whose
//    padded output area exceeds 1.25x the real area, unless nothing passes.
//  * Ranking: that change's fallback weighs occupancy and last-round fill
//    against work per byte of operand traffic; here the same quantities enter
//    an explicit time estimate (waves x per-tile time, per-tile time = max of
//    tensor-core time and operand-load time).
//  * Decode: m <= 16 goes to the memory-bound path ("Gemm Optimization"
//    guide, section 8.3: small M is bandwidth-bound).
#include <algorithm>
#include <cmath>
#include <cstdint>

#include "dgl.h"
#include "plan.h"

namespace dgl {

namespace {

// Cost model, calibrated on GB300 by timing every rung on the benchmark shapes
// (L2 rotated): a launch costs kLaunchUs, each wave of tiles costs
// k_stages x kStageUs[rung] + kTileUs[rung], where a k-stage is 128 bytes of
// K.  The per-stage figure already folds in the operand-load limit (about 64
// B/clk per SM), so 1-CTA 128 x 256 tiles cost more per stage than the CTA
// pair's 256 x 256.
constexpr double kLaunchUs = 5.0;
constexpr double kHbmGBs = 6500.0;              // achievable HBM bandwidth

struct Rung {
  int tile_m, tile_n;  // tile_m 256 = a CTA pair (cta_group::2), 128 rows per CTA; 64 = one CTA, M = 64 MMAs
  double stage_us;     // per 128-byte k-stage
  double tile_us;      // per tile: accumulator drain, epilogue not hidden
  int max_kb;          // the planner offers the rung only up to this many k-stages (0: any)
};
// The 224-wide pair tile fills 4096 columns with 19 tiles, so 4096 x 4096
// outputs make exactly four waves of 76 pairs.  Measured (interleaved,
// L2-rotated): 4095^2 x 1024 28.3 us against 30.9 us on 256 x 256; at K =
// 4096 its tiles take as long as 256-wide ones (bf16 77.5 against 77.7 us,
// E4M3 45.1 against 44.5 us), so it is offered for short K only.
constexpr Rung kLadder[] = {
    {64, 64, 0.200, 1.0, 0},   {64, 128, 0.230, 1.0, 0},   {64, 256, 0.300, 2.0, 0},
    {128, 64, 0.260, 1.0, 0},  {128, 128, 0.265, 1.0, 0},  {128, 256, 0.322, 2.6, 0},
    {256, 128, 0.270, 1.0, 0}, {256, 224, 0.278, 1.6, 16}, {256, 256, 0.278, 2.2, 0},
};

// Measured pins: shapes where the screened model's pick is more than 5% off
// the best rung of a full sweep.  Consulted before the screen and the model,
// as the FlyDSL autotuner consults its measured tile table; a pin may name a
// rung the padding screen would reject when the sweep shows it faster (the
// 597-token prefill pads 597 rows to 768 on CTA pairs and still wins).
struct Pin {
  int dtype;
  int64_t m, n, K;
  int tile_m, tile_n;
};
constexpr Pin kPins[] = {
    {DGL_DTYPE_BF16, 1024, 50257, 512, 128, 256},  // lm_head: short K, epilogue-bound; 58.9 us vs 67.0 us
    {DGL_DTYPE_BF16, 2048, 2048, 2048, 128, 256},  // one wave either way; 17.9 us vs 19.7 us
    {DGL_DTYPE_BF16, 48, 4096, 48, 64, 64},        // 3.57 us vs 3.73 us (128x128), 3.67 us (128x64)
    {DGL_DTYPE_BF16, 528, 528, 1024, 64, 64},      // 7.12 us vs 7.25 us (128x64), 7.52 us (128x128)
    {DGL_DTYPE_BF16, 3402, 4096, 1024, 256, 256},  // 21.7 us vs 22.9 us (128x256)
    {DGL_DTYPE_BF16, 597, 11008, 4096, 256, 256},  // 47.0 us vs 54.9 us (128x256, the screen's pick)
    {DGL_DTYPE_E4M3, 597, 11008, 4096, 256, 256},  // 30.4 us vs 33.4 us
};

}  // namespace

void tile_metrics(int64_t m, int64_t n, int tile_m, int tile_n, int units, dgl_plan_info* out) {
  const int64_t tiles_m = (m + tile_m - 1) / tile_m;
  const int64_t tiles_n = (n + tile_n - 1) / tile_n;
  const int64_t tiles = tiles_m * tiles_n;
  const int64_t rounds = (tiles + units - 1) / units;
  out->num_tiles = static_cast<int32_t>(std::min<int64_t>(tiles, INT32_MAX));
  out->tile_eff = static_cast<double>(m) * static_cast<double>(n) /
                  (static_cast<double>(tiles_m * tile_m) * static_cast<double>(tiles_n * tile_n));
  out->wq_eff = rounds > 0 ? static_cast<double>(tiles) / static_cast<double>(rounds * units) : 0.0;
  out->dim_eff = out->tile_eff * out->wq_eff;
}

double operand_bytes(int dtype, int out_dtype, int64_t m, int64_t n, int64_t K) {
  const double e = dtype == DGL_DTYPE_E4M3 ? 1.0 : 2.0;
  const double o = out_dtype == DGL_OUT_F32 ? 4.0 : 2.0;
  double bytes = (static_cast<double>(m) * K + static_cast<double>(n) * K) * e + static_cast<double>(m) * n * o;
  if (dtype == DGL_DTYPE_E4M3) bytes += 4.0 * static_cast<double>(m + n);
  return bytes;
}

static const Rung* find_rung(int tile_m, int tile_n) {
  for (const Rung& r : kLadder)
    if (r.tile_m == tile_m && r.tile_n == tile_n) return &r;
  return nullptr;
}

constexpr double kFixupUs = 8.0;  // hand-over of fp32 partial tiles: write, wait, read, add (measured)

// stream_k: 0 data-parallel, 1 the tail's k-stages over all workers, S >= 2
// each tail tile over S workers.
static double tc_estimate_us(int dtype, int out_dtype, int64_t m, int64_t n, int64_t K, int tile_m, int tile_n,
                             int num_sms, int stream_k, int* grid_out) {
  const Rung* r = find_rung(tile_m, tile_n);
  const int cg = tile_m == 256 ? 2 : 1;
  const double esize = dtype == DGL_DTYPE_E4M3 ? 1.0 : 2.0;
  const int64_t tiles = ((m + tile_m - 1) / tile_m) * ((n + tile_n - 1) / tile_n);
  const int64_t units = std::max(1, num_sms / cg);  // CTAs or CTA pairs that run at once
  const int64_t groups = std::min<int64_t>(tiles, units);
  const int64_t waves = (tiles + groups - 1) / groups;
  const double k_stages = std::ceil(static_cast<double>(K) * esize / 128.0);
  const double tile_us = k_stages * r->stage_us + r->tile_us;
  double us = kLaunchUs + static_cast<double>(waves) * tile_us;
  if (stream_k) {
    const int64_t full = tiles / units;                       // whole waves, data-parallel
    const double tail_stages = stream_k >= 2 ? std::ceil(k_stages / stream_k)
                                             : static_cast<double>(tiles - full * units) * k_stages / units;
    us = kLaunchUs + static_cast<double>(full) * tile_us + tail_stages * r->stage_us + kFixupUs + r->tile_us;
  }
  const double hbm_us = operand_bytes(dtype, out_dtype, m, n, K) / (kHbmGBs * 1e3) + kLaunchUs;
  if (grid_out) *grid_out = static_cast<int>((stream_k ? units : groups) * cg);
  return std::max(us, hbm_us);
}

// Stream-K pays when the last wave is partial and each worker gets at least
// a few k-stages of the tail.
bool stream_k_eligible(int64_t m, int64_t n, int64_t K, int dtype, int tile_m, int tile_n, int num_sms) {
  if (tile_m == 64) return false;  // 64-row tiles: small problems, no partial-tile hand-over
  const int cg = tile_m == 256 ? 2 : 1;
  const int64_t tiles = ((m + tile_m - 1) / tile_m) * ((n + tile_n - 1) / tile_n);
  const int64_t units = std::max(1, num_sms / cg);
  const int64_t nk = (K * (dtype == DGL_DTYPE_E4M3 ? 1 : 2) + 127) / 128;
  const int64_t tail = tiles % units;
  return tail != 0 && tail * nk >= 4 * units;
}

// Split-K tail: with long K, each tile of a partial last wave that fills at
// most half the workers runs on S = floor(workers / tail) workers (at most 4),
// each taking an equal, tile-aligned range of its k-stages; the worker holding
// the first range adds the others' fp32 partials before the epilogue.  The
// wave of whole tiles before it is unchanged.  Needs at least one whole wave
// before the tail and 64 or more k-blocks of 128 bytes (16 or more per
// range): the hand-over of a partial tile costs about 8 us (measured at
// 4096^3: bf16, 64 k-blocks, 77.9 -> 76.4 us; E4M3, 32 k-blocks, 44.5 ->
// 47.1 us, a loss).  Short K takes the half tiles below.  Returns S, or 0.
int tail_split_ways(int64_t m, int64_t n, int64_t K, int dtype, int tile_m, int tile_n, int num_sms) {
  if (tile_m == 64) return 0;
  const int cg = tile_m == 256 ? 2 : 1;
  const int64_t tiles = ((m + tile_m - 1) / tile_m) * ((n + tile_n - 1) / tile_n);
  const int64_t units = std::max(1, num_sms / cg);
  const int64_t nk = (K * (dtype == DGL_DTYPE_E4M3 ? 1 : 2) + 127) / 128;
  const int64_t tail = tiles % units;
  if (tiles <= units || tail == 0 || nk < 64) return 0;
  int ways = static_cast<int>(std::min<int64_t>(4, units / tail));
  while (ways > 1 && nk / ways < 16) --ways;
  return ways >= 2 ? ways : 0;
}

// Split tail: a 256-wide tile's last, partial wave runs as half tiles when
// there is at least one full wave and the tail fills at most half the
// workers, so the halves still run at once.  Only for short K (at most 16
// k-blocks of 128 bytes): there a tile's fixed cost (fill, epilogue, store)
// dominates and halving it pays; with long K a half tile loads 3/4 of a full
// tile's bytes per k-block for half its MMA work and runs load-bound, and the
// split measured no faster (4096^3) or slower (8192^3).
bool split_tail_eligible(int64_t m, int64_t n, int64_t K, int dtype, int tile_m, int tile_n, int num_sms) {
  if (tile_n != 256 || tile_m == 64) return false;
  const int64_t nk = (K * (dtype == DGL_DTYPE_E4M3 ? 1 : 2) + 127) / 128;
  if (nk > 16) return false;
  const int cg = tile_m == 256 ? 2 : 1;
  const int64_t tiles = ((m + tile_m - 1) / tile_m) * ((n + tile_n - 1) / tile_n);
  const int64_t units = std::max(1, num_sms / cg);
  const int64_t tail = tiles % units;
  return tiles > units && tail > 0 && 2 * tail <= units;
}

int tc_tile_k(int dtype) { return dtype == DGL_DTYPE_E4M3 ? 128 : 64; }

int tc_stages(int tile_m, int tile_n) {
  const int cg = tile_m == 256 ? 2 : 1;
  const int stage = (tile_m == 64 ? 64 : 128) * 128 + tile_n / cg * 128;
  const int s = (232448 - 32768 - 512) / stage;
  return s < 8 ? s : 8;
}

bool tc_supported_tile(int tile_m, int tile_n) { return find_rung(tile_m, tile_n) != nullptr; }

void fill_tc_plan(int dtype, int out_dtype, int64_t m, int64_t n, int64_t K, int tile_m, int tile_n, int num_sms,
                  dgl_plan_info* out, int stream_k) {
  *out = dgl_plan_info{};
  out->path = DGL_PATH_TC;
  out->k_group = 1;
  out->tile_m = tile_m;
  out->tile_n = tile_n;
  out->tile_k = tc_tile_k(dtype);
  out->stages = tc_stages(tile_m, tile_n);
  out->cta_group = tile_m == 256 ? 2 : 1;
  tile_metrics(m, n, tile_m, tile_n, num_sms / out->cta_group, out);
  // stream_k: -2 the planner's default (a split-K tail where
  // tail_split_ways allows one), -1 the model decides between stream-K and
  // none, 0 none, 1 stream-K over all workers (if eligible), S >= 2 a split-K
  // tail over S workers per tile (if the tail allows it)
  out->split_tail = split_tail_eligible(m, n, K, dtype, tile_m, tile_n, num_sms) ? 1 : 0;
  const bool sk_ok = stream_k_eligible(m, n, K, dtype, tile_m, tile_n, num_sms);
  int grid = 0;
  out->est_us = tc_estimate_us(dtype, out_dtype, m, n, K, tile_m, tile_n, num_sms, 0, &grid);
  out->grid = grid;
  out->stream_k = 0;
  int ways = 0;
  if (stream_k == -2) {
    ways = tail_split_ways(m, n, K, dtype, tile_m, tile_n, num_sms);
  } else if (stream_k >= 2 && tile_m != 64) {
    const int cg = tile_m == 256 ? 2 : 1;
    const int64_t tiles = ((m + tile_m - 1) / tile_m) * ((n + tile_n - 1) / tile_n);
    const int64_t units = std::max(1, num_sms / cg);
    const int64_t tail = tiles % units;
    if (tail > 0 && tail * stream_k <= units) ways = stream_k;
  }
  if (ways >= 2) {
    int grid_sk = 0;
    out->est_us = tc_estimate_us(dtype, out_dtype, m, n, K, tile_m, tile_n, num_sms, ways, &grid_sk);
    out->grid = grid_sk;
    out->stream_k = ways;
    out->split_tail = 0;
  } else if (sk_ok && (stream_k == 1 || stream_k == -1)) {
    int grid_sk = 0;
    const double est_sk = tc_estimate_us(dtype, out_dtype, m, n, K, tile_m, tile_n, num_sms, 1, &grid_sk);
    if (stream_k == 1 || est_sk < 0.97 * out->est_us) {
      out->est_us = est_sk;
      out->grid = grid_sk;
      out->stream_k = 1;
      out->split_tail = 0;
    }
  }
}

int decode_parts(int64_t n, int num_sms) {
  // balanced parts of at most 128 rows, a multiple of the SM count when n allows
  const int64_t need = (n + 127) / 128;
  const int64_t waves = (need + num_sms - 1) / num_sms;
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(n, waves * num_sms)));
}

int decode_grid(int64_t n, int num_sms) { return std::min(decode_parts(n, num_sms), num_sms); }

void fill_decode_plan(int dtype, int out_dtype, int64_t m, int64_t n, int64_t K, int num_sms, dgl_plan_info* out) {
  *out = dgl_plan_info{};
  out->path = DGL_PATH_DECODE;
  out->tile_m = 16;
  out->tile_n = static_cast<int32_t>((n + decode_parts(n, num_sms) - 1) / decode_parts(n, num_sms));
  out->tile_k = dtype == DGL_DTYPE_E4M3 ? 128 : 64;
  out->cta_group = 1;
  out->grid = decode_grid(n, num_sms);
  out->num_tiles = decode_parts(n, num_sms);
  const int nk = static_cast<int>((K * (dtype == DGL_DTYPE_E4M3 ? 1 : 2) + 127) / 128);
  const int g = decode_group(out->tile_n, nk);
  out->k_group = g;
  const int ks = decode_ksteps(out->tile_n, nk, g);
  out->tile_k = ks * (dtype == DGL_DTYPE_E4M3 ? 128 : 64);
  out->stages = decode_stages(out->tile_n, ks, g);
  out->tile_eff = static_cast<double>(m) / 16.0;
  out->wq_eff = static_cast<double>(out->num_tiles) /
                (static_cast<double>((out->num_tiles + out->grid - 1) / out->grid) * out->grid);
  out->dim_eff = out->tile_eff * out->wq_eff;
  out->est_us = operand_bytes(dtype, out_dtype, m, n, K) / (kHbmGBs * 1e3) + kLaunchUs;
}

int decode_group(int rows_hi, int nk) {
  // The largest G <= 16 (a power of two) with rows_hi <= 128 / G that divides
  // the number of 128-byte K steps: G steps of a part fill one 128-row operand.
  if (nk <= 0) return 1;
  int g = 16;
  while (g > 1 && (rows_hi > 128 / g || nk % g != 0)) g >>= 1;
  return g;
}

int decode_plane_bytes(int rows_hi, int group) {
  return (group > 1 ? 128 / group : (rows_hi + 7) / 8 * 8) * 128;
}

int decode_stage_bytes(int rows_hi, int ksteps, int group) {
  return ksteps * (2048 + decode_plane_bytes(rows_hi, group));
}

int decode_stages(int rows_hi, int ksteps, int group) {
  const int s = 196608 / decode_stage_bytes(rows_hi, ksteps, group);
  return s < 32 ? s : 32;
}

int decode_ksteps(int rows_hi, int nk, int group) {
  // the widest stage (a multiple of the group) that still leaves at least
  // four in the ring
  int ks = group > 8 ? group : 8;
  while (ks > group && decode_stages(rows_hi, ks, group) < 4) ks >>= 1;
  return ks < nk ? ks : (nk > 0 ? nk : 1);
}

// Block-scaled FP4: one 128 x 256 tile on one CTA, a 3-stage ring of
// 128-byte (256-element) k-stages.  The estimate charges each stage's 48 KB of
// operands at the tile path's load rate, or HBM, whichever is slower.
void fill_mx_plan(int out_dtype, int64_t m, int64_t n, int64_t K, int num_sms, dgl_plan_info* out) {
  *out = dgl_plan_info{};
  out->path = DGL_PATH_TC;
  out->k_group = 1;
  out->tile_m = 128;
  out->tile_n = 256;
  out->tile_k = 256;
  out->stages = 3;
  out->cta_group = 1;
  tile_metrics(m, n, 128, 256, num_sms, out);
  const int64_t tiles = out->num_tiles;
  out->grid = static_cast<int>(std::min<int64_t>(tiles, num_sms));
  const int64_t waves = (tiles + num_sms - 1) / num_sms;
  const double k_stages = std::ceil(static_cast<double>(K) / 256.0);
  const double o = out_dtype == DGL_OUT_F32 ? 4.0 : 2.0;
  const double bytes = (static_cast<double>(m) + n) * K / 2.0 + (static_cast<double>(m) + n) * K / 32.0 +
                       static_cast<double>(m) * n * o;
  const double tc_us = kLaunchUs + static_cast<double>(waves) * (k_stages * 0.40 + 1.5);
  out->est_us = std::max(tc_us, bytes / (kHbmGBs * 1e3) + kLaunchUs);
}

void choose_plan(int dtype, int out_dtype, int64_t m, int64_t n, int64_t K, int num_sms, dgl_plan_info* out) {
  if (m <= 0 || n <= 0) {
    *out = dgl_plan_info{};
    out->path = DGL_PATH_EMPTY;
    return;
  }
  if (dtype == DGL_DTYPE_MXFP4) {
    fill_mx_plan(out_dtype, m, n, K, num_sms, out);
    return;
  }
  if (m <= kDecodeMaxM) {
    fill_decode_plan(dtype, out_dtype, m, n, K, num_sms, out);
    return;
  }
  for (const Pin& pin : kPins) {
    if (pin.dtype == dtype && pin.m == m && pin.n == n && pin.K == K) {
      fill_tc_plan(dtype, out_dtype, m, n, K, pin.tile_m, pin.tile_n, num_sms, out, -2);
      return;
    }
  }
  const double area = static_cast<double>(m) * static_cast<double>(n);
  const int64_t nk = (K * (dtype == DGL_DTYPE_E4M3 ? 1 : 2) + 127) / 128;
  auto offered = [&](const Rung& r) { return r.max_kb == 0 || nk <= r.max_kb; };
  bool any_pass = false;
  for (const Rung& r : kLadder) {
    if (!offered(r)) continue;
    const double padded = std::ceil(static_cast<double>(m) / r.tile_m) * r.tile_m *
                          std::ceil(static_cast<double>(n) / r.tile_n) * r.tile_n;
    if (padded <= 1.25 * area) any_pass = true;
  }
  bool have = false;
  dgl_plan_info best{};
  for (const Rung& r : kLadder) {
    if (!offered(r)) continue;
    const double padded = std::ceil(static_cast<double>(m) / r.tile_m) * r.tile_m *
                          std::ceil(static_cast<double>(n) / r.tile_n) * r.tile_n;
    if (any_pass && padded > 1.25 * area) continue;
    dgl_plan_info cand;
    fill_tc_plan(dtype, out_dtype, m, n, K, r.tile_m, r.tile_n, num_sms, &cand, -2);
    // ties go to the larger tile (later rungs are larger)
    if (!have || cand.est_us <= best.est_us * (1.0 + 1e-9)) {
      best = cand;
      have = true;
    }
  }
  *out = best;
}

}  // namespace dgl

namespace dgl {

bool tc_supported_epi_tile(int tile_m, int tile_n, bool gated) {
  if (!tc_supported_tile(tile_m, tile_n) || tile_m == 64 || (tile_n != 128 && tile_n != 256)) return false;
  return !gated || tile_m == 256;
}

void choose_linear_plan(int dtype, int out_dtype, int64_t m, int64_t n, int64_t K, bool gated, int num_sms,
                        dgl_plan_info* out) {
  if (!gated) {
    choose_plan(dtype, out_dtype, m, n, K, num_sms, out);
    if (out->path == DGL_PATH_TC && !tc_supported_epi_tile(out->tile_m, out->tile_n, false))
      fill_tc_plan(dtype, out_dtype, m, n, K, out->tile_m == 64 ? 128 : out->tile_m, out->tile_n == 64 ? 128 : out->tile_n,
                   num_sms, out, 0);
    return;
  }
  // gate and up rows side by side: a product with 2 n rows of B on CTA pairs
  dgl_plan_info best{};
  bool have = false;
  for (int tile_n : {256, 128}) {
    dgl_plan_info cand;
    fill_tc_plan(dtype, out_dtype, m, 2 * n, K, 256, tile_n, num_sms, &cand, 0);
    if (!have || cand.est_us < best.est_us * 0.97) {
      best = cand;
      have = true;
    }
  }
  *out = best;
}

}  // namespace dgl

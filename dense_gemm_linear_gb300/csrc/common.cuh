// Parameters shared by the host launcher and the kernels.
#pragma once

#include <cstdint>

namespace dgl {

// Bits OR-ed into the device status word when a bounded wait gives up (or a
// kernel finds its launch unusable and exits without work).
enum : int {
  STATUS_TIMEOUT_PRODUCER = 1,
  STATUS_TIMEOUT_MMA = 2,
  STATUS_TIMEOUT_EPILOGUE = 4,
  STATUS_TIMEOUT_DRAIN = 8,
  STATUS_TMEM_MISMATCH = 16,  // a CTA pair's tensor-memory allocations differ
  STATUS_TIMEOUT_FIXUP = 32,  // a stream-K partial tile never arrived
  STATUS_TIMEOUT_SCALES = 64, // block-scaled kernels: a scale slot was never released
  STATUS_SMEM_ALIGN = 128,    // dynamic shared memory not 1024-byte aligned: the kernel did nothing
};

// Programmatic dependent launch modes.  PDL_SERIAL: let the next kernel on
// the stream launch, then wait for the previous one to complete before any
// global access.  PDL_BATCH_HEAD (the first kernel of a batch of GEMMs whose
// operands were all written before the batch): wait first, then let the next
// launch, so no later kernel of the batch starts before that earlier work is
// done.  PDL_BATCH_NEXT (a later kernel of the batch): let the next launch and
// read operands at once; only the epilogue waits for the previous kernel,
// before its first global write, so every kernel of the batch completes after
// the one before it and writes C after it.
enum : int { PDL_SERIAL = 0, PDL_BATCH_HEAD = 1, PDL_BATCH_NEXT = 2 };

// Persistent tcgen05 tile kernel: problem and schedule.
struct TcParams {
  void* C;              // output, row pitch ldc elements
  int64_t ldc;
  int m, n, K;          // valid rows of A/C, valid rows of B (= columns of C), inner extent
  const float* sa;      // E4M3 only: per-row scale of A (m entries)
  const float* sb;      // E4M3 only: per-row scale of B (n entries)
  int tiles_m, tiles_n, num_tiles, num_kb;
  int group_m;          // tile raster: group_m row-tiles share each column sweep
  int c_tma;            // 1: C is written by TMA tensor stores (16-byte aligned pitch and base)
  int* status;          // device status word
  // Schedule.  `workers` CTAs (or CTA pairs) run at once.  Tiles below
  // dp_tiles run whole, worker w taking w, w + workers, ...  The remaining
  // tiles' k-stages ("units", tile-major) are split into `workers` equal
  // contiguous ranges (stream-K): a worker whose range starts inside a tile
  // writes its fp32 partial to its workspace slot and raises its flag; the
  // worker holding a tile's first k-stage adds the partials and stores C.
  int workers;
  int dp_tiles;
  int64_t sk_units;
  // Workers the stream-K units are split over: all of them, or (a split-K
  // tail) tail tiles x S, so that each tail tile's k-stages fall into S equal
  // ranges, one per worker, aligned to the tile.
  int sk_workers;
  float* ws;            // workers x CTAs-per-worker slots of 128 x BN fp32 partials
  int* flags;           // one per slot: 1 once its partial is written, 0 again once it was read
  // Linear-layer epilogue: y = act(acc (* scales) + bias[col]); gated (CTA
  // pairs only): B holds the gate rows, then the up rows from row n_up, and
  // y = act(gate + bias[col]) * (up + bias[n_up + col]).  sb and bias follow
  // B's rows.  bias may be null.
  const float* bias;
  int act;              // 0 identity, 1 GELU (x * Phi(x)), 2 SiLU (x * sigma(x))
  int gated;
  int n_up;
  // Operand majorness: 0 K-major (A [m][K], B [n][K]), 1 MN-major (A [K][m],
  // B [K][n]: the backward-pass layouts; bf16 only).
  int a_mn;
  int b_mn;
  // Split tail: the last, partial wave's tiles (from dp_tiles on) run as
  // half_tiles halves of BN / 2 columns each, one per worker.
  int half_tiles;
  // Block-scaled FP4 (MXFP4): E8M0 scales, K / 32 bytes per row of A (sfa, m
  // rows) and of B (sfb, n rows); K counts E2M1 elements.  sf_vec8: every
  // stage's 8 scale bytes of a row may be read as one aligned 8-byte word.
  const uint8_t* sfa;
  const uint8_t* sfb;
  int sf_vec8;
  // Bits OR-ed into the MMA instruction descriptor: an operand format other
  // than the kernel's own (W4A8: E2M1 in B's format field of a kind::f8f6f4
  // kernel, whose B tiles then hold packed 4-bit codes unpacked by TMA).
  uint32_t idesc_or;
  // B's transaction bytes per stage are its shared-memory bytes >> b_tx_shift:
  // 1 for packed 4-bit B, whose TMA copies count the bytes read from global
  // memory, half of what they write to shared memory
  int b_tx_shift;
  // k-stages of the worker's first tile whose A and B boxes are prefetched
  // into L2 before the wait for the previous kernel (0: none)
  int prefetch_stages;
  // Programmatic dependent launch (PDL_*): where the kernel waits for the
  // previous kernel on the stream and when it lets the next one launch
  int pdl_mode;
};

// Decode (m <= 16) kernel parameters.  A and B are read through tensor maps.
struct DecodeParams {
  const float* sa;
  const float* sb;
  void* C;
  int64_t ldc;
  int m, n;
  int row_bytes;        // K * element size
  int parts;            // B rows are cut into this many balanced parts
  int rows_hi;          // ceil(n / parts): parts of this size use the second B map
  int stages;           // ring depth
  int ksteps;           // 128-byte K steps per stage (a multiple of group)
  int group;            // K steps stacked into one 128-row MMA operand (1, 2, 4, 8, 16)
  int b_plane_bytes;    // one B slot: 128 / group rows (group 1: rows_hi rounded up to 8), x 128 bytes
  int stage_bytes;      // ksteps x (A box (2 KB) + B box)
  int* status;          // device status word
  const float* bias;    // linear-layer epilogue: bias per column of C, or null
  int act;              // 0 identity, 1 GELU, 2 SiLU
  uint32_t idesc_or;    // bits OR-ed into the MMA instruction descriptor (W4A8: E2M1 B rows)
  int b_tx_shift;       // B boxes' transaction bytes = shared-memory bytes >> b_tx_shift (1: packed 4-bit B)
  int prefetch_planes;  // K steps of the CTA's first part of B prefetched into L2 before the wait (0: none)
  // 1: A's map is 3-D, [K steps][m rows][128 bytes], with a box of 16 rows
  // (zero past m) by ksteps K steps (zero past K): one copy brings a stage's
  // A planes (K a whole number of 128-byte steps).  0: one 2-D box of m rows
  // per K step.
  int a3d;
  int pdl_mode;         // as in TcParams
};

// The activations of the linear-layer epilogue.
//   GELU(x) = x * Phi(x), Phi(x) = (1 + erf(x / sqrt 2)) / 2.  erf(z) for
//   z >= 0 is evaluated with formula 7.1.26 of Abramowitz and Stegun,
//   "Handbook of Mathematical Functions" (1964): with t = 1 / (1 + p z),
//   erf(z) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) e^{-z^2}, with an
//   absolute error below 1.5e-7; erf is odd, which gives z < 0.
//   SiLU(x) = x * sigma(x) = x / (1 + e^-x).
// Both use the hardware exponential and reciprocal: the epilogue evaluates
// one activation per output element and must stay shorter than the next
// tile's MMAs.
__device__ __forceinline__ float gelu_as7126(float x) {
  const float z = fabsf(x) * 0.70710678118654752f;
  const float t = __fdividef(1.0f, fmaf(0.3275911f, z, 1.0f));
  float poly = fmaf(1.061405429f, t, -1.453152027f);
  poly = fmaf(poly, t, 1.421413741f);
  poly = fmaf(poly, t, -0.284496736f);
  poly = fmaf(poly, t, 0.254829592f);
  poly *= t;
  const float tail = 0.5f * poly * __expf(-z * z);  // (1 - erf(z)) / 2 = Phi(-|x|)
  const float phi = x >= 0.0f ? 1.0f - tail : tail;
  return x * phi;
}

__device__ __forceinline__ float silu_fast(float x) {
  // e^-x overflows below x = -88; sigma(x) x is then below 1e-36 in size
  return x < -80.0f ? 0.0f * x : __fdividef(x, 1.0f + __expf(-x));
}

__device__ __forceinline__ float apply_act(int act, float x) {
  if (act == 1) return gelu_as7126(x);
  if (act == 2) return silu_fast(x);
  return x;
}

// One piece of a worker's schedule: k-stages [kb0, kb1) of one tile.
struct Segment {
  int tile, kb0, kb1;
  int half;  // 0: the whole tile; 1 / 2: its left / right half (BN / 2 columns)
};

__host__ __device__ inline int64_t sk_range_start(int64_t units, int workers, int w) {
  return units * w / workers;
}

// The worker whose stream-K range holds unit u.
__host__ __device__ inline int sk_worker_of(int64_t units, int workers, int64_t u) {
  int w = static_cast<int>(u * workers / units);
  while (w + 1 < workers && sk_range_start(units, workers, w + 1) <= u) ++w;
  while (w > 0 && sk_range_start(units, workers, w) > u) --w;
  return w;
}

// Walks worker w's segments in order: its data-parallel tiles, then (split
// tail) at most one half tile of the last wave, or (stream-K) its range of
// the last wave's k-stages: the units are cut into sk_workers equal ranges
// (0: one per worker), and workers from sk_workers on get none.  Every role
// of a CTA walks the same sequence.
struct SegmentIter {
  int w, workers, nk, dp_tiles, next_dp, half_tiles, next_half;
  int64_t u, u_end;
  __host__ __device__ SegmentIter(int worker, int num_workers, int num_kb, int dp, int64_t units, int halves = 0,
                                  int sk_workers = 0)
      : w(worker), workers(num_workers), nk(num_kb), dp_tiles(dp), next_dp(worker), half_tiles(halves),
        next_half(worker), u(0), u_end(0) {
    const int skw = sk_workers > 0 ? sk_workers : num_workers;
    if (units > 0 && worker < skw) {
      u = sk_range_start(units, skw, worker);
      u_end = sk_range_start(units, skw, worker + 1);
    }
  }
  __host__ __device__ bool next(Segment& s) {
    s.half = 0;
    if (next_dp < dp_tiles) {
      s.tile = next_dp;
      s.kb0 = 0;
      s.kb1 = nk;
      next_dp += workers;
      return true;
    }
    if (next_half < half_tiles) {
      s.tile = dp_tiles + next_half / 2;
      s.half = 1 + next_half % 2;
      s.kb0 = 0;
      s.kb1 = nk;
      next_half += workers;
      return true;
    }
    if (u < u_end) {
      const int64_t t = u / nk;
      s.tile = dp_tiles + static_cast<int>(t);
      s.kb0 = static_cast<int>(u - t * nk);
      const int64_t left = u_end - u;
      s.kb1 = static_cast<int>(left < nk - s.kb0 ? s.kb0 + left : nk);
      u += s.kb1 - s.kb0;
      return true;
    }
    return false;
  }
};

__host__ __device__ inline void tile_coords(int tile, int tiles_m, int tiles_n, int group_m, int& mb, int& nb) {
  const int per_group = group_m * tiles_n;
  const int g = tile / per_group;
  const int first_m = g * group_m;
  const int rest = tiles_m - first_m;
  const int gsize = rest < group_m ? rest : group_m;
  const int r = tile - g * per_group;
  mb = first_m + r % gsize;
  nb = r / gsize;
}

}  // namespace dgl

// Persistent, warp-specialised tcgen05 GEMM:  C[i,j] = sum_k A[i,k] B[j,k]
// (times sa[i] sb[j] for E4M3; with per-32-element block scales for MXFP4),
// fp32 accumulation in tensor memory.
//
// One CTA per SM (or one CTA pair per two SMs, 256-row tiles) walks a raster
// of 128 x BN output tiles.  Roles:
//   warp 0     TMA producer: fills an S-stage shared-memory ring with the
//              128 x 128-byte slice of A and the BN x 128-byte slice of B for
//              each k-stage.  The tensor maps are bounded at the valid rows
//              and at K, so rows past m or n and the k tail beyond K arrive as
//              zeros and the k-loop carries no predicate (the descriptor-bound
//              M edge of FlyDSL pull request 1303, applied to every extent).
//   warp 1     allocates tensor memory, then one thread issues tcgen05.mma
//              (four K=16 bf16, K=32 E4M3 or K=64 E2M1 steps per 128-byte
//              stage) into one of two TMEM accumulators and commits each stage
//              back to the producer's "empty" barrier.
//   warps 2-9  epilogue, two warps per TMEM lane quarter, each taking half
//              of the 32-column chunks of its 32 rows.  A warp reads its
//              chunks out of TMEM two at a time, releases the accumulator
//              after the last, and per chunk applies the E4M3 row/column
//              scales ("Gemm Optimization" guide, section 7.1:
//              acc * scale_a * scale_b), rounds to bf16 (or keeps
//              fp32), vector stores into a swizzled staging tile, and
//                - a TMA tensor store of the 32 x 32 tile when C's row pitch
//                  is 16-byte aligned (clipped at m and n by the tensor map:
//                  the C-descriptor bound of the FlyDSL change), or
//                - otherwise predicated stores from the staging tile with the
//                  row predicate i < m and column predicate j < n paid once
//                  per tile, outside the k-loop (that change's C-store
//                  predicate).
//              For bf16 C whose rows are not 16-byte aligned (N = 50257,
//              11007, 4095, ...) the quarter's two warps instead stage whole
//              tile rows, each shifted by its own misalignment, so every row's
//              16-byte-aligned body leaves in one bulk copy and only the
//              partial 16-byte units at its two ends take 2-byte stores.
//              The staging transpose is section 7.2's "CShuffle" idea: re-map
//              threads so each store covers contiguous columns of a row.
//   warps 10-13 (MXFP4 only) gather each stage's E8M0 scales into shared
//              memory for the MMA thread to copy into tensor memory.
// The two accumulators let the epilogue of tile t overlap the main loop of
// tile t+1 (the MXFP4 variant has one: see TcConfig).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"

namespace dgl {

// Ring depth that fills the 227 KB per-CTA budget left by the epilogue's
// staging area and the barriers (at most 8 stages).  The dynamic shared
// memory is declared 1024-byte aligned, so no alignment slack is reserved.
constexpr int tc_ring_stages(int stage_bytes, int staging_bytes) {
  const int s = (232448 - staging_bytes - 512) / stage_bytes;
  return s < 8 ? s : 8;
}

template <int BN_, bool FP8_, bool OUT_F32_, bool ROWSTG_, int CG_ = 1, bool EPI_ = false, bool MX_ = false,
          int BM_ = 128>
struct TcConfig {
  static constexpr int CG = CG_;                        // CTAs per MMA: 1, or 2 for a CTA pair (M = 256)
  // EPI: the linear-layer epilogue (bias, activation, and on CTA pairs the
  // gated up projection) is compiled in; plain GEMM variants leave it out.
  static constexpr bool EPI = EPI_;
  // Rows of C per CTA: 128, or 64 for the small rungs of the ladder (one CTA,
  // an M = 64 MMA).  An M = 64 accumulator puts row 16 q + r (r < 16) in
  // tensor-memory lane 32 q + r, so each epilogue warp of lane quarter q holds
  // 16 rows, in its threads 0-15.
  static constexpr int BM = BM_;
  static constexpr int WARP_ROWS = BM / 4;              // tile rows per lane quarter: 32, or 16
  static constexpr int TILE_M = BM * CG;                // rows of C per tile
  static constexpr int BN = BN_;                        // columns of C per tile
  static constexpr int B_ROWS = BN / CG;                // rows of B each CTA loads per stage
  static constexpr bool FP8 = FP8_;
  // MX: block-scaled FP4 (MXFP4).  A and B hold E2M1 codes two to a byte; each
  // 32 elements of K of a row share one E8M0 scale.  kind::mxf4 MMAs read the
  // scales from tensor memory.  Four more warps gather each stage's scales into
  // shared memory, and the MMA thread copies them into a ring of tensor-memory
  // slots after the accumulator.  128 x 256 tiles on one CTA, with a single
  // 256-column accumulator (the other 256 columns hold the scale ring); the
  // epilogue hands it back as soon as it has been read out.
  static constexpr bool MX = MX_;
  static constexpr bool OUT_F32 = OUT_F32_;
  // ROWSTG: bf16 C whose rows are not 16-byte aligned.  The epilogue stages
  // whole tile rows, shifted by each row's misalignment, so the aligned body
  // of every row leaves in one bulk copy.
  static constexpr bool ROWSTG = ROWSTG_;
  static_assert(!(ROWSTG && OUT_F32), "row staging is the bf16-output path");
  static_assert(CG == 1 || CG == 2, "one CTA or a CTA pair");
  static constexpr int ROW_BYTES = 128;                 // one 128-byte swizzle span of K per stage
  static constexpr int BK = FP8 || MX ? 128 : 64;       // tensor-map elements (K) per stage: 128 bytes
  static constexpr int MMA_K_BYTES = 32;                // K=16 bf16, K=32 E4M3 or K=64 E2M1 per instruction
  static constexpr int MMAS_PER_STAGE = ROW_BYTES / MMA_K_BYTES;
  static constexpr int A_STAGE_BYTES = BM * ROW_BYTES;
  static constexpr int B_STAGE_BYTES = B_ROWS * ROW_BYTES;
  static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
  static constexpr int EPI_WARPS = 8;
  static constexpr int CHUNKS = BN / 32;                // 32-column chunks per tile row
  // two warps share a lane quarter: the first takes chunks [0, CB0), the
  // second [CB0, CHUNKS) (4 + 3 of a 224-wide tile's 7)
  static constexpr int CB0 = (CHUNKS + 1) / 2;
  static constexpr int CHUNKS_PER_WARP = CHUNKS / 2;
  static constexpr int OUT_BYTES = OUT_F32 ? 4 : 2;
  static constexpr int STG_ROW = 32 * OUT_BYTES;        // 32 x 32 staging row: 64 B (bf16) or 128 B (fp32)
  static constexpr int STG_BYTES = 32 * STG_ROW;        // one 32 x 32 staging tile: 2 KB (bf16) or 4 KB (fp32)
  // whole-row staging: BN bf16 + 16 bytes of shift room; the pitch is an odd
  // multiple of 16 bytes so rows spread over the banks
  static constexpr int ROW_PITCH = BN * 2 + 16;
  static constexpr int STG_TOTAL = ROWSTG ? 4 * 32 * ROW_PITCH : EPI_WARPS * 4096;
  // MX: per stage, 512-byte scale atoms for each 128 rows and each 4 k-blocks:
  // 2 of A's, 2 per 128 rows of B
  static constexpr int SCALE_ATOMS = MX ? 2 + 2 * (BN / 128) : 0;
  static constexpr int SCALE_STAGE_BYTES = 512 * SCALE_ATOMS;
  static constexpr int STAGES = tc_ring_stages(STAGE_BYTES + SCALE_STAGE_BYTES, STG_TOTAL);
  static constexpr int SCALE_WARPS = MX ? 4 : 0;
  static constexpr int THREADS = 64 + EPI_WARPS * 32 + SCALE_WARPS * 32;
  // fp32 accumulators of BN columns: two, so the epilogue of one tile
  // overlaps the main loop of the next, or one with MX 128 x 256 tiles
  static constexpr int ACC_BUFS = MX && BN == 256 ? 1 : 2;
  // a 224-wide accumulator is placed 256 columns apart (allocations are
  // powers of two)
  static constexpr int ACC_STRIDE = BN == 224 ? 256 : BN;
  static constexpr int TMEM_COLS = MX ? 512 : 2 * ACC_STRIDE;
  // MX scale ring: slot s holds stage s's scale atoms, 4 columns each
  static constexpr int SCALE_COL0 = ACC_BUFS * BN;
  static constexpr int SCALE_SLOT_COLS = 4 * SCALE_ATOMS;
  static constexpr int BAR_BYTES = 8 * (2 * STAGES + 6) + 8 + 32;
  // stream-K: one CTA's fp32 partial tile, and how many fit in the ring
  static constexpr int SLOT_BYTES = 128 * BN * 4;
  static constexpr int RING_SLOTS = STAGES * STAGE_BYTES / SLOT_BYTES;
  // fix-up staging per epilogue warp: 2 KB pieces, two of them when room allows
  static constexpr int FX_WARP_BYTES = ROWSTG ? 16 * ROW_PITCH : 4096;
  static constexpr int FX_BUFS = FX_WARP_BYTES >= 4096 ? 2 : 1;
  static constexpr int SMEM_BYTES =
      STAGES * (STAGE_BYTES + SCALE_STAGE_BYTES) + STG_TOTAL + BAR_BYTES;
  static_assert(BN == 64 || BN == 128 || BN == 256 || (BN == 224 && CG == 2 && !EPI && !MX),
                "tile widths of the ladder (224: plain GEMM on CTA pairs)");
  static_assert(BM == 128 || (BM == 64 && CG == 1 && !EPI && !MX), "64-row tiles: one CTA, plain GEMM");
  static_assert(STAGES >= 3, "ring too shallow");
  static_assert((ROW_PITCH / 16) % 2 == 1, "row pitch: odd multiple of 16 bytes");
  static_assert(TMEM_COLS == 128 || TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation: power of two");
  static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
  static_assert(!MX || ((BN == 128 || BN == 256) && CG == 1 && !FP8 && !EPI), "block-scaled FP4: 128-row tiles, one CTA");
  static_assert(!MX || SCALE_COL0 + STAGES * SCALE_SLOT_COLS <= TMEM_COLS, "scale ring fits in tensor memory");
  static_assert(B_STAGE_BYTES % 1024 == 0, "B stage tiles stay 1024-byte aligned");
  // stream-K (partial tiles handed over through a workspace) runs on the
  // 128-row tiles only; the host never splits a 64-row tile's k-stages
  static constexpr bool STREAM_K = BM == 128;
  static_assert(RING_SLOTS >= 1 || !STREAM_K, "a partial tile fits in the ring");
  static_assert(FX_WARP_BYTES >= 2048 && FX_WARP_BYTES % 16 == 0, "fix-up staging piece");
};

// Byte offset of 16-byte unit `c16` of staging row `r`, in the layout a TMA
// store with the 64-byte (bf16 rows) or 128-byte (fp32 rows) swizzle reads.
template <int STG_ROW>
__device__ __forceinline__ uint32_t stg_offset(int r, int c16) {
  if constexpr (STG_ROW == 64)
    return static_cast<uint32_t>(r * 64 + ((c16 ^ ((r >> 1) & 3)) << 4));
  else
    return static_cast<uint32_t>(r * 128 + ((c16 ^ (r & 7)) << 4));
}

// Stores NW packed words (2 NW bf16 values, value 2i in the low half of w[i])
// to shared memory so that value j lands at byte a + D + 2 j: a is 16-byte
// aligned and D (the global row's misalignment) is even and below 16.  The
// 16-byte words that the values fill completely go out as 16-byte stores;
// only the partial words at the two ends take 4- and 2-byte stores.  With
// one thread per staged row and rows 16-byte aligned at an odd multiple of
// 16 bytes apart, every 8-lane phase of a 16-byte store covers all 32 banks,
// where 4-byte stores at a common column put four lanes on each bank.
//   q = D / 4 words of offset, and x[i], the 4 bytes landing at a + 4 q + 4 i,
//   is w[i] when D % 4 == 0, else the high half of w[i - 1] and the low half
//   of w[i]; 16-byte word s (16 s .. 16 s + 15) then holds x[4 s - q .. 4 s + 3 - q].
template <int NW>
__device__ __forceinline__ void sts_row_shifted(uint32_t a, const uint32_t (&w)[NW], int D) {
  static_assert(NW % 4 == 0 && NW >= 8, "whole 16-byte words");
  const int q = D >> 2;
  const uint32_t sel = (D & 2) ? 0x5432u : 0x7654u;
  uint32_t x[NW + 1];
  x[0] = __byte_perm(0u, w[0], sel);
#pragma unroll
  for (int i = 1; i < NW; ++i) x[i] = __byte_perm(w[i - 1], w[i], sel);
  x[NW] = __byte_perm(w[NW - 1], 0u, sel);
  auto pick = [&](int k) -> uint32_t {  // x[k - q], k a compile-time index >= 3
    return q == 0 ? x[k] : q == 1 ? x[k - 1] : q == 2 ? x[k - 2] : x[k - 3];
  };
  // full words s = 1 .. NW / 4 - 1 (word 0 is full only when D == 0)
#pragma unroll
  for (int sw = 1; sw < NW / 4; ++sw)
    sts_v4(a + 16 * sw, pick(4 * sw), pick(4 * sw + 1), pick(4 * sw + 2), pick(4 * sw + 3));
  // head: bytes D .. 15 of word 0 are x[0 .. 3 - q] (x[0]'s high half only when D % 4 == 2)
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (i + q <= 3) {
      const uint32_t addr = a + 4 * (q + i);
      if (i == 0 && (D & 2))
        sts_u16(addr + 2, x[0] >> 16);
      else
        sts_u32(addr, x[i]);
    }
  }
  // tail: bytes 0 .. D - 1 of word NW / 4 are x[NW - q .. NW - 1], then x[NW]'s low half
  const uint32_t t0 = a + 4 * NW;
  if (q >= 1) sts_u32(t0, q == 1 ? x[NW - 1] : q == 2 ? x[NW - 2] : x[NW - 3]);
  if (q >= 2) sts_u32(t0 + 4, q == 2 ? x[NW - 1] : x[NW - 2]);
  if (q >= 3) sts_u32(t0 + 8, x[NW - 1]);
  if (D & 2) sts_u16(t0 + 4 * q, x[NW] & 0xFFFFu);
}

// Operand tiles in shared memory.  A K-major operand (rows of K contiguous)
// arrives as one TMA box of BK elements by `rows` rows.  An MN-major operand
// (stored [K][MN], MN contiguous: the backward-pass layouts) arrives as
// rows / 64 boxes of 64 MN elements by BK = 64 K rows, 8 KB each, placed one
// after another; each box is a column of 128-byte swizzle atoms (8 K rows by
// 64 MN elements) at a 1024-byte stride.  (MN-major operands are bf16 only.)
constexpr int MN_BOX_BYTES = 64 * 64 * 2;
constexpr int MN_K_STEP_BYTES = 2 * 1024;  // one bf16 MMA's K = 16: two 8-row atoms

// k0: the stage's first K element; row0: its first row (K-major) or MN index (MN-major).
__device__ __forceinline__ void load_operand(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int k0, int row0,
                                             int rows, int mn_major, uint64_t pol) {
  if (!mn_major) {
    tma_load_2d(dst, map, bar, k0, row0, pol);
    return;
  }
  for (int i = 0; i < rows / 64; ++i) tma_load_2d(dst + i * MN_BOX_BYTES, map, bar, row0 + 64 * i, k0, pol);
}

__device__ __forceinline__ void load_operand_pair(uint8_t* dst, const CUtensorMap* map, uint32_t leader_bar, int k0,
                                                  int row0, int rows, int mn_major, uint64_t pol) {
  if (!mn_major) {
    tma_load_2d_pair(dst, map, leader_bar, k0, row0, pol);
    return;
  }
  for (int i = 0; i < rows / 64; ++i)
    tma_load_2d_pair(dst + i * MN_BOX_BYTES, map, leader_bar, row0 + 64 * i, k0, pol);
}

// The worker's k-stages in schedule order, one (tile row, tile column,
// k-stage) at a time: the segments of SegmentIter, flattened.
struct StageIter {
  SegmentIter it;
  Segment sg;
  int kb = 0, kb1 = 0, mb = 0, nb = 0;
  int tiles_m, tiles_n, group_m;
  __device__ StageIter(int worker, const TcParams& prm)
      : it(worker, prm.workers, prm.num_kb, prm.dp_tiles, prm.sk_units, prm.half_tiles, prm.sk_workers),
        tiles_m(prm.tiles_m),
        tiles_n(prm.tiles_n), group_m(prm.group_m) {}
  __device__ bool next(int& mb_out, int& nb_out, int& kb_out) {
    while (kb >= kb1) {
      if (!it.next(sg)) return false;
      tile_coords(sg.tile, tiles_m, tiles_n, group_m, mb, nb);
      kb = sg.kb0;
      kb1 = sg.kb1;
    }
    mb_out = mb;
    nb_out = nb;
    kb_out = kb++;
    return true;
  }
};

// The 8 E8M0 scale bytes of k-blocks 8 kb .. 8 kb + 7 of row r, as two
// little-endian words (k-blocks 8 kb .. + 3, then + 4 .. + 7).  Rows past
// `rows` and k-blocks past `nkblk` read as 127 (a scale of 1): their operand
// elements are the tensor maps' zero fill.
__device__ __forceinline__ void scale_words(const uint8_t* sf, int rows, int r, int kb, int nkblk, int vec8,
                                            uint32_t& lo, uint32_t& hi) {
  lo = hi = 0x7F7F7F7Fu;
  const int k0 = kb * 8;
  if (vec8) {
    // one predicated 8-byte load: the thread does not wait for it here
    ldg_pred_v2(sf + static_cast<int64_t>(r < rows ? r : 0) * nkblk + k0, r < rows, lo, hi);
    return;
  }
  if (r >= rows) return;
  const uint8_t* row = sf + static_cast<int64_t>(r) * nkblk;
  uint32_t b[8];
#pragma unroll
  for (int t = 0; t < 8; ++t) b[t] = k0 + t < nkblk ? row[k0 + t] : 0x7Fu;
  lo = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
  hi = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
}

// Next accumulator buffer and its barrier phase: alternate between two, or
// reuse the only one.
template <int BUFS>
__device__ __forceinline__ void next_acc(uint32_t& acc, uint32_t& acc_phase) {
  if constexpr (BUFS == 2) {
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1;
  } else {
    acc_phase ^= 1;
  }
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmC,
                   const TcParams p) {
  constexpr int BM = Cfg::BM, BN = Cfg::BN, STAGES = Cfg::STAGES, CG = Cfg::CG;
  // The 128-byte-swizzled operand tiles need 1024-byte alignment, which the
  // declaration requests; a launch that did not get it reports and exits
  // (every CTA of a pair sees the same layout, so both leave together).  It
  // still completes only after the previous kernel on the stream, as a kernel
  // that ran would.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(p.status, STATUS_SMEM_ALIGN);
    griddep_wait();
    return;
  }
  uint8_t* sA = smem_raw;
  uint8_t* sB = sA + STAGES * Cfg::A_STAGE_BYTES;
  uint8_t* sSc = sB + STAGES * Cfg::B_STAGE_BYTES;       // MX scale slots (none otherwise)
  uint8_t* sStg = sSc + STAGES * Cfg::SCALE_STAGE_BYTES; // 1024-aligned: stage sizes are multiples of 1 KB
  uint64_t* full = reinterpret_cast<uint64_t*>(sStg + Cfg::STG_TOTAL);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* fixbar = drain + 1;                          // stream-K: partial tiles landed in the ring
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fixbar + 1);
  volatile int* qflag = reinterpret_cast<volatile int*>(tmem_slot + 1);  // 8 epilogue-warp flags

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA pair: rank 0 (the leader) issues the MMAs and owns the barriers the
  // MMA waits on; each CTA loads its own 128 rows of A and B_ROWS rows of B
  // and stores its own 128 rows of C.
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
  const int cluster_id = blockIdx.x / CG;  // the worker index of the schedule (p.workers == gridDim.x / CG)

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // the (leader's) producer's expect-tx arrival, and with MX one arrival
      // per scale warp once the stage's scales are in shared memory
      mbar_init(&full[s], 1 + Cfg::SCALE_WARPS);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], Cfg::EPI_WARPS * CG);
    }
    mbar_init(drain, 1);
    mbar_init(fixbar, 1);
    fence_mbarrier_init();
    fence_proxy_async_shared();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (p.half_tiles) tma_prefetch_desc(&tmBh);
    if (p.c_tma) tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    if constexpr (CG == 2) {
      tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before_sync();
  if constexpr (CG == 2)
    cluster_sync();  // barriers of both CTAs are initialised before either signals the other
  else
    __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  if (warp == 0 && lane == 0 && p.prefetch_stages > 0 && !p.a_mn && !p.b_mn) {
    // While the previous kernel on the stream finishes, warm L2 with the first
    // k-stages of this CTA's first tile.  The prefetch only moves lines
    // into L2, the point where every SM's global writes land, so what the
    // loads read after the wait below is current whatever the previous kernel
    // wrote.
    SegmentIter it0(cluster_id, p.workers, p.num_kb, p.dp_tiles, p.sk_units, p.half_tiles, p.sk_workers);
    Segment s0;
    if (it0.next(s0) && !s0.half) {
      int mb, nb;
      tile_coords(s0.tile, p.tiles_m, p.tiles_n, p.group_m, mb, nb);
      const int a_row = mb * Cfg::TILE_M + static_cast<int>(rank) * BM;
      const int b_row = (Cfg::EPI && CG == 2 && p.gated) ? (rank == 0 ? 0 : p.n_up) + nb * Cfg::B_ROWS
                                                         : nb * BN + static_cast<int>(rank) * Cfg::B_ROWS;
      const int kb1 = min(s0.kb1, s0.kb0 + min(STAGES, p.prefetch_stages));
      for (int kb = s0.kb0; kb < kb1; ++kb) {
        tma_prefetch_l2_2d(&tmA, kb * Cfg::BK, a_row);
        tma_prefetch_l2_2d(&tmB, kb * Cfg::BK, b_row);
      }
    }
  }
  // set-up touched no global data: let the next kernel launch, then wait for
  // the previous one before reading operands or writing C (a later GEMM of a
  // batch reads its operands at once and waits in the epilogue)
  if (p.pdl_mode == PDL_BATCH_HEAD) {
    griddep_wait();
    griddep_launch_dependents();
  } else {
    griddep_launch_dependents();
    if (p.pdl_mode == PDL_SERIAL) griddep_wait();
  }

  int fail = 0;
  if constexpr (CG == 2) {
    // the leader's MMAs write this CTA's tensor memory at the leader's address
    if (threadIdx.x == 0 && rank != 0) {
      uint32_t leader_base;
      asm volatile("ld.shared::cluster.u32 %0, [%1];"
                   : "=r"(leader_base)
                   : "r"(mapa_shared(smem_u32(tmem_slot), 0))
                   : "memory");
      if (leader_base != tmem_base) fail = STATUS_TMEM_MISMATCH;
    }
  }
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      SegmentIter it(cluster_id, p.workers, p.num_kb, p.dp_tiles, p.sk_units, p.half_tiles, p.sk_workers);
      Segment sg;
      while (!fail && it.next(sg)) {
        int mb, nb;
        tile_coords(sg.tile, p.tiles_m, p.tiles_n, p.group_m, mb, nb);
        const int a_row = mb * Cfg::TILE_M + static_cast<int>(rank) * BM;
        // gated pairs: the leader loads gate rows, the peer the matching up rows
        // half tiles: each CTA loads its BN / (2 CG) rows of the half through
        // the half-height map (tmBh), and the stage carries fewer bytes
        const int b_row = (Cfg::EPI && CG == 2 && p.gated) ? (rank == 0 ? 0 : p.n_up) + nb * Cfg::B_ROWS
                          : sg.half ? nb * BN + (sg.half - 1) * (BN / 2) + static_cast<int>(rank) * (Cfg::B_ROWS / 2)
                                    : nb * BN + static_cast<int>(rank) * Cfg::B_ROWS;
        const CUtensorMap* tmb = sg.half ? &tmBh : &tmB;
        const int b_rows = sg.half ? Cfg::B_ROWS / 2 : Cfg::B_ROWS;
        // a stage's transaction bytes: what the copies read from global
        // memory (packed 4-bit B lands in twice its size of shared memory)
        const uint32_t stage_bytes =
            Cfg::A_STAGE_BYTES + ((sg.half ? Cfg::B_STAGE_BYTES / 2 : Cfg::B_STAGE_BYTES) >> p.b_tx_shift);
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          const bool ok = mbar_wait(&empty[stage], phase ^ 1);
          if (!ok) {
            fail = STATUS_TIMEOUT_PRODUCER;
            break;
          }
          if constexpr (CG == 2) {
            // Both CTAs' loads complete on the leader's barrier; the leader
            // alone announces the pair's bytes.  A peer's bytes may land
            // before that announcement: the transaction count goes negative
            // for a moment and the phase still waits for the leader's arrival.
            const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
            if (rank == 0) mbar_arrive_expect_tx(&full[stage], stage_bytes * CG);
            load_operand_pair(sA + stage * Cfg::A_STAGE_BYTES, &tmA, fb, kb * Cfg::BK, a_row, BM, p.a_mn, pol);
            load_operand_pair(sB + stage * Cfg::B_STAGE_BYTES, p.b_mn ? &tmB : tmb, fb, kb * Cfg::BK, b_row, b_rows,
                              p.b_mn, pol);
          } else {
            mbar_arrive_expect_tx(&full[stage], stage_bytes);
            load_operand(sA + stage * Cfg::A_STAGE_BYTES, &tmA, &full[stage], kb * Cfg::BK, a_row, BM, p.a_mn, pol);
            load_operand(sB + stage * Cfg::B_STAGE_BYTES, p.b_mn ? &tmB : tmb, &full[stage], kb * Cfg::BK, b_row, b_rows,
                         p.b_mn, pol);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Copies still in flight land before this CTA may exit.  One CTA waits
      // for the completion of its last STAGES loads; in a pair the loads land
      // on the leader's barriers, so each producer waits instead for the MMA
      // to have consumed its last STAGES stages (which implies they landed).
      // Both are already complete on the normal path.
      const int64_t first = issued > STAGES ? issued - STAGES : 0;
      for (int64_t q = first; q < issued; ++q) {
        const uint32_t par = static_cast<uint32_t>((q / STAGES) & 1);
        const bool ok = CG == 2 ? mbar_wait(&empty[q % STAGES], par) : mbar_wait(&full[q % STAGES], par);
        if (!ok) fail |= STATUS_TIMEOUT_DRAIN;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && rank == 0) {
      // MN-major operands set the instruction's transpose bits (15: A, 16: B)
      const uint32_t idesc_major = (p.a_mn ? 1u << 15 : 0u) | (p.b_mn ? 1u << 16 : 0u) | p.idesc_or;
      const uint32_t idesc_full = idesc_f32acc(Cfg::FP8 ? 0u : 1u, Cfg::TILE_M, BN) | idesc_major;
      const uint32_t idesc_half = idesc_f32acc(Cfg::FP8 ? 0u : 1u, Cfg::TILE_M, BN / 2) | idesc_major;
      // Shared-memory descriptors differ only in their low word: the address
      // field (bits 0-13) and the leading offset (bits 16-29: unused for a
      // K-major tile, 8192 bytes between an MN-major tile's 64-element
      // boxes).  Each MMA's pair is then two 32-bit adds, which keeps the
      // single issuing thread ahead of the tensor pipe.
      const uint32_t a_lo0 = smem_desc_sw128_lo(smem_u32(sA)) + (p.a_mn ? ((8192u >> 4) - 1u) << 16 : 0u);
      const uint32_t b_lo0 = smem_desc_sw128_lo(smem_u32(sB)) + (p.b_mn ? ((8192u >> 4) - 1u) << 16 : 0u);
      const uint32_t sc_lo0 = Cfg::MX ? smem_desc_rows16_lo(smem_u32(sSc)) : 0u;  // MX scale atoms
      const uint32_t a_kstep = (p.a_mn ? MN_K_STEP_BYTES : Cfg::MMA_K_BYTES) >> 4;
      const uint32_t b_kstep = (p.b_mn ? MN_K_STEP_BYTES : Cfg::MMA_K_BYTES) >> 4;
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool issued_any = false;
      SegmentIter it(cluster_id, p.workers, p.num_kb, p.dp_tiles, p.sk_units, p.half_tiles, p.sk_workers);
      Segment sg;
      while (!fail && it.next(sg)) {
        const bool ok = mbar_wait(&tempty[acc], acc_phase ^ 1);
        if (!ok) {
          fail = STATUS_TIMEOUT_MMA;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * Cfg::ACC_STRIDE;
        const uint32_t idesc = sg.half ? idesc_half : idesc_full;  // a half tile: N = BN / 2
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          // (MX: the stage's scales are in shared memory too)
          const bool ok2 = mbar_wait(&full[stage], phase);
          if (!ok2) {
            fail = STATUS_TIMEOUT_MMA;
            break;
          }
          tc_fence_after_sync();
          if constexpr (Cfg::MX) {
            // the stage's 512-byte scale atoms into its tensor-memory slot,
            // atom a to columns 4 a .. 4 a + 3; the MMAs below run after
            const uint32_t sc_lo = sc_lo0 + static_cast<uint32_t>((stage * Cfg::SCALE_STAGE_BYTES) >> 4);
            const uint32_t tcol = tmem_base + Cfg::SCALE_COL0 + stage * Cfg::SCALE_SLOT_COLS;
#pragma unroll
            for (int a = 0; a < Cfg::SCALE_ATOMS; ++a)
              tmem_cp_32x128b_warpx4(tcol + 4 * a, desc_rows16_from_lo(sc_lo + 32 * a));
          }
          const uint32_t a_lo = a_lo0 + static_cast<uint32_t>((stage * Cfg::A_STAGE_BYTES) >> 4);
          const uint32_t b_lo = b_lo0 + static_cast<uint32_t>((stage * Cfg::B_STAGE_BYTES) >> 4);
          const uint32_t acc_first = kb != sg.kb0 ? 1u : 0u;
#pragma unroll
          for (int k = 0; k < Cfg::MMAS_PER_STAGE; ++k) {
            const uint64_t ad = desc_sw128_from_lo(a_lo + k * a_kstep);
            const uint64_t bd = desc_sw128_from_lo(b_lo + k * b_kstep);
            const uint32_t accumulate = k != 0 ? 1u : acc_first;
            if constexpr (CG == 2) {
              if constexpr (Cfg::FP8)
                umma_e4m3_pair(d_tmem, ad, bd, idesc, accumulate);
              else
                umma_bf16_pair(d_tmem, ad, bd, idesc, accumulate);
            } else {
              if constexpr (Cfg::MX) {
                // instruction k covers k-blocks 2k, 2k + 1: word k / 2 of the
                // slot's atoms, starting at byte 2 (k % 2).  Atoms: A's k-blocks
                // 0-3 and 4-7, then for each of those B's rows 0-127 (and
                // 128-255).  One N = BN instruction reads B's scales for rows
                // 128 r .. 128 r + 127 from the r-th 4-column group after the
                // address it is given (measured: the parity tests pass with it).
                const uint32_t id = static_cast<uint32_t>(k & 1) * 2u;
                const uint32_t slot = tmem_base + Cfg::SCALE_COL0 + stage * Cfg::SCALE_SLOT_COLS;
                constexpr int NH = BN / 128;
                umma_mxf4(d_tmem, ad, bd, idesc_mxf4(Cfg::TILE_M, BN, id, id), slot + 4 * (k >> 1),
                          slot + 8 + 4 * NH * (k >> 1), accumulate);
              } else if constexpr (Cfg::FP8) {
                umma_e4m3(d_tmem, ad, bd, idesc, accumulate);
              } else {
                umma_bf16(d_tmem, ad, bd, idesc, accumulate);
              }
            }
          }
          issued_any = true;
          if constexpr (CG == 2)
            umma_commit_pair_multicast(&empty[stage], 0x3);  // both CTAs' producers may refill
          else
            umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (fail) break;
        if constexpr (CG == 2)
          umma_commit_pair_multicast(&tfull[acc], 0x3);  // both CTAs' epilogues
        else
          umma_commit(&tfull[acc]);
        next_acc<Cfg::ACC_BUFS>(acc, acc_phase);
      }
      // Every MMA this thread issued has finished before TMEM is released.
      if (issued_any) {
        if constexpr (CG == 2)
          umma_commit_pair_multicast(drain, 0x1);
        else
          umma_commit(drain);
        if (!mbar_wait(drain, 0)) fail |= STATUS_TIMEOUT_DRAIN;
      }
    }
  } else if (warp < 2 + Cfg::EPI_WARPS) {
    // ------------------------------------------------------------ epilogue
    // C, the split schedule's workspace and its flags are written here only
    if (p.pdl_mode == PDL_BATCH_NEXT) griddep_wait();
    const int e = warp - 2;                 // 0..7
    const int q = warp & 3;                 // TMEM lanes 32q .. 32q+31 are reachable from this warp
    const int half = e >> 2;                // this warp takes chunks [c_first, c_first + nc)
    constexpr int CPW = Cfg::CHUNKS_PER_WARP;
    constexpr bool EVEN = Cfg::CHUNKS % 2 == 0;
    const int c_first = EVEN ? half * CPW : (half ? Cfg::CB0 : 0);
    const int nc = EVEN ? CPW : (half ? Cfg::CHUNKS - Cfg::CB0 : Cfg::CB0);
    uint8_t* stg = Cfg::ROWSTG ? sStg + q * 32 * Cfg::ROW_PITCH : sStg + e * 4096;
    const uint32_t stg_addr = smem_u32(stg);
    uint32_t acc = 0, acc_phase = 0, fx_phase = 0;
    SegmentIter it(cluster_id, p.workers, p.num_kb, p.dp_tiles, p.sk_units, p.half_tiles, p.sk_workers);
    Segment sg;
    while (it.next(sg)) {
      int mb, nb;
      tile_coords(sg.tile, p.tiles_m, p.tiles_n, p.group_m, mb, nb);
      // all lanes decide together: tcgen05.ld below is warp-collective
      bool ready = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase));
      if constexpr (Cfg::ROWSTG) {
        // The quarter's two warps meet at named barriers below, so they must
        // also agree on giving up.  This barrier also orders the previous
        // tile's bulk copies (finished reading the staging rows) before the
        // rows are rewritten.
        if (half == 0) bulk_wait_read0();
        if (lane == 0) qflag[2 * q + half] = ready ? 1 : 0;
        named_bar_sync(1 + q, 64);
        ready = qflag[2 * q] != 0 && qflag[2 * q + 1] != 0;
      }
      if (!ready) {
        fail = STATUS_TIMEOUT_EPILOGUE;
        break;
      }
      tc_fence_after_sync();
      const int row0 = mb * Cfg::TILE_M + static_cast<int>(rank) * BM + q * Cfg::WARP_ROWS;
      const bool row_lane = lane < Cfg::WARP_ROWS;  // this thread holds a row of the tile
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * Cfg::ACC_STRIDE;

      // ---- stream-K: a segment that does not hold the tile's first k-stage
      // hands its fp32 partial tile over through the workspace; the segment
      // that does adds every partial into tensor memory before the usual
      // epilogue.  Slot layout (per CTA of the worker): float4 number
      // ((c * 4 + q) * 8 + t) * 32 + lane holds columns 32c + 4t .. 32c + 4t + 3
      // of slab row 32q + lane, so each warp's 32 x 32 chunk is 4 KB of
      // contiguous memory, written and read with bulk copies.
      if (Cfg::STREAM_K && sg.kb0 > 0) {
        uint8_t* slot = reinterpret_cast<uint8_t*>(p.ws) + (static_cast<int64_t>(cluster_id) * CG + rank) * Cfg::SLOT_BYTES;
        const uint32_t fx = Cfg::ROWSTG ? stg_addr + half * Cfg::FX_WARP_BYTES : stg_addr;
        int piece = 0;
#pragma unroll 1
        for (int u = 0; u < nc; ++u) {
          const int c = c_first + u;
          uint32_t v[32];
          tmem_ld_32x32b_x32(t_row + c * 32, v);
          tmem_ld_wait();
          reg_fence(v);
#pragma unroll
          for (int h = 0; h < 2; ++h, ++piece) {
            const uint32_t buf = fx + (Cfg::FX_BUFS == 2 ? (piece & 1) * 2048 : 0);
            // the copy that last read this buffer (or an earlier tile's store) is done with it
            if (lane == 0) {
              if (Cfg::FX_BUFS == 2 && piece > 0)
                bulk_wait_read1();
              else
                bulk_wait_read0();
            }
            __syncwarp();
#pragma unroll
            for (int tt = 0; tt < 4; ++tt) {
              const int t = 4 * h + tt;
              sts_v4(buf + (tt * 32 + lane) * 16, v[4 * t], v[4 * t + 1], v[4 * t + 2], v[4 * t + 3]);
            }
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) {
              bulk_store_1d(slot + (c * 4 + q) * 4096 + h * 2048, buf, 2048);
              bulk_commit();
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          if constexpr (CG == 2)
            mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
          else
            mbar_arrive(&tempty[acc]);
          bulk_wait0();  // this warp's pieces are in global memory
          fence_proxy_async_global();
          __threadfence();
        }
        named_bar_sync(5, Cfg::EPI_WARPS * 32);  // every epilogue warp's pieces are written
        if (warp == 2 && lane == 0) st_release_gpu(p.flags + cluster_id * CG + rank, 1);
        next_acc<Cfg::ACC_BUFS>(acc, acc_phase);
        continue;
      }
      if (Cfg::STREAM_K && sg.kb1 < p.num_kb) {
        // Finisher: the tile's other k-stages belong to workers cluster_id + 1
        // .. w_last (an empty range holds none).  This is the worker's last
        // segment, so every MMA has finished and the operand ring is free:
        // partial tiles are bulk-copied into it, RING_SLOTS at a time.
        const int64_t t_rel = sg.tile - p.dp_tiles;
        const int w_last = sk_worker_of(p.sk_units, p.sk_workers, (t_rel + 1) * p.num_kb - 1);
        auto nonempty = [&](int w) {
          return sk_range_start(p.sk_units, p.sk_workers, w) != sk_range_start(p.sk_units, p.sk_workers, w + 1);
        };
        const uint32_t ring = smem_u32(sA);
        int wc = cluster_id + 1;
        while (true) {
          while (wc <= w_last && !nonempty(wc)) ++wc;
          if (wc > w_last) break;
          const int w_first = wc;
          int nb = 0;
          for (; wc <= w_last && nb < Cfg::RING_SLOTS; ++wc)
            if (nonempty(wc)) ++nb;
          if (warp == 2 && lane == 0) {
            int i = 0;
            for (int w = w_first; w < wc; ++w) {
              if (!nonempty(w)) continue;
              if (!wait_flag_gpu(p.flags + w * CG + rank, 1)) fail |= STATUS_TIMEOUT_FIXUP;
              if (i == 0) {
                fence_proxy_async_global();
                fence_proxy_async_shared();
                mbar_arrive_expect_tx(fixbar, static_cast<uint32_t>(nb * Cfg::SLOT_BYTES));
              }
              const uint8_t* src =
                  reinterpret_cast<const uint8_t*>(p.ws) + (static_cast<int64_t>(w) * CG + rank) * Cfg::SLOT_BYTES;
              for (int off = 0; off < Cfg::SLOT_BYTES; off += 32768)
                bulk_load_1d(ring + i * Cfg::SLOT_BYTES + off, src + off, min(32768, Cfg::SLOT_BYTES - off), fixbar);
              ++i;
            }
          }
          if (!mbar_wait(fixbar, fx_phase)) fail |= STATUS_TIMEOUT_FIXUP;
          fx_phase ^= 1;
          if (warp == 2 && lane == 0) {
            // the partials are in shared memory: clear their flags for the
            // next launch on this workspace
            for (int w = w_first; w < wc; ++w)
              if (nonempty(w)) p.flags[w * CG + rank] = 0;
          }
#pragma unroll 1
          for (int u = 0; u < nc; ++u) {
            const int c = c_first + u;
            uint32_t v[32];
            tmem_ld_32x32b_x32(t_row + c * 32, v);
            tmem_ld_wait();
            reg_fence(v);
#pragma unroll 1
            for (int i = 0; i < nb; ++i) {
              const uint32_t src = ring + i * Cfg::SLOT_BYTES + ((c * 4 + q) * 8 * 32 + lane) * 16;
#pragma unroll
              for (int t = 0; t < 8; ++t) {
                const float4 x = lds_v4f(src + t * 512);
                v[4 * t] = __float_as_uint(__uint_as_float(v[4 * t]) + x.x);
                v[4 * t + 1] = __float_as_uint(__uint_as_float(v[4 * t + 1]) + x.y);
                v[4 * t + 2] = __float_as_uint(__uint_as_float(v[4 * t + 2]) + x.z);
                v[4 * t + 3] = __float_as_uint(__uint_as_float(v[4 * t + 3]) + x.w);
              }
            }
            tmem_st_32x32b_x32(t_row + c * 32, v);
          }
          tmem_st_wait();
          named_bar_sync(5, Cfg::EPI_WARPS * 32);  // the ring is read before the next copies land in it
        }
      }

      // Output columns of this tile: BN, or BN / 2 when a gated pair's MMA
      // computes the gate (leader's B rows) and up (peer's B rows) halves.
      const bool gated = Cfg::EPI && CG == 2 && p.gated != 0;
      const int out_w = (gated || sg.half) ? BN / 2 : BN;
      const int ocol0 = sg.half ? nb * BN + (sg.half - 1) * (BN / 2) : nb * out_w;
      float row_scale = 0.0f;
      if constexpr (Cfg::FP8) row_scale = (row_lane && row0 + lane < p.m) ? p.sa[row0 + lane] : 0.0f;
      // row staging (bf16 C, rows not 16-byte aligned): this thread's row
      const int row = row0 + lane;
      const int ncols = min(out_w, p.n - ocol0);
      const int L = (Cfg::ROWSTG && row_lane && row < p.m) ? 2 * ncols : 0;  // valid bytes of the row's segment
      uint8_t* rowp = L > 0 ? reinterpret_cast<uint8_t*>(static_cast<__nv_bfloat16*>(p.C) +
                                                         static_cast<int64_t>(row) * p.ldc + ocol0)
                            : nullptr;
      const int delta = static_cast<int>(reinterpret_cast<uintptr_t>(rowp) & 15);
      const uint32_t srow = stg_addr + lane * Cfg::ROW_PITCH + delta;  // staged byte 0 of the segment
      uint32_t buf = 0;

      // Rounds output chunk `oc` (columns ocol0 + 32 oc ..; this thread's row
      // in v) and stores it, or stages it for the row copy below.
      auto emit = [&](uint32_t(&v)[32], int oc) {
        if constexpr (Cfg::ROWSTG) {
          // ---- stage whole rows, shifted by each row's misalignment
          uint32_t w[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(v[2 * t]), __uint_as_float(v[2 * t + 1]));
            w[t] = *reinterpret_cast<uint32_t*>(&h2);
          }
          sts_row_shifted<16>(srow - delta + 64 * oc, w, delta);
        } else {
          // bf16 chunks alternate between two 2 KB staging tiles, so a chunk's
          // TMA store may still be reading one while the next chunk fills the
          // other; fp32 chunks fill the whole 4 KB tile.
          const int col0 = ocol0 + oc * 32;
          uint8_t* stg_u = stg + buf * Cfg::STG_BYTES;
          const uint32_t stg_addr_u = stg_addr + buf * Cfg::STG_BYTES;
          // the store that last used this staging tile has finished reading it
          if (p.c_tma && lane == 0) {
            if constexpr (Cfg::OUT_F32)
              bulk_wait_read0();
            else
              bulk_wait_read1();
          }
          __syncwarp();
          // this thread's row (lane) of the 32 x 32 chunk -> staging, 16 bytes at a time
          if constexpr (Cfg::OUT_F32) {
#pragma unroll
            for (int c16 = 0; c16 < 8; ++c16)
              sts_v4(stg_addr_u + stg_offset<Cfg::STG_ROW>(lane, c16), v[4 * c16], v[4 * c16 + 1], v[4 * c16 + 2],
                     v[4 * c16 + 3]);
          } else {
#pragma unroll
            for (int c16 = 0; c16 < 4; ++c16) {
              uint32_t w[4];
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                __nv_bfloat162 h2 =
                    __floats2bfloat162_rn(__uint_as_float(v[8 * c16 + 2 * t]), __uint_as_float(v[8 * c16 + 2 * t + 1]));
                w[t] = *reinterpret_cast<uint32_t*>(&h2);
              }
              sts_v4(stg_addr_u + stg_offset<Cfg::STG_ROW>(lane, c16), w[0], w[1], w[2], w[3]);
            }
          }
          // A TMA store writes whole 16-byte units of a row, so a chunk that
          // ends inside one (n * element size not a multiple of 16) takes the
          // predicated path instead.
          const bool tma_ok = p.c_tma && (col0 + 32 <= p.n || (p.n * Cfg::OUT_BYTES) % 16 == 0);
          if (tma_ok) {
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0 && row0 < p.m && col0 < p.n) {
              tma_store_2d(&tmC, stg_u, col0, row0);
              bulk_commit();
            }
          } else {
            __syncwarp();
            // one row per step, a column per lane
            const int col = col0 + lane;
#pragma unroll 4
            for (int rr = 0; rr < Cfg::WARP_ROWS; ++rr) {
              const int grow = row0 + rr;
              if (grow < p.m && col < p.n) {
                if constexpr (Cfg::OUT_F32) {
                  const float y =
                      *reinterpret_cast<const float*>(stg_u + stg_offset<128>(rr, lane >> 2) + (lane & 3) * 4);
                  static_cast<float*>(p.C)[static_cast<int64_t>(grow) * p.ldc + col] = y;
                } else {
                  const uint16_t y =
                      *reinterpret_cast<const uint16_t*>(stg_u + stg_offset<64>(rr, lane >> 3) + (lane & 7) * 2);
                  reinterpret_cast<uint16_t*>(p.C)[static_cast<int64_t>(grow) * p.ldc + col] = y;
                }
              }
            }
            __syncwarp();
          }
          if constexpr (!Cfg::OUT_F32) buf ^= 1u;
        }
      };
      auto hand_back = [&]() {
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          if constexpr (CG == 2)
            mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));  // the leader's MMA waits on it
          else
            mbar_arrive(&tempty[acc]);
        }
      };

      bool gated_done = false;
      if constexpr (BN == 256) {
        if (sg.half) {
          // ---- a half tile of the split tail: BN / 2 columns in TMEM
          // columns [0, BN / 2); this warp takes CPW / 2 of their chunks
          gated_done = true;
          constexpr int HCPW = CPW / 2;
#pragma unroll 1
          for (int u = 0; u < HCPW; ++u) {
            const int oc = half * HCPW + u;
            uint32_t v[32];
            tmem_ld_32x32b_x32(t_row + oc * 32, v);
            tmem_ld_wait();
            reg_fence(v);
            if (u + 1 == HCPW) hand_back();
            const int col = ocol0 + oc * 32 + lane;
            if constexpr (Cfg::FP8) {
              const float col_scale = col < p.n ? p.sb[col] : 0.0f;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                v[j] = __float_as_uint((__uint_as_float(v[j]) * row_scale) * __shfl_sync(0xffffffffu, col_scale, j));
            }
            if constexpr (Cfg::EPI) {
              if (p.act != 0 || p.bias != nullptr) {
                const float b = (p.bias && col < p.n) ? p.bias[col] : 0.0f;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  v[j] = __float_as_uint(apply_act(p.act, __uint_as_float(v[j]) + __shfl_sync(0xffffffffu, b, j)));
              }
            }
            emit(v, oc);
          }
        }
      }
      if constexpr (Cfg::EPI && CG == 2) {
        if (gated && !gated_done) {
          gated_done = true;
          // ---- gated linear layer: output chunk oc combines gate chunk oc with
          // up chunk oc + CHUNKS / 2; this warp takes CPW / 2 output chunks.
          constexpr int OCPW = CPW / 2 > 0 ? CPW / 2 : 1;
  #pragma unroll 1
          for (int u = 0; u < OCPW; ++u) {
            const int oc = half * OCPW + u;
            uint32_t g[32], v[32];
            tmem_ld_32x32b_x32(t_row + oc * 32, g);
            tmem_ld_32x32b_x32(t_row + (oc + Cfg::CHUNKS / 2) * 32, v);
            tmem_ld_wait();
            reg_fence(g);
            reg_fence(v);
            if (u + 1 == OCPW) hand_back();
            const int col = ocol0 + oc * 32 + lane;
            const bool in = col < p.n;
            float sg = 1.0f, su = 1.0f, bg = 0.0f, bu = 0.0f;
            if constexpr (Cfg::FP8) {
              sg = in ? p.sb[col] : 0.0f;
              su = in ? p.sb[p.n_up + col] : 0.0f;
            }
            if (p.bias && in) {
              bg = p.bias[col];
              bu = p.bias[p.n_up + col];
            }
  #pragma unroll
            for (int j = 0; j < 32; ++j) {
              float x = __uint_as_float(g[j]), y = __uint_as_float(v[j]);
              if constexpr (Cfg::FP8) {
                x = (x * row_scale) * __shfl_sync(0xffffffffu, sg, j);
                y = (y * row_scale) * __shfl_sync(0xffffffffu, su, j);
              }
              x = apply_act(p.act, x + __shfl_sync(0xffffffffu, bg, j));
              y += __shfl_sync(0xffffffffu, bu, j);
              v[j] = __float_as_uint(x * y);
            }
            emit(v, oc);
          }
        }
      }
      if (!gated_done) {
        // The warp's share of the accumulator (chunks c_first .. c_first + nc
        // - 1) is read two chunks at a time, which bounds the registers it
        // holds; the buffer goes back to the MMA once the last chunk has been
        // read.
        const bool epi = Cfg::EPI && (p.act != 0 || p.bias != nullptr);
        auto group = [&](auto g_const, int c0, bool last) {
          constexpr int G = decltype(g_const)::value;
          uint32_t r[G][32];
#pragma unroll
          for (int uu = 0; uu < G; ++uu) tmem_ld_32x32b_x32(t_row + (c0 + uu) * 32, r[uu]);
          tmem_ld_wait();
#pragma unroll
          for (int uu = 0; uu < G; ++uu) reg_fence(r[uu]);
          if (last) hand_back();

          if constexpr (Cfg::FP8) {
#pragma unroll
            for (int uu = 0; uu < G; ++uu) {
              const int col0 = ocol0 + (c0 + uu) * 32;
              const float col_scale = (col0 + lane < p.n) ? p.sb[col0 + lane] : 0.0f;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                r[uu][j] = __float_as_uint((__uint_as_float(r[uu][j]) * row_scale) *
                                           __shfl_sync(0xffffffffu, col_scale, j));
            }
          }
          if (Cfg::EPI && epi) {
            // linear-layer epilogue: bias per column, then the activation
#pragma unroll
            for (int uu = 0; uu < G; ++uu) {
              const int col = ocol0 + (c0 + uu) * 32 + lane;
              const float b = (p.bias && col < p.n) ? p.bias[col] : 0.0f;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                r[uu][j] = __float_as_uint(
                    apply_act(p.act, __uint_as_float(r[uu][j]) + __shfl_sync(0xffffffffu, b, j)));
            }
          }
          if constexpr (Cfg::ROWSTG) {
            // the G chunks are adjacent in the row: stage them as one span,
            // so only its two ends take narrow stores
            uint32_t w[16 * G];
#pragma unroll
            for (int uu = 0; uu < G; ++uu) {
#pragma unroll
              for (int t = 0; t < 16; ++t) {
                __nv_bfloat162 h2 =
                    __floats2bfloat162_rn(__uint_as_float(r[uu][2 * t]), __uint_as_float(r[uu][2 * t + 1]));
                w[16 * uu + t] = *reinterpret_cast<uint32_t*>(&h2);
              }
            }
            sts_row_shifted<16 * G>(srow - delta + 64 * c0, w, delta);
          } else {
#pragma unroll
            for (int uu = 0; uu < G; ++uu) emit(r[uu], c0 + uu);
          }
        };
#pragma unroll
        for (int g0 = 0; g0 < Cfg::CB0; g0 += 2) {
          if (g0 >= nc) break;
          if (g0 + 2 <= nc)
            group(std::integral_constant<int, 2>{}, c_first + g0, g0 + 2 == nc);
          else
            group(std::integral_constant<int, 1>{}, c_first + g0, true);
        }
      }

      if constexpr (Cfg::ROWSTG) {
        // Each staged row's 16-byte-aligned body leaves in one bulk copy (the
        // quarter's first warp, a row per lane); the partial 16-byte units at
        // its two ends, in 2-byte stores (the second warp).
        fence_proxy_async_shared();
        named_bar_sync(1 + q, 64);
        if (half == 0) {
          if (L > 0) {
            const int head = min(L, (16 - delta) & 15);
            const int body = ((L - head) >> 4) << 4;
            if (body > 0) {
              bulk_store_1d(rowp + head, srow + head, static_cast<uint32_t>(body));
              bulk_commit();
            }
          }
        } else {
          // The quarter's 32 rows have 64 end units.  Eight lanes take one
          // unit, a bf16 each, so a store instruction writes four units and
          // each unit's bytes leave as one request, where one lane per row
          // would need up to three 2-, 4- or 8-byte stores per unit.
#pragma unroll 1
          for (int pass = 0; pass < 16; ++pass) {
            const int u = 4 * pass + (lane >> 3);  // unit: row u / 2 of the quarter, its head (even) or tail (odd)
            const int r = u >> 1;
            const int urow = row0 + r;
            const int uL = (r < Cfg::WARP_ROWS && urow < p.m) ? 2 * ncols : 0;  // valid bytes of that row
            uint8_t* up = reinterpret_cast<uint8_t*>(static_cast<__nv_bfloat16*>(p.C) +
                                                     static_cast<int64_t>(uL > 0 ? urow : 0) * p.ldc + ocol0);
            const int ud = static_cast<int>(reinterpret_cast<uintptr_t>(up) & 15);
            const int uhead = min(uL, (16 - ud) & 15);
            const int ubody = ((uL - uhead) >> 4) << 4;
            // byte x of the row's segment: the head unit spans x = -ud .. 15 - ud
            const int x = (u & 1) ? uhead + ubody + 2 * (lane & 7) : 2 * (lane & 7) - ud;
            if (x >= 0 && x < ((u & 1) ? uL : uhead))
              *reinterpret_cast<uint16_t*>(up + x) =
                  static_cast<uint16_t>(lds_u16(stg_addr + r * Cfg::ROW_PITCH + ud + x));
          }
        }
      }
      next_acc<Cfg::ACC_BUFS>(acc, acc_phase);
    }
    if ((Cfg::ROWSTG ? half == 0 : (p.c_tma && lane == 0))) bulk_wait0();
  }

  if constexpr (Cfg::MX) {
    if (warp >= 2 + Cfg::EPI_WARPS) {
      // ---------------------------------------------------------- scale warps (MX)
      // Stage s's E8M0 scales go to shared-memory slot s once the MMAs (and
      // the copy) that read the slot's previous contents are done: the
      // stage's "empty" barrier.  A slot holds 512-byte atoms (A's k-blocks
      // 0-3 and 4-7 of the stage, then B's per 128-row half).  Row 32 j + l of the
      // tile has its four scale bytes at atom offset 16 l + 4 j, which is the
      // layout the MMA thread's 32-lane, 128-bit copy replicated to the four
      // lane quarters turns into the one kind::mxf4 reads: lane 32 w + l,
      // column 4 a + j holds row 32 j + l's word of atom a.  Warp q handles
      // rows 32 q .. 32 q + 31 of A and of B, then arrives on the stage's
      // full barrier beside the producer, so the MMA thread waits once.
      const int q = warp & 3;
      const int nkblk = p.K / 32;
      // Loads run SD stages ahead of the shared-memory stores (a register
      // queue, unrolled so every index is static); they are predicated rather
      // than selected afterwards, so nothing waits for them before the store.
      constexpr int SD = 4;
      constexpr int NH = BN / 128;
      StageIter ahead(cluster_id, p), cur(cluster_id, p);
      uint32_t w[SD][Cfg::SCALE_ATOMS];
      // atom order: A's k-blocks 0-3, 4-7, then B's: for k-blocks 0-3 each
      // 128-row half, then for 4-7 each half
      auto gather = [&](uint32_t(&x)[Cfg::SCALE_ATOMS], int mb, int nb, int kb) {
        scale_words(p.sfa, p.m, mb * BM + 32 * q + lane, kb, nkblk, p.sf_vec8, x[0], x[1]);
#pragma unroll
        for (int h = 0; h < NH; ++h)
          scale_words(p.sfb, p.n, nb * BN + 128 * h + 32 * q + lane, kb, nkblk, p.sf_vec8, x[2 + h], x[2 + NH + h]);
      };
      int mb, nb, kb;
#pragma unroll
      for (int d = 0; d < SD; ++d)
        if (ahead.next(mb, nb, kb)) gather(w[d], mb, nb, kb);
      uint32_t stage = 0, phase = 0;
      bool more = true;
      while (more && !fail) {
#pragma unroll
        for (int d = 0; d < SD; ++d) {
          if (!more || fail) break;
          if (!cur.next(mb, nb, kb)) {
            more = false;
            break;
          }
          const bool ok = __all_sync(0xffffffffu, mbar_wait(&empty[stage], phase ^ 1));
          if (!ok) {
            fail = STATUS_TIMEOUT_SCALES;
            break;
          }
          const uint32_t slot = smem_u32(sSc + stage * Cfg::SCALE_STAGE_BYTES) + 16 * lane + 4 * q;
#pragma unroll
          for (int a = 0; a < Cfg::SCALE_ATOMS; ++a) sts_u32(slot + 512 * a, w[d][a]);
          fence_proxy_async_shared();  // the tensor-memory copy reads the slot through the async proxy
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
          if (ahead.next(mb, nb, kb)) gather(w[d], mb, nb, kb);
        }
      }
    }
  }

  if (fail) atomicOr(p.status, fail);
  tc_fence_before_sync();
  if constexpr (CG == 2)
    cluster_sync();  // neither CTA leaves while the other may still touch its memory
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    if constexpr (CG == 2)
      tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace dgl

// Decode-shape GEMM (m <= 16 rows of A), the memory-bound case: with L = 1
// the token count M of the MLP GEMM is the batch size B ("GEMM analysis in
// TraceLens", section "Prefill versus decode"), so each call streams the whole
// weight matrix B once for a handful of rows of A, and the arithmetic
// intensity is about m flop per byte of B ("Gemm Optimization" guide,
// section 8.3: small M is memory-bound).
//
// Design: a TMA streaming pipeline with the operand roles swapped.
//   * B's rows are cut into P balanced parts (each floor(n/P) or ceil(n/P)
//     rows, at most 128); a CTA walks parts blockIdx.x, +gridDim.x, ...
//   * warp 0 streams each part through a shared-memory ring of ~192 KB.  A
//     stage holds `ks` consecutive 128-byte steps of K ("planes"): per plane
//     one TMA box of the part's B rows, and A's rows for all the stage's
//     planes in one 3-D box (or, when K ends inside a plane, one box of A's m
//     rows per plane; bytes past K arrive as zeros), all with the 128-byte
//     swizzle.  The planes' loads go out back to back so adjacent pieces of
//     each B row reach the memory system together.
//   * warp 1 issues tcgen05.mma with the part's B rows as the 128-row operand
//     and A's 16 rows as the N = 16 operand: D[row of B][row of A] accumulates
//     in tensor memory (two 16-column buffers, alternating by part).  The MMA
//     is asynchronous, so no warp waits on a chain of dependent products and
//     the stream is limited only by memory.  Rows of either operand past its
//     box (B rows past the part, A rows past m) read whatever the ring holds
//     there; each feeds only its own row or column of D, which is never
//     stored.
//   * A part of at most 128 / G rows (G = 2, 4, 8 or 16) fills the 128-row
//     operand with G consecutive K steps instead: slot s (rows s R .. s R +
//     R - 1, R = 128 / G) holds the part's rows at K step k0 + s, and the
//     N = 16 G operand holds A's rows at the same G steps, slot s at columns
//     16 s .. 16 s + 15.  The diagonal blocks D[slot s][A slot s] accumulate
//     the part's products over the K steps congruent to s; the off-diagonal
//     blocks mix K steps and are never read.  One MMA then does the work of
//     G, which matters because a small-N MMA costs about the same whatever
//     its valid rows.
//   * warps 2-5 read D (lane = row of B, 16 columns = rows of A), scale
//     (E4M3), round and store C[i][j]: for each i the warp's 32 lanes write 32
//     consecutive columns.  With G > 1 they first add the G diagonal blocks
//     through shared memory, in slot order.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace dgl {

constexpr int DEC_MAX_ROWS = 128;                  // rows of B per part (the MMA's M)
constexpr int DEC_THREADS = 192;                   // producer, MMA, 4 epilogue warps
constexpr int DEC_MAX_STAGES = 32;
constexpr int DEC_RING_BYTES = 196608;             // 192 KB of stages
// The 128-row MMA operand of the ring's last plane reaches up to 16 KB past
// that plane's start; the slack keeps every such read inside the allocation.
constexpr int DEC_SLACK_BYTES = 16384;
// G > 1: the 128 stacked rows' 16 partial sums, padded to 17 floats a row so
// that a warp's 32 rows fall in 32 different banks
constexpr int DEC_RED_STRIDE = 17;
constexpr int DEC_RED_BYTES = 128 * DEC_RED_STRIDE * 4;
// dynamic shared memory: the ring, the barriers and (stacked K steps only)
// the partial sums
__host__ __device__ constexpr int dec_smem_bytes(bool stack) {
  return 1024 + DEC_RING_BYTES + DEC_SLACK_BYTES + 8 * (2 * DEC_MAX_STAGES + 7) + 8 + (stack ? DEC_RED_BYTES : 0);
}
constexpr int DEC_A_BOX_BYTES = 16 * 128;
// Independent accumulators per part: the four MMAs of a 128-byte K step go to
// separate 16 G-column TMEM accumulators (four, or 16 / G when G >= 8, so
// that two buffers fit in 512 columns), so consecutive MMAs do not wait on
// one another's result; the epilogue adds them.
__host__ __device__ constexpr int dec_nacc(int group) { return group >= 8 ? 16 / group : 4; }

// Row range of part `part` of n rows cut into `parts` balanced pieces.
__device__ __forceinline__ void part_rows(int part, int parts, int n, int& r0, int& r1) {
  r0 = static_cast<int>(static_cast<int64_t>(part) * n / parts);
  r1 = static_cast<int>(static_cast<int64_t>(part + 1) * n / parts);
}

// STACK: G = p.group > 1 K steps per MMA; otherwise G = 1 at compile time.
template <bool FP8, bool OUT_F32, bool STACK>
__global__ void __launch_bounds__(DEC_THREADS, 1)
    decode_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB_lo,
                       const __grid_constant__ CUtensorMap tmB_hi, const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + DEC_RING_BYTES + DEC_SLACK_BYTES);
  uint64_t* empty = full + DEC_MAX_STAGES;
  uint64_t* tfull = empty + DEC_MAX_STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* redbar = drain + 1;  // G > 1: partial sums written [0], read [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(redbar + 2);
  float* red = reinterpret_cast<float*>(redbar + 3);
  const int stages = p.stages;
  const int stage_bytes = p.stage_bytes;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(drain, 1);
    mbar_init(&redbar[0], 4);
    mbar_init(&redbar[1], 4);
    fence_mbarrier_init();
    fence_proxy_async_shared();
  }
  const int G = STACK ? p.group : 1;
  const int nacc = dec_nacc(G);
  const int acc_cols = nacc * 16 * G;            // one accumulator buffer (of two)
  const uint32_t tmem_cols = 2 * acc_cols;       // 128, 256 or 512: a power of two
  if (warp == 1) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const int nk = (p.row_bytes + 127) >> 7;   // 128-byte steps of K
  // The producer's set-up for its first part (row range, cache policies) is
  // done before the wait for the previous kernel, since it reads no global
  // memory (a %globaltimer trace put the 64-bit part arithmetic at about
  // 0.35 us between the wait and the first load).
  int first_r0 = 0, first_r1 = 0;
  uint64_t pol_a = 0, pol_b = 0;
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB_lo);
    tma_prefetch_desc(&tmB_hi);
    part_rows(blockIdx.x, p.parts, p.n, first_r0, first_r1);
    pol_a = l2_policy_evict_last();
    pol_b = l2_policy_evict_first();
    // While the previous kernel on the stream finishes, warm L2 with the first
    // K steps of this CTA's first part of B.  The prefetch only moves
    // lines into L2, the point where every SM's global writes land, so what
    // the loads read after the wait below is current whatever the previous
    // kernel wrote.
    const CUtensorMap* mb = (first_r1 - first_r0) == p.rows_hi ? &tmB_hi : &tmB_lo;
    const int planes = min(nk, p.prefetch_planes);
    for (int j = 0; j < planes; ++j) tma_prefetch_l2_2d(mb, j * (FP8 ? 128 : 64), first_r0);
  }
  // a later GEMM of a batch reads its operands at once and waits in the
  // epilogue (PDL_BATCH_NEXT); see common.cuh
  if (p.pdl_mode == PDL_BATCH_HEAD) {
    griddep_wait();
    griddep_launch_dependents();
  } else {
    griddep_launch_dependents();
    if (p.pdl_mode == PDL_SERIAL) griddep_wait();
  }

  const int ks = p.ksteps;                    // planes per stage
  const int b_plane = p.b_plane_bytes;        // one B box, rows rounded up to 8, x 128 bytes
  const int a_bytes = ks * DEC_A_BOX_BYTES;   // A planes first, then B planes
  int fail = 0;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int kstep = FP8 ? 128 : 64;  // elements per 128 bytes
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      for (int part = blockIdx.x; part < p.parts && !fail; part += gridDim.x) {
        int r0 = first_r0, r1 = first_r1;
        if (part != static_cast<int>(blockIdx.x)) part_rows(part, p.parts, p.n, r0, r1);
        const CUtensorMap* mb = (r1 - r0) == p.rows_hi ? &tmB_hi : &tmB_lo;
        // A box of m rows + B box of the part's rows, counted as the bytes the
        // copies read (packed 4-bit B: 64 a row for 128 bytes of shared memory)
        const uint32_t tx = p.m * 128 + ((r1 - r0) * 128 >> p.b_tx_shift);
        for (int kb0 = 0; kb0 < nk; kb0 += ks) {
          if (!mbar_wait(&empty[stage], phase ^ 1)) {
            fail = STATUS_TIMEOUT_PRODUCER;
            break;
          }
          const int planes = min(ks, nk - kb0);
          uint8_t* sbase = ring + stage * stage_bytes;
          if (p.a3d) {
            // A's box always carries ks planes of 16 rows (zeros past m and K);
            // a small part's stage then costs one copy for A instead of ks
            mbar_arrive_expect_tx(&full[stage], ks * DEC_A_BOX_BYTES + planes * (tx - p.m * 128));
            tma_load_3d(sbase, &tmA, &full[stage], 0, 0, kb0, pol_a);
            for (int j = 0; j < planes; ++j)
              tma_load_2d(sbase + a_bytes + j * b_plane, mb, &full[stage], (kb0 + j) * kstep, r0, pol_b);
          } else {
            mbar_arrive_expect_tx(&full[stage], tx * planes);
            for (int j = 0; j < planes; ++j) {
              tma_load_2d(sbase + j * DEC_A_BOX_BYTES, &tmA, &full[stage], (kb0 + j) * kstep, 0, pol_a);
              tma_load_2d(sbase + a_bytes + j * b_plane, mb, &full[stage], (kb0 + j) * kstep, r0, pol_b);
            }
          }
          ++issued;
          if (++stage == static_cast<uint32_t>(stages)) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      const int64_t first = issued > stages ? issued - stages : 0;
      for (int64_t q = first; q < issued; ++q)
        if (!mbar_wait(&full[q % stages], static_cast<uint32_t>((q / stages) & 1))) fail |= STATUS_TIMEOUT_DRAIN;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f32acc(FP8 ? 0u : 1u, 128, 16 * G) | p.idesc_or;
      const uint32_t ring_lo = smem_desc_sw128_lo(smem_u32(ring));
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool issued_any = false;
      for (int part = blockIdx.x; part < p.parts && !fail; part += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1)) {
          fail = STATUS_TIMEOUT_MMA;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * acc_cols;
        for (int kb0 = 0; kb0 < nk; kb0 += ks) {
          if (!mbar_wait(&full[stage], phase)) {
            fail = STATUS_TIMEOUT_MMA;
            break;
          }
          tc_fence_after_sync();
          const int planes = min(ks, nk - kb0);
          // Descriptors differ only in their low word (the address field), so
          // each MMA's pair is two 32-bit adds: a small-N MMA is short enough
          // that the issuing thread's instruction count shows.
          uint32_t w_lo = ring_lo + static_cast<uint32_t>((stage * stage_bytes + a_bytes) >> 4);  // B rows
          uint32_t x_lo = ring_lo + static_cast<uint32_t>((stage * stage_bytes) >> 4);            // A rows
          uint32_t accumulate = kb0 != 0;  // accumulator k mod nacc starts at the part's first group
          // planes is a multiple of G: each group of G planes is one
          // 128-row B operand (G slots) and one 16 G-row A operand
          for (int j = 0; j < planes; j += G) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t wd = desc_sw128_from_lo(w_lo + 2 * k);
              const uint64_t xd = desc_sw128_from_lo(x_lo + 2 * k);
              const uint32_t a = static_cast<uint32_t>(k & (nacc - 1));
              const uint32_t accumulate_k = accumulate | (k >= nacc ? 1u : 0u);
              if constexpr (FP8)
                umma_e4m3(d_tmem + a * 16 * G, wd, xd, idesc, accumulate_k);
              else
                umma_bf16(d_tmem + a * 16 * G, wd, xd, idesc, accumulate_k);
            }
            accumulate = 1;
            w_lo += static_cast<uint32_t>((G * b_plane) >> 4);
            x_lo += static_cast<uint32_t>((G * DEC_A_BOX_BYTES) >> 4);
          }
          issued_any = true;
          umma_commit(&empty[stage]);
          if (++stage == static_cast<uint32_t>(stages)) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (fail) break;
        umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (issued_any) {
        umma_commit(drain);
        if (!mbar_wait(drain, 0)) fail |= STATUS_TIMEOUT_DRAIN;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // C is written here only
    if (p.pdl_mode == PDL_BATCH_NEXT) griddep_wait();
    const int q = warp & 3;  // TMEM lanes 32q .. 32q+31: rows 32q .. 32q+31 of the stacked operand
    uint32_t acc = 0, acc_phase = 0, red_phase = 0;
    for (int part = blockIdx.x; part < p.parts; part += gridDim.x) {
      int r0, r1;
      part_rows(part, p.parts, p.n, r0, r1);
      const bool ready = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase));
      if (!ready) {
        fail = STATUS_TIMEOUT_EPILOGUE;
        break;
      }
      tc_fence_after_sync();
      const uint32_t t = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * acc_cols;
      if constexpr (!STACK) {
        uint32_t r[16];
        {
          uint32_t r2[32];
          tmem_ld_32x32b_x32(t, r2);           // accumulators 0 and 1
          tmem_ld_wait();
          reg_fence(r2);
#pragma unroll
          for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r2[i]) + __uint_as_float(r2[16 + i]));
          tmem_ld_32x32b_x32(t + 32, r2);      // accumulators 2 and 3
          tmem_ld_wait();
          reg_fence(r2);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            r[i] = __float_as_uint(__uint_as_float(r[i]) + (__uint_as_float(r2[i]) + __uint_as_float(r2[16 + i])));
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        const int col = r0 + q * 32 + lane;   // column of C = row of B
        if (col < r1) {
          float sbv = 1.0f;
          if constexpr (FP8) sbv = p.sb[col];
          const float bv = p.bias ? p.bias[col] : 0.0f;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (i < p.m) {
              float v = __uint_as_float(r[i]);
              if constexpr (FP8) v = (v * p.sa[i]) * sbv;
              v = apply_act(p.act, v + bv);
              if constexpr (OUT_F32)
                static_cast<float*>(p.C)[static_cast<int64_t>(i) * p.ldc + col] = v;
              else
                static_cast<__nv_bfloat16*>(p.C)[static_cast<int64_t>(i) * p.ldc + col] = __float2bfloat16_rn(v);
            }
          }
        }
      } else {
        // ---- G slots of R rows: this lane's stacked row r is the part's row
        // r mod R at the K steps of slot r / R, whose 16 sums sit in columns
        // 16 (r / R) .. + 15 of each accumulator.  A warp's 32 rows span
        // S = 32 / R slots when R < 32; nacc * S is 4 for every G.
        const int R = 128 / G;
        const int lgR = __ffs(R) - 1;
        const int r = 32 * q + lane;
        const int slot = r >> lgR;
        const int S = R >= 32 ? 1 : 32 / R;
        const int slot0 = (32 * q) >> lgR;
        uint32_t x[4][16];
#pragma unroll
        for (int u = 0; u < 4; ++u) tmem_ld_32x32b_x16(t + (u / S) * 16 * G + 16 * (slot0 + u % S), x[u]);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 4; ++u) reg_fence16(x[u]);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        float* mine = red + r * DEC_RED_STRIDE;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float v = 0.0f;
#pragma unroll
          for (int u = 0; u < 4; ++u) v += (slot == slot0 + u % S) ? __uint_as_float(x[u][i]) : 0.0f;
          mine[i] = v;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&redbar[0]);
        if (!__all_sync(0xffffffffu, mbar_wait(&redbar[0], red_phase))) {
          fail = STATUS_TIMEOUT_EPILOGUE;
          break;
        }
        // output (i, row): the sum of the G slots' partials, in slot order;
        // consecutive threads take consecutive rows (columns of C)
        const int rows = r1 - r0;
        for (int idx = r; idx < (p.m << lgR); idx += 128) {
          const int i = idx >> lgR;
          const int pr = idx & (R - 1);
          if (pr < rows) {
            const float* src = red + pr * DEC_RED_STRIDE + i;
            float v = src[0];
            for (int sl = 1; sl < G; ++sl) v += src[sl * R * DEC_RED_STRIDE];
            const int col = r0 + pr;
            if constexpr (FP8) v = (v * p.sa[i]) * p.sb[col];
            v = apply_act(p.act, v + (p.bias ? p.bias[col] : 0.0f));
            if constexpr (OUT_F32)
              static_cast<float*>(p.C)[static_cast<int64_t>(i) * p.ldc + col] = v;
            else
              static_cast<__nv_bfloat16*>(p.C)[static_cast<int64_t>(i) * p.ldc + col] = __float2bfloat16_rn(v);
          }
        }
        if (part + static_cast<int>(gridDim.x) < p.parts) {
          // every warp has read the partials before the next part's land
          __syncwarp();
          if (lane == 0) mbar_arrive(&redbar[1]);
          if (!__all_sync(0xffffffffu, mbar_wait(&redbar[1], red_phase))) {
            fail = STATUS_TIMEOUT_EPILOGUE;
            break;
          }
        }
        red_phase ^= 1;
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  if (fail) atomicOr(p.status, fail);
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

}  // namespace dgl

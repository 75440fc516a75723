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
//     one TMA box of the part's B rows and one box of A's m rows (bytes past
//     K arrive as zeros), both with the 128-byte swizzle.  The planes' loads
//     go out back to back so adjacent pieces of each B row reach the memory
//     system together.
//   * warp 1 issues tcgen05.mma with the part's B rows as the 128-row operand
//     and A's 16 rows as the N = 16 operand: D[row of B][row of A] accumulates
//     in tensor memory (two 16-column buffers, alternating by part).  The MMA
//     is asynchronous, so no warp waits on a chain of dependent products and
//     the stream is limited only by memory.  Rows of either operand past its
//     box (B rows past the part, A rows past m) read whatever the ring holds
//     there; each feeds only its own row or column of D, which is never
//     stored.
//   * warps 2-5 read D (lane = row of B, 16 columns = rows of A), scale
//     (E4M3), round and store C[i][j]: for each i the warp's 32 lanes write 32
//     consecutive columns.
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
constexpr int DEC_SMEM_BYTES = 1024 + DEC_RING_BYTES + DEC_SLACK_BYTES + 8 * (2 * DEC_MAX_STAGES + 5) + 8;
constexpr int DEC_A_BOX_BYTES = 16 * 128;
// Independent accumulators per part: the four MMAs of a 128-byte K step go to
// four separate 16-column TMEM accumulators, so consecutive MMAs do not wait
// on one another's result; the epilogue adds the four.
constexpr int DEC_NACC = 4;
constexpr int DEC_ACC_COLS = 16 * DEC_NACC;         // one accumulator buffer (of two)
constexpr int DEC_TMEM_COLS = 2 * DEC_ACC_COLS;

// Row range of part `part` of n rows cut into `parts` balanced pieces.
__device__ __forceinline__ void part_rows(int part, int parts, int n, int& r0, int& r1) {
  r0 = static_cast<int>(static_cast<int64_t>(part) * n / parts);
  r1 = static_cast<int>(static_cast<int64_t>(part + 1) * n / parts);
}

template <bool FP8, bool OUT_F32>
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
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
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
    fence_mbarrier_init();
    fence_proxy_async_shared();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, DEC_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  griddep_launch_dependents();
  griddep_wait();

  const int nk = (p.row_bytes + 127) >> 7;   // 128-byte steps of K
  const int ks = p.ksteps;                    // planes per stage
  const int b_plane = p.b_plane_bytes;        // one B box, rows rounded up to 8, x 128 bytes
  const int a_bytes = ks * DEC_A_BOX_BYTES;   // A planes first, then B planes
  int fail = 0;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB_lo);
      tma_prefetch_desc(&tmB_hi);
      const uint64_t pol_a = l2_policy_evict_last();
      const uint64_t pol_b = l2_policy_evict_first();
      const int kstep = FP8 ? 128 : 64;  // elements per 128 bytes
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      for (int part = blockIdx.x; part < p.parts && !fail; part += gridDim.x) {
        int r0, r1;
        part_rows(part, p.parts, p.n, r0, r1);
        const CUtensorMap* mb = (r1 - r0) == p.rows_hi ? &tmB_hi : &tmB_lo;
        const uint32_t tx = (p.m + (r1 - r0)) * 128;  // A box of m rows + B box of the part's rows
        for (int kb0 = 0; kb0 < nk; kb0 += ks) {
          if (!mbar_wait(&empty[stage], phase ^ 1)) {
            fail = STATUS_TIMEOUT_PRODUCER;
            break;
          }
          const int planes = min(ks, nk - kb0);
          uint8_t* sbase = ring + stage * stage_bytes;
          mbar_arrive_expect_tx(&full[stage], tx * planes);
          for (int j = 0; j < planes; ++j) {
            tma_load_2d(sbase + j * DEC_A_BOX_BYTES, &tmA, &full[stage], (kb0 + j) * kstep, 0, pol_a);
            tma_load_2d(sbase + a_bytes + j * b_plane, mb, &full[stage], (kb0 + j) * kstep, r0, pol_b);
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
      constexpr uint32_t idesc = idesc_f32acc(FP8 ? 0u : 1u, 128, 16);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool issued_any = false;
      for (int part = blockIdx.x; part < p.parts && !fail; part += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1)) {
          fail = STATUS_TIMEOUT_MMA;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * DEC_ACC_COLS;
        for (int kb0 = 0; kb0 < nk; kb0 += ks) {
          if (!mbar_wait(&full[stage], phase)) {
            fail = STATUS_TIMEOUT_MMA;
            break;
          }
          tc_fence_after_sync();
          const int planes = min(ks, nk - kb0);
          const uint32_t sbase = smem_u32(ring + stage * stage_bytes);
          for (int j = 0; j < planes; ++j) {
            const uint32_t w_addr = sbase + a_bytes + j * b_plane;   // B rows: the 128-row operand
            const uint32_t x_addr = sbase + j * DEC_A_BOX_BYTES;     // A rows: the 16-row operand
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t wd = smem_desc_sw128(w_addr + 32 * k);
              const uint64_t xd = smem_desc_sw128(x_addr + 32 * k);
              const uint32_t accumulate_k = (kb0 | j) != 0;  // accumulator k starts at the part's first plane
              if constexpr (FP8)
                umma_e4m3(d_tmem + 16 * k, wd, xd, idesc, accumulate_k);
              else
                umma_bf16(d_tmem + 16 * k, wd, xd, idesc, accumulate_k);
            }
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
    const int q = warp & 3;  // TMEM lanes 32q .. 32q+31: rows 32q .. 32q+31 of the part
    uint32_t acc = 0, acc_phase = 0;
    for (int part = blockIdx.x; part < p.parts; part += gridDim.x) {
      int r0, r1;
      part_rows(part, p.parts, p.n, r0, r1);
      const bool ready = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase));
      if (!ready) {
        fail = STATUS_TIMEOUT_EPILOGUE;
        break;
      }
      tc_fence_after_sync();
      uint32_t r[16];
      {
        uint32_t r2[32];
        const uint32_t t = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * DEC_ACC_COLS;
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
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  if (fail) atomicOr(p.status, fail);
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, DEC_TMEM_COLS);
  }
}

}  // namespace dgl

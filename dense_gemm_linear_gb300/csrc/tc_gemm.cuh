// Persistent, warp-specialised tcgen05 GEMM:  C[i,j] = sum_k A[i,k] B[j,k]
// (times sa[i] sb[j] for E4M3), fp32 accumulation in tensor memory.
//
// One CTA per SM walks a raster of 128 x BN output tiles.  Roles:
//   warp 0     TMA producer: fills an S-stage shared-memory ring with the
//              128 x 128-byte slice of A and the BN x 128-byte slice of B for
//              each k-stage.  The tensor maps are bounded at the valid rows
//              and at K, so rows past m or n and the k tail beyond K arrive as
//              zeros and the k-loop carries no predicate (the descriptor-bound
//              edge of "FlyDSL pull request 1303", changes to the RDNA3 GEMM).
//   warp 1     allocates tensor memory, then one thread issues tcgen05.mma
//              (four K=16 bf16 or K=32 E4M3 steps per 128-byte stage) into one
//              of two TMEM accumulators and commits each stage back to the
//              producer's "empty" barrier.
//   warps 2-5  epilogue: tcgen05.ld of the finished accumulator (one row per
//              thread), per-row / per-column scales for E4M3 ("Gemm
//              Optimization" guide, section 7.1: acc * scale_a * scale_b),
//              round to bf16 or keep fp32, then a transpose through shared
//              memory so each warp store covers 32 consecutive columns of one
//              row, with the column predicate j < n and row predicate i < m
//              paid once per tile, outside the k-loop (section 7.2's
//              CShuffle idea; the C-store predicate of the FlyDSL change).
// The two accumulators let the epilogue of tile t overlap the main loop of
// tile t+1.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace dgl {

template <int BN_, int STAGES_, bool FP8_, bool OUT_F32_>
struct TcConfig {
  static constexpr int BM = 128;
  static constexpr int BN = BN_;
  static constexpr int STAGES = STAGES_;
  static constexpr bool FP8 = FP8_;
  static constexpr bool OUT_F32 = OUT_F32_;
  static constexpr int ROW_BYTES = 128;                 // one 128-byte swizzle span of K per stage
  static constexpr int BK = FP8 ? 128 : 64;             // K elements per stage
  static constexpr int MMA_K_BYTES = 32;                // K=16 bf16 or K=32 E4M3 per instruction
  static constexpr int MMAS_PER_STAGE = ROW_BYTES / MMA_K_BYTES;
  static constexpr int A_STAGE_BYTES = BM * ROW_BYTES;
  static constexpr int B_STAGE_BYTES = BN * ROW_BYTES;
  static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
  static constexpr int EPI_WARPS = 4;
  static constexpr int STG_PITCH = 33;                  // floats; odd pitch keeps the transpose conflict-free
  static constexpr int STG_FLOATS = 32 * STG_PITCH;
  static constexpr int THREADS = 64 + EPI_WARPS * 32;
  static constexpr int TMEM_COLS = 2 * BN;              // two fp32 accumulators of BN columns
  static constexpr int BAR_BYTES = 8 * (2 * STAGES + 5) + 8;
  static constexpr int SMEM_BYTES =
      1024 /* alignment slack */ + STAGES * STAGE_BYTES + EPI_WARPS * STG_FLOATS * 4 + BAR_BYTES;
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "UMMA N for M=128 must be a multiple of 16, <= 256");
  static_assert(TMEM_COLS == 64 || TMEM_COLS == 128 || TMEM_COLS == 256 || TMEM_COLS == 512,
                "TMEM allocation must be a power of two >= 32 columns");
  static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
};

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const TcParams p) {
  constexpr int BM = Cfg::BM, BN = Cfg::BN, STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + STAGES * Cfg::A_STAGE_BYTES;
  float* stg = reinterpret_cast<float*>(sB + STAGES * Cfg::B_STAGE_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(stg + Cfg::EPI_WARPS * Cfg::STG_FLOATS);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], Cfg::EPI_WARPS);
    }
    mbar_init(drain, 1);
    fence_mbarrier_init();
    fence_proxy_async_shared();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  int fail = 0;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      for (int tile = blockIdx.x; tile < p.num_tiles && !fail; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, mb, nb);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1)) {
            fail = STATUS_TIMEOUT_PRODUCER;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], Cfg::STAGE_BYTES);
          tma_load_2d(sA + stage * Cfg::A_STAGE_BYTES, &tmA, &full[stage], kb * Cfg::BK, mb * BM, pol);
          tma_load_2d(sB + stage * Cfg::B_STAGE_BYTES, &tmB, &full[stage], kb * Cfg::BK, nb * BN, pol);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Copies still in flight land before this CTA may exit: wait for the
      // completion of the last STAGES loads issued (already complete on the
      // normal path).
      const int64_t first = issued > STAGES ? issued - STAGES : 0;
      for (int64_t q = first; q < issued; ++q) {
        if (!mbar_wait(&full[q % STAGES], static_cast<uint32_t>((q / STAGES) & 1))) fail |= STATUS_TIMEOUT_DRAIN;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f32acc(Cfg::FP8 ? 0u : 1u, BM, BN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool issued_any = false;
      for (int tile = blockIdx.x; tile < p.num_tiles && !fail; tile += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1)) {
          fail = STATUS_TIMEOUT_MMA;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase)) {
            fail = STATUS_TIMEOUT_MMA;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_addr = smem_u32(sA + stage * Cfg::A_STAGE_BYTES);
          const uint32_t b_addr = smem_u32(sB + stage * Cfg::B_STAGE_BYTES);
#pragma unroll
          for (int k = 0; k < Cfg::MMAS_PER_STAGE; ++k) {
            const uint64_t ad = smem_desc_sw128(a_addr + k * Cfg::MMA_K_BYTES);
            const uint64_t bd = smem_desc_sw128(b_addr + k * Cfg::MMA_K_BYTES);
            const uint32_t accumulate = (kb | k) != 0;
            if constexpr (Cfg::FP8)
              umma_e4m3(d_tmem, ad, bd, idesc, accumulate);
            else
              umma_bf16(d_tmem, ad, bd, idesc, accumulate);
          }
          issued_any = true;
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (fail) break;
        umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      // Every MMA this thread issued has finished before TMEM is released.
      if (issued_any) {
        umma_commit(drain);
        if (!mbar_wait(drain, 0)) fail |= STATUS_TIMEOUT_DRAIN;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lanes 32q .. 32q+31 are reachable from this warp
    float* my_stg = stg + (warp - 2) * Cfg::STG_FLOATS;
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      int mb, nb;
      tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, mb, nb);
      // all lanes decide together: tcgen05.ld below is warp-collective
      const bool ready = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase));
      if (!ready) {
        fail = STATUS_TIMEOUT_EPILOGUE;
        break;
      }
      tc_fence_after_sync();
      const int row0 = mb * BM + q * 32;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      float row_scale = 1.0f;
      if constexpr (Cfg::FP8) row_scale = (row0 + lane < p.m) ? p.sa[row0 + lane] : 0.0f;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c * 32, r);
        tmem_ld_wait();
        if (c == BN / 32 - 1) {
          // accumulator fully read: hand it back to the MMA warp
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[acc]);
        }
        const int col0 = nb * BN + c * 32;
        float col_scale = 1.0f;
        if constexpr (Cfg::FP8) col_scale = (col0 + lane < p.n) ? p.sb[col0 + lane] : 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float v = __uint_as_float(r[j]);
          if constexpr (Cfg::FP8) v = (v * row_scale) * __shfl_sync(0xffffffffu, col_scale, j);
          my_stg[lane * Cfg::STG_PITCH + j] = v;
        }
        __syncwarp();
        const int col = col0 + lane;
        if (col < p.n) {
#pragma unroll 4
          for (int rr = 0; rr < 32; ++rr) {
            const int row = row0 + rr;
            if (row >= p.m) break;
            const float v = my_stg[rr * Cfg::STG_PITCH + lane];
            if constexpr (Cfg::OUT_F32)
              static_cast<float*>(p.C)[static_cast<int64_t>(row) * p.ldc + col] = v;
            else
              static_cast<__nv_bfloat16*>(p.C)[static_cast<int64_t>(row) * p.ldc + col] = __float2bfloat16_rn(v);
          }
        }
        __syncwarp();
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
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace dgl

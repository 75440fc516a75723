// Host-side dispatch of the tcgen05 kernel over its compile-time variants
// (tile width, output type, whole-row staging), shared by the bf16 and E4M3
// translation units.
#pragma once

#include <atomic>

#include "launch.h"
#include "tc_gemm.cuh"

namespace dgl {

template <int BN, bool FP8, bool OUT_F32, bool ROWSTG, int CG, bool EPI, bool MX = false, int BM = 128>
cudaError_t tc_launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tbh, const CUtensorMap& tc,
                          const TcParams& p, int grid, cudaStream_t stream) {
  using Cfg = TcConfig<BN, FP8, OUT_F32, ROWSTG, CG, EPI, MX, BM>;
  auto kern = tc_gemm_kernel<Cfg>;
  static std::atomic<uint64_t> attr_done{0};  // one bit per device
  cudaError_t e = set_smem_attr_once(kern, Cfg::SMEM_BYTES, attr_done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  // the kernel waits for its predecessor on the stream (griddep_wait) before
  // any global access, so it may be launched while that one finishes
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if constexpr (CG == 2) {
    // CTA pairs: a cluster of two CTAs per output tile
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CG;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, tbh, tc, p);
}

template <int BN, bool FP8, int CG, bool EPI, int BM = 128>
cudaError_t tc_launch_bn(int out, bool row_staging, const CUtensorMap& ta, const CUtensorMap& tb,
                         const CUtensorMap& tbh, const CUtensorMap& tc, const TcParams& p, int grid,
                         cudaStream_t stream) {
  if (out == 1) return tc_launch_one<BN, FP8, true, false, CG, EPI, false, BM>(ta, tb, tbh, tc, p, grid, stream);
  if (row_staging)
    return tc_launch_one<BN, FP8, false, true, CG, EPI, false, BM>(ta, tb, tbh, tc, p, grid, stream);
  return tc_launch_one<BN, FP8, false, false, CG, EPI, false, BM>(ta, tb, tbh, tc, p, grid, stream);
}

// 64-row tiles (one CTA, M = 64 MMAs): plain GEMM variants only, compiled
// in their own translation units.
template <bool FP8>
cudaError_t tc_launch_m64(int out, int tile_n, bool row_staging, const CUtensorMap& ta, const CUtensorMap& tb,
                          const CUtensorMap& tc, const TcParams& p, int grid, cudaStream_t stream) {
  switch (tile_n) {
    case 64: return tc_launch_bn<64, FP8, 1, false, 64>(out, row_staging, ta, tb, tb, tc, p, grid, stream);
    case 128: return tc_launch_bn<128, FP8, 1, false, 64>(out, row_staging, ta, tb, tb, tc, p, grid, stream);
    case 256: return tc_launch_bn<256, FP8, 1, false, 64>(out, row_staging, ta, tb, tb, tc, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

// EPI: the linear-layer variants, compiled for the 128- and 256-wide tiles
// only (tc_supported_epi_tile); the plain variants cover the ladder's 128- and
// 256-row tiles (the 64-row ones: tc_launch_m64).
template <bool FP8, bool EPI>
cudaError_t tc_launch(int out, int tile_m, int tile_n, bool row_staging, const CUtensorMap& ta, const CUtensorMap& tb,
                      const CUtensorMap& tbh, const CUtensorMap& tc, const TcParams& p, int grid, cudaStream_t stream) {
  if (tile_m == 128) {
    switch (tile_n) {
      case 64:
        if constexpr (EPI) return cudaErrorInvalidValue;
        else return tc_launch_bn<64, FP8, 1, EPI>(out, row_staging, ta, tb, tbh, tc, p, grid, stream);
      case 128: return tc_launch_bn<128, FP8, 1, EPI>(out, row_staging, ta, tb, tbh, tc, p, grid, stream);
      case 256: return tc_launch_bn<256, FP8, 1, EPI>(out, row_staging, ta, tb, tbh, tc, p, grid, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  if (tile_m == 256) {
    switch (tile_n) {
      case 128: return tc_launch_bn<128, FP8, 2, EPI>(out, row_staging, ta, tb, tbh, tc, p, grid, stream);
      case 224:
        if constexpr (EPI) return cudaErrorInvalidValue;
        else return tc_launch_bn<224, FP8, 2, EPI>(out, row_staging, ta, tb, tbh, tc, p, grid, stream);
      case 256: return tc_launch_bn<256, FP8, 2, EPI>(out, row_staging, ta, tb, tbh, tc, p, grid, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace dgl

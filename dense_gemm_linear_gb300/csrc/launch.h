// Host-side launch entry points of the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

#include <atomic>

namespace dgl {

// Raise a kernel's dynamic shared-memory limit once per device.
template <class Kernel>
cudaError_t set_smem_attr_once(Kernel kern, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// tcgen05 tile kernel.  out: 0 bf16, 1 fp32.  tile_m: 128 (one CTA per tile)
// or 256 (a CTA pair per tile, launched as clusters of two), or 64 (passed on
// to the 64-row variants below; tbh unused).  tile_n: 64, 128 or 256, and 224
// on CTA pairs (plain GEMM only).
// row_staging (bf16 output only): C rows are not 16-byte aligned, so the
// epilogue stages whole rows and writes each row's aligned body in bulk.
// tc: tensor map of C for TMA stores (used when p.c_tma is set).
// tbh: B's map with half-height boxes, for the half tiles of a split tail.
cudaError_t launch_tc_bf16(int out, int tile_m, int tile_n, bool row_staging, const CUtensorMap& ta,
                           const CUtensorMap& tb, const CUtensorMap& tbh, const CUtensorMap& tc, const TcParams& p,
                           int grid, cudaStream_t stream);
cudaError_t launch_tc_e4m3(int out, int tile_m, int tile_n, bool row_staging, const CUtensorMap& ta,
                           const CUtensorMap& tb, const CUtensorMap& tbh, const CUtensorMap& tc, const TcParams& p,
                           int grid, cudaStream_t stream);
// The same with the linear-layer epilogue compiled in (p.bias, p.act,
// p.gated); tile_n 128 or 256 only.
cudaError_t launch_tc_bf16_epi(int out, int tile_m, int tile_n, bool row_staging, const CUtensorMap& ta,
                               const CUtensorMap& tb, const CUtensorMap& tbh, const CUtensorMap& tc,
                               const TcParams& p, int grid, cudaStream_t stream);
cudaError_t launch_tc_e4m3_epi(int out, int tile_m, int tile_n, bool row_staging, const CUtensorMap& ta,
                               const CUtensorMap& tb, const CUtensorMap& tbh, const CUtensorMap& tc,
                               const TcParams& p, int grid, cudaStream_t stream);
// 64-row tiles (tile_m 64: one CTA per tile, M = 64 MMAs; tile_n 64, 128 or
// 256), plain GEMM only.  The C map tc has 16-row boxes: each epilogue warp
// holds 16 rows of such a tile.
cudaError_t launch_tc_bf16_m64(int out, int tile_n, bool row_staging, const CUtensorMap& ta, const CUtensorMap& tb,
                               const CUtensorMap& tc, const TcParams& p, int grid, cudaStream_t stream);
cudaError_t launch_tc_e4m3_m64(int out, int tile_n, bool row_staging, const CUtensorMap& ta, const CUtensorMap& tb,
                               const CUtensorMap& tc, const TcParams& p, int grid, cudaStream_t stream);
// Block-scaled FP4 (MXFP4) tile kernel: 128 x 256 tiles, one CTA per tile;
// ta / tb: byte maps of the packed operands (K / 2 bytes per row); p.sfa,
// p.sfb: the E8M0 scales.
cudaError_t launch_tc_mxfp4(int out, bool row_staging, const CUtensorMap& ta, const CUtensorMap& tb,
                            const CUtensorMap& tc, const TcParams& p, int grid, cudaStream_t stream);
// Decode kernel: ta = A map (16-row box), tb_lo / tb_hi = B maps whose box
// heights are the two part sizes floor(n/parts) and ceil(n/parts).
cudaError_t launch_decode(int dtype, int out, const CUtensorMap& ta, const CUtensorMap& tb_lo,
                          const CUtensorMap& tb_hi, const DecodeParams& p, int grid, cudaStream_t stream);
cudaError_t launch_zero_fill(int out, void* C, int64_t ldc, int m, int n, cudaStream_t stream);

}  // namespace dgl

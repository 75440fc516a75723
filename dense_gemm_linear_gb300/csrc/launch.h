// Host-side launch entry points of the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace dgl {

// tcgen05 tile kernel.  out: 0 bf16, 1 fp32.  tile_n: 64, 128 or 256.
// row_staging (bf16 output only): C rows are not 16-byte aligned, so the
// epilogue stages whole rows and writes each row's aligned body in bulk.
// tc: tensor map of C for TMA stores (used when p.c_tma is set).
cudaError_t launch_tc_bf16(int out, int tile_n, bool row_staging, const CUtensorMap& ta, const CUtensorMap& tb,
                           const CUtensorMap& tc, const TcParams& p, int grid, cudaStream_t stream);
cudaError_t launch_tc_e4m3(int out, int tile_n, bool row_staging, const CUtensorMap& ta, const CUtensorMap& tb,
                           const CUtensorMap& tc, const TcParams& p, int grid, cudaStream_t stream);
cudaError_t launch_decode(int dtype, int out, const DecodeParams& p, int grid, cudaStream_t stream);
cudaError_t launch_zero_fill(int out, void* C, int64_t ldc, int m, int n, cudaStream_t stream);

}  // namespace dgl

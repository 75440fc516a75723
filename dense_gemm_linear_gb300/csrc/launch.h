// Host-side launch entry points of the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace dgl {

// Ring depth of the tcgen05 kernel for each tile width (fixed at compile time;
// each fills about 192 KB of shared memory).
constexpr int tc_stages_for(int tile_n) { return tile_n == 64 ? 8 : (tile_n == 128 ? 6 : 4); }

// Dynamic shared memory the tcgen05 kernel needs for a tile width (bytes).
int tc_smem_bytes(int tile_n, bool fp8);

// dtype: 0 bf16, 1 E4M3.  out: 0 bf16, 1 fp32.  tile_n: 64, 128 or 256.
cudaError_t launch_tc_bf16(int out, int tile_n, const CUtensorMap& ta, const CUtensorMap& tb, const TcParams& p,
                           int grid, cudaStream_t stream);
cudaError_t launch_tc_e4m3(int out, int tile_n, const CUtensorMap& ta, const CUtensorMap& tb, const TcParams& p,
                           int grid, cudaStream_t stream);
cudaError_t launch_decode(int dtype, int out, const DecodeParams& p, int grid, cudaStream_t stream);
cudaError_t launch_zero_fill(int out, void* C, int64_t ldc, int m, int n, cudaStream_t stream);

}  // namespace dgl

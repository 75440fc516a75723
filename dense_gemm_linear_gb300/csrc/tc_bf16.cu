// bf16 x bf16 -> fp32 accumulate instantiations of the tcgen05 tile kernel.
#include "tc_launch.cuh"

namespace dgl {

cudaError_t launch_tc_bf16(int out, int tile_m, int tile_n, bool row_staging, const CUtensorMap& ta,
                          const CUtensorMap& tb, const CUtensorMap& tbh, const CUtensorMap& tc, const TcParams& p,
                          int grid, cudaStream_t stream) {
  if (tile_m == 64) return launch_tc_bf16_m64(out, tile_n, row_staging, ta, tb, tc, p, grid, stream);
  return tc_launch<false, false>(out, tile_m, tile_n, row_staging, ta, tb, tbh, tc, p, grid, stream);
}

}  // namespace dgl

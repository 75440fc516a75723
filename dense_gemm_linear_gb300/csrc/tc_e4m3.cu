// E4M3 x E4M3 -> fp32 accumulate instantiations of the tcgen05 tile kernel,
// with the per-row / per-column scale epilogue.
#include "tc_launch.cuh"

namespace dgl {

cudaError_t launch_tc_e4m3(int out, int tile_m, int tile_n, bool row_staging, const CUtensorMap& ta,
                          const CUtensorMap& tb, const CUtensorMap& tbh, const CUtensorMap& tc, const TcParams& p,
                          int grid, cudaStream_t stream) {
  if (tile_m == 64) return launch_tc_e4m3_m64(out, tile_n, row_staging, ta, tb, tc, p, grid, stream);
  return tc_launch<true, false>(out, tile_m, tile_n, row_staging, ta, tb, tbh, tc, p, grid, stream);
}

}  // namespace dgl

// E4M3 instantiations of the tcgen05 tile kernel on 64-row tiles (one CTA,
// M = 64 MMAs), with the per-row / per-column scale epilogue.
#include "tc_launch.cuh"

namespace dgl {

cudaError_t launch_tc_e4m3_m64(int out, int tile_n, bool row_staging, const CUtensorMap& ta, const CUtensorMap& tb,
                               const CUtensorMap& tc, const TcParams& p, int grid, cudaStream_t stream) {
  return tc_launch_m64<true>(out, tile_n, row_staging, ta, tb, tc, p, grid, stream);
}

}  // namespace dgl

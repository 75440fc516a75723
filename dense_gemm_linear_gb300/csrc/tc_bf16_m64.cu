// bf16 instantiations of the tcgen05 tile kernel on 64-row tiles (one CTA,
// M = 64 MMAs): the small rungs of the tile ladder.
#include "tc_launch.cuh"

namespace dgl {

cudaError_t launch_tc_bf16_m64(int out, int tile_n, bool row_staging, const CUtensorMap& ta, const CUtensorMap& tb,
                               const CUtensorMap& tc, const TcParams& p, int grid, cudaStream_t stream) {
  return tc_launch_m64<false>(out, tile_n, row_staging, ta, tb, tc, p, grid, stream);
}

}  // namespace dgl

// Block-scaled FP4 (MXFP4) instantiations of the tcgen05 tile kernel:
// kind::mxf4 MMAs with E8M0 scales per 32 elements of K, 128 x 256 tiles.
#include "tc_launch.cuh"

namespace dgl {

cudaError_t launch_tc_mxfp4(int out, bool row_staging, const CUtensorMap& ta, const CUtensorMap& tb,
                            const CUtensorMap& tc, const TcParams& p, int grid, cudaStream_t stream) {
  if (out == 1) return tc_launch_one<256, false, true, false, 1, false, true>(ta, tb, tb, tc, p, grid, stream);
  if (row_staging) return tc_launch_one<256, false, false, true, 1, false, true>(ta, tb, tb, tc, p, grid, stream);
  return tc_launch_one<256, false, false, false, 1, false, true>(ta, tb, tb, tc, p, grid, stream);
}

}  // namespace dgl

// bf16 x bf16 -> fp32 accumulate instantiations of the tcgen05 tile kernel.
#include "launch.h"
#include "tc_gemm.cuh"

namespace dgl {

namespace {

template <int BN, bool OUT_F32>
cudaError_t launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const TcParams& p, int grid,
                       cudaStream_t stream) {
  using Cfg = TcConfig<BN, tc_stages_for(BN), false, OUT_F32>;
  auto kern = tc_gemm_kernel<Cfg>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(ta, tb, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_bf16(int out, int tile_n, const CUtensorMap& ta, const CUtensorMap& tb, const TcParams& p,
                           int grid, cudaStream_t stream) {
  const bool f32 = out == 1;
  switch (tile_n) {
    case 64:
      return f32 ? launch_one<64, true>(ta, tb, p, grid, stream) : launch_one<64, false>(ta, tb, p, grid, stream);
    case 128:
      return f32 ? launch_one<128, true>(ta, tb, p, grid, stream) : launch_one<128, false>(ta, tb, p, grid, stream);
    case 256:
      return f32 ? launch_one<256, true>(ta, tb, p, grid, stream) : launch_one<256, false>(ta, tb, p, grid, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

int tc_smem_bytes(int tile_n, bool fp8) {
  // fp8 and bf16 stages have the same byte layout
  (void)fp8;
  switch (tile_n) {
    case 64: return TcConfig<64, tc_stages_for(64), false, false>::SMEM_BYTES;
    case 128: return TcConfig<128, tc_stages_for(128), false, false>::SMEM_BYTES;
    case 256: return TcConfig<256, tc_stages_for(256), false, false>::SMEM_BYTES;
    default: return -1;
  }
}

}  // namespace dgl

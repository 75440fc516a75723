// Instantiations of the decode-shape kernel, plus the K = 0 zero fill.
#include "decode_gemm.cuh"
#include "launch.h"

namespace dgl {

namespace {

template <bool FP8, bool OUT_F32, bool STACK>
cudaError_t launch_one(const CUtensorMap& ta, const CUtensorMap& tb_lo, const CUtensorMap& tb_hi,
                       const DecodeParams& p, int grid, cudaStream_t stream) {
  auto kern = decode_gemm_kernel<FP8, OUT_F32, STACK>;
  constexpr int smem = dec_smem_bytes(STACK);
  static std::atomic<uint64_t> attr_done{0};  // one bit per device
  cudaError_t e = set_smem_attr_once(kern, smem, attr_done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(DEC_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  // the kernel waits for its predecessor (griddep_wait) before any global access
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, ta, tb_lo, tb_hi, p);
}

template <typename T>
__global__ void zero_fill_kernel(T* C, int64_t ldc, int m, int n) {
  const int64_t total = static_cast<int64_t>(m) * n;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t i = idx / n, j = idx - i * n;
    C[i * ldc + j] = T(0.0f);
  }
}

}  // namespace

cudaError_t launch_decode(int dtype, int out, const CUtensorMap& ta, const CUtensorMap& tb_lo,
                          const CUtensorMap& tb_hi, const DecodeParams& p, int grid, cudaStream_t stream) {
  const bool f32 = out == 1;
  if (p.group > 1) {
    if (dtype == 1)
      return f32 ? launch_one<true, true, true>(ta, tb_lo, tb_hi, p, grid, stream)
                 : launch_one<true, false, true>(ta, tb_lo, tb_hi, p, grid, stream);
    return f32 ? launch_one<false, true, true>(ta, tb_lo, tb_hi, p, grid, stream)
               : launch_one<false, false, true>(ta, tb_lo, tb_hi, p, grid, stream);
  }
  if (dtype == 1)
    return f32 ? launch_one<true, true, false>(ta, tb_lo, tb_hi, p, grid, stream)
               : launch_one<true, false, false>(ta, tb_lo, tb_hi, p, grid, stream);
  return f32 ? launch_one<false, true, false>(ta, tb_lo, tb_hi, p, grid, stream)
             : launch_one<false, false, false>(ta, tb_lo, tb_hi, p, grid, stream);
}

cudaError_t launch_zero_fill(int out, void* C, int64_t ldc, int m, int n, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(m) * n;
  const int grid = static_cast<int>(total / 256 + 1 < 4096 ? total / 256 + 1 : 4096);
  if (out == 1)
    zero_fill_kernel<float><<<grid, 256, 0, stream>>>(static_cast<float*>(C), ldc, m, n);
  else
    zero_fill_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(static_cast<__nv_bfloat16*>(C), ldc, m, n);
  return cudaGetLastError();
}

}  // namespace dgl

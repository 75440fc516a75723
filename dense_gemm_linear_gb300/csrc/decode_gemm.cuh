// Decode-shape GEMM (m <= 16 rows of A), the memory-bound case: with L = 1
// the token count M of the MLP GEMM is the batch size B ("GEMM analysis in
// TraceLens", section "Prefill versus decode"), so each call streams the whole
// weight matrix B once for a handful of rows of A, and the arithmetic
// intensity is about m flop per byte of B ("Gemm Optimization" guide,
// section 8.3: small M is memory-bound).
//
// Design: no tensor-memory pipeline at all.  Each CTA owns a contiguous,
// balanced range of B rows (n / grid rows, any remainder spread one row at a
// time) and all 16 warps split K.  A lane loads 16 bytes of one B row per
// 64-byte chunk (8 rows x 64 bytes per warp load) with non-allocating
// streaming loads, and feeds them to mma.sync (m16n8k16 bf16 or m16n8k32
// E4M3, fp32 accumulate) with the m <= 16 rows of A as the 16-row operand.
// Because a dot product may visit k in any order, the 16 bytes a lane holds
// are assigned to the instruction's k slots by a fixed permutation, and the
// lane's A fragment is loaded with the same permutation: the 16 bytes of A
// rows g and g+8 at the same byte offset.  The per-warp partial sums of each
// 8-row group are reduced across warps through shared memory in fixed warp
// order (deterministic), then scaled (E4M3), rounded and stored with
// consecutive threads on consecutive columns of C.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace dgl {

constexpr int DEC_WARPS = 16;
constexpr int DEC_THREADS = DEC_WARPS * 32;
constexpr int DEC_BATCH = 8;        // 64-byte chunks per warp per batch (one 16-byte load per lane each)
constexpr int DEC_BLOCK_GROUPS = 16;  // 8-row groups reduced per shared-memory pass (128 rows)
constexpr int DEC_SMEM_BYTES = DEC_BLOCK_GROUPS * DEC_WARPS * 128 * 4;

__device__ __forceinline__ void mma_bf16_m16n8k16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                  uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_e4m3_m16n8k32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                  uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <bool FP8, bool OUT_F32>
__global__ void __launch_bounds__(DEC_THREADS, 1) decode_gemm_kernel(const DecodeParams p) {
  extern __shared__ float red[];  // [DEC_BLOCK_GROUPS][DEC_WARPS][16 rows of A][8 rows of B]
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;  // A row (and B row within the 8-row group)
  const int t = lane & 3;   // 16-byte slot within a 64-byte chunk

  const int64_t r_begin = static_cast<int64_t>(blockIdx.x) * p.n / gridDim.x;
  const int64_t r_end = static_cast<int64_t>(blockIdx.x + 1) * p.n / gridDim.x;

  const int nchunks = (p.row_bytes + 63) >> 6;
  const int cpw = (nchunks + DEC_WARPS - 1) / DEC_WARPS;
  const int c_begin = warp * cpw;
  const int c_end = min(nchunks, c_begin + cpw);
  const int nbatches = c_end > c_begin ? (c_end - c_begin + DEC_BATCH - 1) / DEC_BATCH : 0;

  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  uint4 xa[DEC_BATCH], ya[DEC_BATCH];
  auto load_a = [&](int cb) {
#pragma unroll
    for (int u = 0; u < DEC_BATCH; ++u) {
      const int c = cb + u;
      const int off = c * 64 + t * 16;
      const bool ok = c < c_end && off < p.row_bytes;
      xa[u] = (ok && g < p.m) ? ldg_v4(p.A + static_cast<int64_t>(g) * p.row_bytes + off) : zero;
      ya[u] = (ok && g + 8 < p.m) ? ldg_v4(p.A + static_cast<int64_t>(g + 8) * p.row_bytes + off) : zero;
    }
  };
  if (nbatches == 1) load_a(c_begin);

  for (int64_t blk = r_begin; blk < r_end; blk += 8 * DEC_BLOCK_GROUPS) {
    const int64_t blk_end = min(r_end, blk + 8 * DEC_BLOCK_GROUPS);
    const int ngroups = static_cast<int>((blk_end - blk + 7) >> 3);
    for (int gi = 0; gi < ngroups; ++gi) {
      const int64_t row = blk + gi * 8 + g;
      const bool row_ok = row < blk_end;
      const uint8_t* brow = p.B + row * p.row_bytes;
      float acc0[4] = {0.f, 0.f, 0.f, 0.f};
      float acc1[4] = {0.f, 0.f, 0.f, 0.f};
      for (int b = 0; b < nbatches; ++b) {
        const int cb = c_begin + b * DEC_BATCH;
        if (nbatches > 1) load_a(cb);
        uint4 rb[DEC_BATCH];
#pragma unroll
        for (int u = 0; u < DEC_BATCH; ++u) {
          const int c = cb + u;
          const int off = c * 64 + t * 16;
          rb[u] = (row_ok && c < c_end && off < p.row_bytes) ? ldg_stream_v4(brow + off) : zero;
        }
#pragma unroll
        for (int u = 0; u < DEC_BATCH; ++u) {
          float(&acc)[4] = (u & 1) ? acc1 : acc0;
          if constexpr (FP8) {
            mma_e4m3_m16n8k32(acc, xa[u].x, ya[u].x, xa[u].y, ya[u].y, rb[u].x, rb[u].y);
            mma_e4m3_m16n8k32(acc, xa[u].z, ya[u].z, xa[u].w, ya[u].w, rb[u].z, rb[u].w);
          } else {
            mma_bf16_m16n8k16(acc, xa[u].x, ya[u].x, xa[u].y, ya[u].y, rb[u].x, rb[u].y);
            mma_bf16_m16n8k16(acc, xa[u].z, ya[u].z, xa[u].w, ya[u].w, rb[u].z, rb[u].w);
          }
        }
      }
      // accumulator fragment: d0 (g, 2t), d1 (g, 2t+1), d2 (g+8, 2t), d3 (g+8, 2t+1)
      float* dst = red + (gi * DEC_WARPS + warp) * 128;
      dst[g * 8 + 2 * t] = acc0[0] + acc1[0];
      dst[g * 8 + 2 * t + 1] = acc0[1] + acc1[1];
      dst[(g + 8) * 8 + 2 * t] = acc0[2] + acc1[2];
      dst[(g + 8) * 8 + 2 * t + 1] = acc0[3] + acc1[3];
    }
    __syncthreads();
    const int ncols = static_cast<int>(blk_end - blk);
    for (int idx = threadIdx.x; idx < p.m * ncols; idx += DEC_THREADS) {
      const int i = idx / ncols;
      const int c = idx - i * ncols;
      const float* src = red + ((c >> 3) * DEC_WARPS) * 128 + i * 8 + (c & 7);
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < DEC_WARPS; ++w) s += src[w * 128];
      const int64_t col = blk + c;
      if constexpr (FP8) s = (s * p.sa[i]) * p.sb[col];
      if constexpr (OUT_F32)
        static_cast<float*>(p.C)[i * p.ldc + col] = s;
      else
        static_cast<__nv_bfloat16*>(p.C)[i * p.ldc + col] = __float2bfloat16_rn(s);
    }
    __syncthreads();
  }
}

}  // namespace dgl

// Parameters shared by the host launcher and the kernels.
#pragma once

#include <cstdint>

namespace dgl {

// Bits OR-ed into the device status word when a bounded wait gives up.
enum : int {
  STATUS_TIMEOUT_PRODUCER = 1,
  STATUS_TIMEOUT_MMA = 2,
  STATUS_TIMEOUT_EPILOGUE = 4,
  STATUS_TIMEOUT_DRAIN = 8,
  STATUS_TMEM_MISMATCH = 16,  // a CTA pair's tensor-memory allocations differ
};

// Persistent tcgen05 tile kernel: problem and schedule.
struct TcParams {
  void* C;              // output, row pitch ldc elements
  int64_t ldc;
  int m, n, K;          // valid rows of A/C, valid rows of B (= columns of C), inner extent
  const float* sa;      // E4M3 only: per-row scale of A (m entries)
  const float* sb;      // E4M3 only: per-row scale of B (n entries)
  int tiles_m, tiles_n, num_tiles, num_kb;
  int group_m;          // tile raster: group_m row-tiles share each column sweep
  int c_tma;            // 1: C is written by TMA tensor stores (16-byte aligned pitch and base)
  int* status;          // device status word
};

// Decode (m <= 16) kernel parameters.  A and B are read through tensor maps.
struct DecodeParams {
  const float* sa;
  const float* sb;
  void* C;
  int64_t ldc;
  int m, n;
  int row_bytes;        // K * element size
  int parts;            // B rows are cut into this many balanced parts
  int rows_hi;          // ceil(n / parts): parts of this size use the second B map
  int stages;           // ring depth
  int ksteps;           // 128-byte K steps per stage
  int b_plane_bytes;    // one B box: rows_hi rounded up to 8, x 128 bytes
  int stage_bytes;      // ksteps x (A box (2 KB) + B box)
  int* status;          // device status word
};

__host__ __device__ inline void tile_coords(int tile, int tiles_m, int tiles_n, int group_m, int& mb, int& nb) {
  const int per_group = group_m * tiles_n;
  const int g = tile / per_group;
  const int first_m = g * group_m;
  const int rest = tiles_m - first_m;
  const int gsize = rest < group_m ? rest : group_m;
  const int r = tile - g * per_group;
  mb = first_m + r % gsize;
  nb = r / gsize;
}

}  // namespace dgl

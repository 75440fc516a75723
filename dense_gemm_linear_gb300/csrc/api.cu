// C ABI: argument validation, per-device state, plan cache, TMA tensor maps
// and kernel dispatch.  See include/dgl.h for the contract of each call.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <unordered_map>

#include "common.cuh"
#include "dgl.h"
#include "launch.h"
#include "plan.h"

namespace dgl {

// Per-device status word: kernels OR timeout bits into it.
__device__ int g_status_word;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  int cc_major = 0, cc_minor = 0;
  int smem_optin = 0;
  int* status = nullptr;  // device address of g_status_word on this device
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

struct PlanKey {
  int dev, dtype, out;
  int64_t m, n, K;
  bool operator==(const PlanKey& o) const {
    return dev == o.dev && dtype == o.dtype && out == o.out && m == o.m && n == o.n && K == o.K;
  }
};
struct PlanKeyHash {
  size_t operator()(const PlanKey& k) const {
    size_t h = std::hash<int64_t>()(k.m);
    h = h * 1000003u ^ std::hash<int64_t>()(k.n);
    h = h * 1000003u ^ std::hash<int64_t>()(k.K);
    h = h * 1000003u ^ static_cast<size_t>(k.dev * 16 + k.dtype * 4 + k.out);
    return h;
  }
};
std::unordered_map<PlanKey, dgl_plan_info, PlanKeyHash> g_plans;

// Stream-K workspace, one per (device, stream): fp32 partial tiles and one
// epoch flag per partial slot.  Launches on one stream run in order, so they
// can share it; each launch gets a fresh epoch so stale flags never match.
struct Workspace {
  float* ws = nullptr;
  size_t ws_bytes = 0;
  int* flags = nullptr;
  int nflags = 0;
  int epoch = 0;
};
std::map<std::pair<int, cudaStream_t>, Workspace> g_workspaces;

dgl_status acquire_workspace(int dev, cudaStream_t stream, size_t bytes, int nflags, float** ws, int** flags,
                             int* epoch) {
  std::lock_guard<std::mutex> lock(g_mu);
  Workspace& w = g_workspaces[std::make_pair(dev, stream)];
  if (w.ws_bytes < bytes || w.nflags < nflags || w.epoch == INT32_MAX) {
    // growing frees the old buffers, which waits for work still using them
    if (w.ws) cudaFree(w.ws);
    if (w.flags) cudaFree(w.flags);
    w = Workspace{};
    const size_t want = bytes > (size_t(24) << 20) ? bytes : (size_t(24) << 20);
    const int want_flags = nflags > 512 ? nflags : 512;
    if (cudaMalloc(reinterpret_cast<void**>(&w.ws), want) != cudaSuccess) return DGL_ERR_CUDA;
    if (cudaMalloc(reinterpret_cast<void**>(&w.flags), sizeof(int) * want_flags) != cudaSuccess) {
      cudaFree(w.ws);
      w = Workspace{};
      return DGL_ERR_CUDA;
    }
    if (cudaMemset(w.flags, 0, sizeof(int) * want_flags) != cudaSuccess) return DGL_ERR_CUDA;
    w.ws_bytes = want;
    w.nflags = want_flags;
  }
  *ws = w.ws;
  *flags = w.flags;
  *epoch = ++w.epoch;
  return DGL_OK;
}

// ---- scratch of dgl_gemm_noalloc: a fixed device array instead of cudaMalloc.
// Layout: DGL_NOALLOC_SCRATCH_BYTES of fp32 partial tiles, then one epoch flag
// per partial slot.  Every device that loads the library holds it until exit.
constexpr int kNoallocFlags = 160;
static __device__ __align__(256) uint8_t g_noalloc_scratch[DGL_NOALLOC_SCRATCH_BYTES + kNoallocFlags * sizeof(int)];

// The array as this device sees it.  Host code cannot use the array's name as
// an address (it stands for a host-side shadow), so set-up asks the runtime
// for the device address once per device, with that device current.
struct StaticScratch {
  bool ready = false;
  float* ws = nullptr;
  size_t ws_bytes = 0;
  int* flags = nullptr;
  int nflags = 0;
  int epoch = 0;  // last epoch handed out; flags hold earlier epochs or zero
};
StaticScratch g_noalloc[kMaxDevices];

dgl_status get_device(int* dev_out, DeviceState** st_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DGL_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DGL_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    if (cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&st.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&st.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&st.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return DGL_ERR_CUDA;
    if (st.cc_major != 10 || st.cc_minor != 3) return DGL_ERR_UNSUPPORTED;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&st.status), g_status_word) != cudaSuccess)
      return DGL_ERR_CUDA;
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return DGL_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    st.ready = true;
  }
  *dev_out = dev;
  *st_out = &st;
  return DGL_OK;
}

// 2-D tensor map over a row-major [rows, inner] matrix with a 128-byte-wide
// box of box_rows rows and the 128-byte swizzle.  Reads outside
// [0, inner) x [0, rows) return zeros.
bool encode_operand_map(CUtensorMap* map, const void* base, bool e4m3, int64_t inner, int64_t rows,
                        int box_rows, int64_t pitch) {
  const CUtensorMapDataType dt = e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int64_t esize = e4m3 ? 1 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch * esize)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D tensor map over an MN-major bf16 operand stored [K][mn] (row pitch
// `pitch` elements): boxes of 64 MN elements (128 bytes) by 64 K rows with
// the 128-byte swizzle, the layout the MN-major UMMA descriptor reads.
bool encode_operand_map_mn(CUtensorMap* map, const void* base, int64_t mn, int64_t K, int64_t pitch) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(mn), static_cast<cuuint64_t>(K)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch * 2)};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D tensor map over C [rows, cols] (row pitch ldc elements) for 32 x 32
// TMA stores from the epilogue's swizzled staging tile.  Writes outside
// [0, cols) x [0, rows) are dropped.
bool encode_output_map(CUtensorMap* map, void* base, bool f32, int64_t cols, int64_t rows, int64_t ldc) {
  const CUtensorMapDataType dt = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int64_t esize = f32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldc * esize)};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Small direct-mapped cache of encoded tensor maps.  A map depends only on
// the address, extents, pitch, box and element type, so a buffer reused from
// call to call (weights, persistent activations) is encoded once.
struct MapKey {
  const void* base;
  int64_t d0, d1, pitch;
  int box_rows, kind;  // kind: 0 bf16 operand, 1 E4M3 operand, 2 bf16 output, 3 fp32 output, 4 MN-major bf16
  bool operator==(const MapKey& o) const {
    return base == o.base && d0 == o.d0 && d1 == o.d1 && pitch == o.pitch && box_rows == o.box_rows &&
           kind == o.kind;
  }
};
struct MapSlot {
  bool valid = false;
  MapKey key{};
  CUtensorMap map;
};
constexpr int kMapSlots = 512;
std::mutex g_map_mu;
MapSlot g_map_cache[kMapSlots];

size_t map_slot(const MapKey& k) {
  size_t h = reinterpret_cast<uintptr_t>(k.base) >> 4;
  h = h * 0x9E3779B97F4A7C15ull ^ static_cast<size_t>(k.d0);
  h = h * 0x9E3779B97F4A7C15ull ^ static_cast<size_t>(k.d1);
  h = h * 0x9E3779B97F4A7C15ull ^ static_cast<size_t>(k.pitch * 131 + k.box_rows * 7 + k.kind);
  return (h >> 17) % kMapSlots;
}

template <class Encode>
bool cached_map(CUtensorMap* out, const MapKey& key, Encode encode) {
  const size_t slot = map_slot(key);
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (g_map_cache[slot].valid && g_map_cache[slot].key == key) {
      *out = g_map_cache[slot].map;
      return true;
    }
  }
  if (!encode(out)) return false;
  std::lock_guard<std::mutex> lock(g_map_mu);
  g_map_cache[slot].valid = true;
  g_map_cache[slot].key = key;
  g_map_cache[slot].map = *out;
  return true;
}

bool cached_operand_map(CUtensorMap* map, const void* base, bool e4m3, int64_t inner, int64_t rows, int box_rows,
                        int64_t pitch = 0) {
  if (pitch <= 0) pitch = inner;
  const MapKey key{base, inner, rows, pitch, box_rows, e4m3 ? 1 : 0};
  return cached_map(map, key,
                    [&](CUtensorMap* m) { return encode_operand_map(m, base, e4m3, inner, rows, box_rows, pitch); });
}

bool cached_operand_map_mn(CUtensorMap* map, const void* base, int64_t mn, int64_t K, int64_t pitch) {
  const MapKey key{base, mn, K, pitch, 64, 4};
  return cached_map(map, key, [&](CUtensorMap* m) { return encode_operand_map_mn(m, base, mn, K, pitch); });
}

bool cached_output_map(CUtensorMap* map, void* base, bool f32, int64_t cols, int64_t rows, int64_t ldc) {
  const MapKey key{base, cols, rows, ldc, 32, f32 ? 3 : 2};
  return cached_map(map, key, [&](CUtensorMap* m) { return encode_output_map(m, base, f32, cols, rows, ldc); });
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct Problem {
  int dtype, out;
  const void *A, *B;
  const float *sa, *sb;
  void* C;
  int64_t M, N, K, m, n;
  // linear-layer epilogue (dgl_linear): bias per column, activation, gated up projection
  const float* bias = nullptr;
  int act = 0;
  int gated = 0;
  // operand layouts (dgl_gemm_bf16_ex): MN-major A is [K][m], B is [K][n];
  // lda / ldb are row pitches in elements (0: the packed pitch)
  int a_mn = 0;
  int b_mn = 0;
  int64_t lda = 0;
  int64_t ldb = 0;
};

dgl_status validate(Problem& pr) {
  if (pr.dtype != DGL_DTYPE_BF16 && pr.dtype != DGL_DTYPE_E4M3) return DGL_ERR_ARG;
  if (pr.out != DGL_OUT_BF16 && pr.out != DGL_OUT_F32) return DGL_ERR_ARG;
  if (pr.M < 0 || pr.N < 0 || pr.K < 0 || pr.m < 0 || pr.n < 0) return DGL_ERR_ARG;
  if (pr.m == 0) pr.m = pr.M;
  if (pr.n == 0) pr.n = pr.N;
  if (pr.m > pr.M || pr.n > pr.N) return DGL_ERR_ARG;
  if (pr.act < DGL_ACT_NONE || pr.act > DGL_ACT_SILU || (pr.gated != 0 && pr.gated != 1)) return DGL_ERR_ARG;
  if (pr.M > INT32_MAX || pr.N > INT32_MAX || pr.K > INT32_MAX) return DGL_ERR_SHAPE;
  if (pr.gated && 2 * pr.n > INT32_MAX) return DGL_ERR_SHAPE;  // B holds 2 n rows
  if (pr.bias && !aligned(pr.bias, 4)) return DGL_ERR_ALIGN;
  if (pr.m == 0 || pr.n == 0) return DGL_OK;  // empty product
  if (!pr.C) return DGL_ERR_ARG;
  if (!aligned(pr.C, pr.out == DGL_OUT_F32 ? 4 : 2)) return DGL_ERR_ALIGN;
  if (pr.K == 0) return DGL_OK;  // empty sum: zero fill, operands unused
  if (!pr.A || !pr.B) return DGL_ERR_ARG;
  const int64_t esize = pr.dtype == DGL_DTYPE_E4M3 ? 1 : 2;
  if ((pr.K * esize) % 16 != 0) return DGL_ERR_ALIGN;
  if (!aligned(pr.A, 16) || !aligned(pr.B, 16)) return DGL_ERR_ALIGN;
  if (pr.K * esize > INT32_MAX) return DGL_ERR_SHAPE;
  if (pr.a_mn || pr.b_mn) {
    if (pr.dtype != DGL_DTYPE_BF16 || pr.gated || pr.act || pr.bias) return DGL_ERR_UNSUPPORTED;
  }
  // row pitches: at least the row's extent, and a multiple of 16 bytes (the TMA stride rule)
  const int64_t a_row = pr.a_mn ? pr.m : pr.K, b_row = pr.b_mn ? pr.n : pr.K;
  if (pr.lda == 0) pr.lda = a_row;
  if (pr.ldb == 0) pr.ldb = b_row;
  if (pr.lda < a_row || pr.ldb < b_row) return DGL_ERR_ARG;
  if ((pr.lda * esize) % 16 != 0 || (pr.ldb * esize) % 16 != 0) return DGL_ERR_ALIGN;
  if (pr.lda > INT32_MAX || pr.ldb > INT32_MAX) return DGL_ERR_SHAPE;
  if (pr.dtype == DGL_DTYPE_E4M3) {
    if (!pr.sa || !pr.sb) return DGL_ERR_ARG;
    if (!aligned(pr.sa, 4) || !aligned(pr.sb, 4)) return DGL_ERR_ALIGN;
  }
  return DGL_OK;
}

dgl_status run(Problem pr, const dgl_plan_info* forced, cudaStream_t stream, StaticScratch* fixed = nullptr) {
  dgl_status st = validate(pr);
  if (st != DGL_OK) return st;
  if (pr.m == 0 || pr.n == 0) return DGL_OK;
  int dev = 0;
  DeviceState* ds = nullptr;
  st = get_device(&dev, &ds);
  if (st != DGL_OK) return st;
  if (pr.K == 0) {
    return launch_zero_fill(pr.out, pr.C, pr.N, static_cast<int>(pr.m), static_cast<int>(pr.n), stream) ==
                   cudaSuccess
               ? DGL_OK
               : DGL_ERR_CUDA;
  }

  // The linear-layer epilogue runs in its own kernel variants (128- and
  // 256-wide tiles, CTA pairs when gated) and on the decode path (not gated).
  const bool linear = pr.act != 0 || pr.bias != nullptr || pr.gated != 0;
  dgl_plan_info plan;
  if (forced) {
    if (forced->path == DGL_PATH_DECODE) {
      if (pr.m > kDecodeMaxM || pr.gated || pr.a_mn || pr.b_mn || pr.lda != pr.K || pr.ldb != pr.K)
        return DGL_ERR_UNSUPPORTED;
      fill_decode_plan(pr.dtype, pr.out, pr.m, pr.n, pr.K, ds->num_sms, &plan);
    } else if (forced->path == DGL_PATH_TC) {
      if (!tc_supported_tile(forced->tile_m, forced->tile_n)) return DGL_ERR_UNSUPPORTED;
      if (linear && !tc_supported_epi_tile(forced->tile_m, forced->tile_n, pr.gated != 0)) return DGL_ERR_UNSUPPORTED;
      fill_tc_plan(pr.dtype, pr.out, pr.m, pr.gated ? 2 * pr.n : pr.n, pr.K, forced->tile_m, forced->tile_n,
                   ds->num_sms, &plan, forced->stream_k ? 1 : 0);
      plan.split_tail = forced->split_tail && !plan.stream_k ? 1 : 0;
    } else {
      return DGL_ERR_UNSUPPORTED;
    }
    if (forced->grid > 0) plan.grid = forced->grid;
  } else if (linear) {
    choose_linear_plan(pr.dtype, pr.out, pr.m, pr.n, pr.K, pr.gated != 0, ds->num_sms, &plan);
  } else if (pr.a_mn || pr.b_mn || pr.lda != pr.K || pr.ldb != pr.K) {
    // the decode path reads packed K-major operands only
    choose_plan(pr.dtype, pr.out, pr.m, pr.n, pr.K, ds->num_sms, &plan);
    if (plan.path != DGL_PATH_TC) fill_tc_plan(pr.dtype, pr.out, pr.m, pr.n, pr.K, 128, 128, ds->num_sms, &plan, 0);
  } else {
    PlanKey key{dev, pr.dtype, pr.out, pr.m, pr.n, pr.K};
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_plans.find(key);
    if (it == g_plans.end()) {
      choose_plan(pr.dtype, pr.out, pr.m, pr.n, pr.K, ds->num_sms, &plan);
      g_plans.emplace(key, plan);
    } else {
      plan = it->second;
    }
  }

  const bool e4m3 = pr.dtype == DGL_DTYPE_E4M3;
  const int esize = e4m3 ? 1 : 2;
  if (plan.path == DGL_PATH_DECODE) {
    const int parts = decode_parts(pr.n, ds->num_sms);
    const int rows_lo = static_cast<int>(pr.n / parts);
    const int rows_hi = static_cast<int>((pr.n + parts - 1) / parts);
    CUtensorMap ta, tb_lo, tb_hi;
    if (!cached_operand_map(&ta, pr.A, e4m3, pr.K, pr.m, static_cast<int>(pr.m)) ||
        !cached_operand_map(&tb_lo, pr.B, e4m3, pr.K, pr.n, rows_lo) ||
        !cached_operand_map(&tb_hi, pr.B, e4m3, pr.K, pr.n, rows_hi))
      return DGL_ERR_CUDA;
    DecodeParams p;
    p.sa = pr.sa;
    p.sb = pr.sb;
    p.C = pr.C;
    p.ldc = pr.N;
    p.m = static_cast<int>(pr.m);
    p.n = static_cast<int>(pr.n);
    p.row_bytes = static_cast<int>(pr.K * esize);
    p.parts = parts;
    p.rows_hi = rows_hi;
    const int nk = static_cast<int>((pr.K * esize + 127) / 128);
    const int g = decode_group(rows_hi, nk);
    int ks = decode_ksteps(rows_hi, nk, g);
    if (forced && forced->tile_k > 0) {
      // a forced plan may choose the stage width (K elements, a multiple of
      // 128 bytes and of the group's steps)
      const int want = static_cast<int>(forced->tile_k * esize / 128);
      if (want < 1 || want > 16 || want % g != 0 || forced->tile_k * esize % 128 != 0 ||
          decode_stages(rows_hi, want, g) < 2)
        return DGL_ERR_UNSUPPORTED;
      ks = want;
    }
    p.group = g;
    p.ksteps = ks;
    p.b_plane_bytes = decode_plane_bytes(rows_hi, g);
    p.stage_bytes = decode_stage_bytes(rows_hi, ks, g);
    p.stages = decode_stages(rows_hi, ks, g);
    p.status = ds->status;
    p.bias = pr.bias;
    p.act = pr.act;
    const int grid = forced && forced->grid > 0 ? (forced->grid < parts ? forced->grid : parts)
                                                : decode_grid(pr.n, ds->num_sms);
    return launch_decode(pr.dtype, pr.out, ta, tb_lo, tb_hi, p, grid, stream) == cudaSuccess ? DGL_OK
                                                                                            : DGL_ERR_CUDA;
  }

  CUtensorMap ta, tb, tc;
  // each CTA of a pair loads its own 128 rows of A and half the tile's rows of B
  const int cg = plan.cta_group == 2 ? 2 : 1;
  // a gated layer's B holds the gate rows, then the up rows
  const int64_t b_rows = pr.gated ? 2 * pr.n : pr.n;
  const bool map_ok =
      (pr.a_mn ? cached_operand_map_mn(&ta, pr.A, pr.m, pr.K, pr.lda)
               : cached_operand_map(&ta, pr.A, e4m3, pr.K, pr.m, 128, pr.lda)) &&
      (pr.b_mn ? cached_operand_map_mn(&tb, pr.B, b_rows, pr.K, pr.ldb)
               : cached_operand_map(&tb, pr.B, e4m3, pr.K, b_rows, plan.tile_n / cg, pr.ldb));
  if (!map_ok) return DGL_ERR_CUDA;
  // B with half-height boxes, for the half tiles of a split tail (else unused)
  CUtensorMap tbh = tb;
  if (plan.split_tail && !pr.b_mn && plan.tile_n == 256 &&
      !cached_operand_map(&tbh, pr.B, e4m3, pr.K, b_rows, plan.tile_n / cg / 2, pr.ldb))
    return DGL_ERR_CUDA;
  const bool f32 = pr.out == DGL_OUT_F32;
  const bool c_tma = aligned(pr.C, 16) && (pr.N * (f32 ? 4 : 2)) % 16 == 0;
  std::memset(&tc, 0, sizeof(tc));
  if (c_tma && !cached_output_map(&tc, pr.C, f32, pr.n, pr.m, pr.N)) return DGL_ERR_CUDA;
  TcParams p;
  p.C = pr.C;
  p.ldc = pr.N;
  p.m = static_cast<int>(pr.m);
  p.n = static_cast<int>(pr.n);
  p.K = static_cast<int>(pr.K);
  p.sa = pr.sa;
  p.sb = pr.sb;
  p.tiles_m = static_cast<int>((pr.m + plan.tile_m - 1) / plan.tile_m);
  // a gated tile's MMA covers tile_n rows of B: tile_n / 2 output columns
  const int out_w = pr.gated ? plan.tile_n / 2 : plan.tile_n;
  p.tiles_n = static_cast<int>((pr.n + out_w - 1) / out_w);
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.num_kb = static_cast<int>((pr.K * esize + 127) / 128);
  p.group_m = 16;
  p.c_tma = c_tma ? 1 : 0;
  p.status = ds->status;
  p.bias = pr.bias;
  p.act = pr.act;
  p.gated = pr.gated;
  p.n_up = static_cast<int>(pr.n);
  p.a_mn = pr.a_mn;
  p.b_mn = pr.b_mn;
  // grid counts CTAs; a pair per tile when cg == 2
  int grid = plan.grid > 0 ? plan.grid : p.num_tiles * cg;
  if (!plan.stream_k && grid > p.num_tiles * cg) grid = p.num_tiles * cg;
  if (grid > ds->num_sms) grid = ds->num_sms;
  grid = grid / cg * cg;
  if (grid < cg) grid = cg;
  p.workers = grid / cg;
  p.dp_tiles = p.num_tiles;
  p.sk_units = 0;
  p.half_tiles = 0;
  p.ws = nullptr;
  p.flags = nullptr;
  p.epoch = 0;
  if (plan.split_tail && !plan.stream_k && !pr.gated && plan.tile_n == 256 && p.num_tiles > p.workers) {
    // the last, partial wave as half tiles, one per worker
    const int tail = p.num_tiles % p.workers;
    if (tail > 0 && 2 * tail <= p.workers) {
      p.dp_tiles = p.num_tiles - tail;
      p.half_tiles = 2 * tail;
    }
  }
  if (plan.stream_k && p.num_tiles % p.workers != 0) {
    p.dp_tiles = p.num_tiles / p.workers * p.workers;
    p.sk_units = static_cast<int64_t>(p.num_tiles - p.dp_tiles) * p.num_kb;
    const size_t slot_floats = static_cast<size_t>(128) * plan.tile_n;
    const size_t bytes = sizeof(float) * slot_floats * static_cast<size_t>(grid);
    if (fixed) {
      // the caller's problem needs more partial tiles than the array holds
      if (bytes > fixed->ws_bytes || grid > fixed->nflags) return DGL_ERR_SHAPE;
      std::lock_guard<std::mutex> lock(g_mu);
      if (fixed->epoch == INT32_MAX) {
        // epochs ran out: clear the flags so that counting can restart
        if (cudaMemsetAsync(fixed->flags, 0, sizeof(int) * fixed->nflags, stream) != cudaSuccess) return DGL_ERR_CUDA;
        fixed->epoch = 0;
      }
      p.ws = fixed->ws;
      p.flags = fixed->flags;
      p.epoch = ++fixed->epoch;
    } else {
      const dgl_status wst = acquire_workspace(dev, stream, bytes, grid, &p.ws, &p.flags, &p.epoch);
      if (wst != DGL_OK) return wst;
    }
  }
  if (ds->smem_optin < 232448) return DGL_ERR_UNSUPPORTED;  // every variant is sized for 227 KB
  const bool row_staging = !c_tma && !f32;
  cudaError_t e;
  if (linear)
    e = e4m3 ? launch_tc_e4m3_epi(pr.out, plan.tile_m, plan.tile_n, row_staging, ta, tb, tbh, tc, p, grid, stream)
             : launch_tc_bf16_epi(pr.out, plan.tile_m, plan.tile_n, row_staging, ta, tb, tbh, tc, p, grid, stream);
  else
    e = e4m3 ? launch_tc_e4m3(pr.out, plan.tile_m, plan.tile_n, row_staging, ta, tb, tbh, tc, p, grid, stream)
             : launch_tc_bf16(pr.out, plan.tile_m, plan.tile_n, row_staging, ta, tb, tbh, tc, p, grid, stream);
  return e == cudaSuccess ? DGL_OK : DGL_ERR_CUDA;
}

// Block-scaled FP4 (MXFP4): A and B as byte tensors of K / 2 bytes per row
// (TMA moves the packed E2M1 codes untouched), E8M0 scales read by the
// kernel's scale warps, 128 x 256 tiles.
dgl_status run_mxfp4(Problem pr, const uint8_t* sfa, const uint8_t* sfb, cudaStream_t stream) {
  if (pr.out != DGL_OUT_BF16 && pr.out != DGL_OUT_F32) return DGL_ERR_ARG;
  if (pr.M < 0 || pr.N < 0 || pr.K < 0 || pr.m < 0 || pr.n < 0) return DGL_ERR_ARG;
  if (pr.m == 0) pr.m = pr.M;
  if (pr.n == 0) pr.n = pr.N;
  if (pr.m > pr.M || pr.n > pr.N) return DGL_ERR_ARG;
  if (pr.M > INT32_MAX || pr.N > INT32_MAX || pr.K > INT32_MAX) return DGL_ERR_SHAPE;
  if (pr.m == 0 || pr.n == 0) return DGL_OK;
  if (!pr.C) return DGL_ERR_ARG;
  if (!aligned(pr.C, pr.out == DGL_OUT_F32 ? 4 : 2)) return DGL_ERR_ALIGN;
  if (pr.K % 32 != 0) return DGL_ERR_ALIGN;
  if (pr.K > 0) {
    if (!pr.A || !pr.B || !sfa || !sfb) return DGL_ERR_ARG;
    if (!aligned(pr.A, 16) || !aligned(pr.B, 16)) return DGL_ERR_ALIGN;
  }
  int dev = 0;
  DeviceState* ds = nullptr;
  dgl_status st = get_device(&dev, &ds);
  if (st != DGL_OK) return st;
  if (pr.K == 0)
    return launch_zero_fill(pr.out, pr.C, pr.N, static_cast<int>(pr.m), static_cast<int>(pr.n), stream) ==
                   cudaSuccess
               ? DGL_OK
               : DGL_ERR_CUDA;
  if (ds->smem_optin < 232448) return DGL_ERR_UNSUPPORTED;
  dgl_plan_info plan;
  fill_mx_plan(pr.out, pr.m, pr.n, pr.K, ds->num_sms, &plan);
  const int64_t row_bytes = pr.K / 2;
  CUtensorMap ta, tb, tc;
  if (!cached_operand_map(&ta, pr.A, true, row_bytes, pr.m, plan.tile_m) ||
      !cached_operand_map(&tb, pr.B, true, row_bytes, pr.n, plan.tile_n))
    return DGL_ERR_CUDA;
  const bool f32 = pr.out == DGL_OUT_F32;
  const bool c_tma = aligned(pr.C, 16) && (pr.N * (f32 ? 4 : 2)) % 16 == 0;
  std::memset(&tc, 0, sizeof(tc));
  if (c_tma && !cached_output_map(&tc, pr.C, f32, pr.n, pr.m, pr.N)) return DGL_ERR_CUDA;
  TcParams p;
  std::memset(&p, 0, sizeof(p));
  p.C = pr.C;
  p.ldc = pr.N;
  p.m = static_cast<int>(pr.m);
  p.n = static_cast<int>(pr.n);
  p.K = static_cast<int>(pr.K);
  p.tiles_m = static_cast<int>((pr.m + plan.tile_m - 1) / plan.tile_m);
  p.tiles_n = static_cast<int>((pr.n + plan.tile_n - 1) / plan.tile_n);
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.num_kb = static_cast<int>((row_bytes + 127) / 128);
  p.group_m = 16;
  p.c_tma = c_tma ? 1 : 0;
  p.status = ds->status;
  p.n_up = p.n;
  const int grid = plan.grid;
  p.workers = grid;
  p.dp_tiles = p.num_tiles;
  p.sfa = sfa;
  p.sfb = sfb;
  p.sf_vec8 = (pr.K % 256 == 0 && aligned(sfa, 8) && aligned(sfb, 8)) ? 1 : 0;
  const bool row_staging = !c_tma && !f32;
  return launch_tc_mxfp4(pr.out, row_staging, ta, tb, tc, p, grid, stream) == cudaSuccess ? DGL_OK : DGL_ERR_CUDA;
}

// First use on a device: look up the array's device address and clear its
// flags (synchronous; later calls enqueue work only).
dgl_status noalloc_setup(int dev, StaticScratch** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  StaticScratch& sc = g_noalloc[dev];
  if (!sc.ready) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return DGL_ERR_CUDA;
    uint8_t* base = static_cast<uint8_t*>(ptr);
    int* flags = reinterpret_cast<int*>(base + DGL_NOALLOC_SCRATCH_BYTES);
    if (cudaMemset(flags, 0, sizeof(int) * kNoallocFlags) != cudaSuccess) return DGL_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return DGL_ERR_CUDA;
    sc.ws = reinterpret_cast<float*>(base);
    sc.ws_bytes = DGL_NOALLOC_SCRATCH_BYTES;
    sc.flags = flags;
    sc.nflags = kNoallocFlags;
    sc.epoch = 0;
    sc.ready = true;
  }
  *out = &sc;
  return DGL_OK;
}

}  // namespace
}  // namespace dgl

using namespace dgl;

extern "C" {

dgl_status dgl_gemm_bf16(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t m_valid,
                         int64_t n_valid, int32_t out_dtype, void* stream) {
  Problem pr{DGL_DTYPE_BF16, out_dtype, A, B, nullptr, nullptr, C, M, N, K, m_valid, n_valid};
  return run(pr, nullptr, static_cast<cudaStream_t>(stream));
}

dgl_status dgl_gemm_fp8(const void* A, const void* B, const float* sa, const float* sb, void* C, int64_t M,
                        int64_t N, int64_t K, int64_t m_valid, int64_t n_valid, int32_t out_dtype, void* stream) {
  Problem pr{DGL_DTYPE_E4M3, out_dtype, A, B, sa, sb, C, M, N, K, m_valid, n_valid};
  return run(pr, nullptr, static_cast<cudaStream_t>(stream));
}

dgl_status dgl_gemm_mxfp4(const void* A, const void* B, const uint8_t* sfa, const uint8_t* sfb, void* C, int64_t M,
                          int64_t N, int64_t K, int64_t m_valid, int64_t n_valid, int32_t out_dtype, void* stream) {
  Problem pr{DGL_DTYPE_MXFP4, out_dtype, A, B, nullptr, nullptr, C, M, N, K, m_valid, n_valid};
  return run_mxfp4(pr, sfa, sfb, static_cast<cudaStream_t>(stream));
}

dgl_status dgl_gemm_planned(int32_t dtype, const void* A, const void* B, const float* sa, const float* sb, void* C,
                            int64_t M, int64_t N, int64_t K, int64_t m_valid, int64_t n_valid, int32_t out_dtype,
                            const dgl_plan_info* plan, void* stream) {
  if (!plan) return DGL_ERR_ARG;
  Problem pr{dtype, out_dtype, A, B, dtype == DGL_DTYPE_E4M3 ? sa : nullptr,
             dtype == DGL_DTYPE_E4M3 ? sb : nullptr, C, M, N, K, m_valid, n_valid};
  return run(pr, plan, static_cast<cudaStream_t>(stream));
}

dgl_status dgl_linear(int32_t dtype, const void* A, const void* B, const float* sa, const float* sb,
                      const float* bias, void* C, int64_t M, int64_t N, int64_t K, int64_t m_valid, int64_t n_valid,
                      int32_t out_dtype, int32_t act, int32_t gated, const dgl_plan_info* plan, void* stream) {
  Problem pr{dtype, out_dtype, A, B, dtype == DGL_DTYPE_E4M3 ? sa : nullptr,
             dtype == DGL_DTYPE_E4M3 ? sb : nullptr, C, M, N, K, m_valid, n_valid};
  pr.bias = bias;
  pr.act = act;
  pr.gated = gated;
  return run(pr, plan, static_cast<cudaStream_t>(stream));
}

dgl_status dgl_plan(int32_t dtype, int64_t m, int64_t n, int64_t K, int32_t out_dtype, int32_t num_sms,
                    dgl_plan_info* out) {
  if (!out) return DGL_ERR_ARG;
  if (dtype != DGL_DTYPE_BF16 && dtype != DGL_DTYPE_E4M3 && dtype != DGL_DTYPE_MXFP4) return DGL_ERR_ARG;
  if (out_dtype != DGL_OUT_BF16 && out_dtype != DGL_OUT_F32) return DGL_ERR_ARG;
  if (m < 0 || n < 0 || K < 0) return DGL_ERR_ARG;
  if (m > INT32_MAX || n > INT32_MAX || K > INT32_MAX) return DGL_ERR_SHAPE;
  if (num_sms <= 0) {
    int dev = 0;
    DeviceState* ds = nullptr;
    const dgl_status st = get_device(&dev, &ds);
    if (st != DGL_OK) return st;
    num_sms = ds->num_sms;
  }
  choose_plan(dtype, out_dtype, m, n, K, num_sms, out);
  return DGL_OK;
}

dgl_status dgl_gemm_bf16_ex(int32_t a_major, int32_t b_major, const void* A, int64_t lda, const void* B, int64_t ldb,
                           void* C, int64_t ldc, int64_t m, int64_t n, int64_t K, int32_t out_dtype,
                           const dgl_plan_info* plan, void* stream) {
  if ((a_major != DGL_K_MAJOR && a_major != DGL_MN_MAJOR) || (b_major != DGL_K_MAJOR && b_major != DGL_MN_MAJOR))
    return DGL_ERR_ARG;
  if (lda < 0 || ldb < 0 || ldc < 0 || m < 0 || n < 0) return DGL_ERR_ARG;
  Problem pr{DGL_DTYPE_BF16, out_dtype, A, B, nullptr, nullptr, C, m, ldc == 0 ? n : ldc, K, m, n};
  if (pr.N < n) return DGL_ERR_ARG;
  pr.a_mn = a_major == DGL_MN_MAJOR;
  pr.b_mn = b_major == DGL_MN_MAJOR;
  pr.lda = lda;
  pr.ldb = ldb;
  return run(pr, plan, static_cast<cudaStream_t>(stream));
}

dgl_status dgl_plan_linear(int32_t dtype, int64_t m, int64_t n, int64_t K, int32_t out_dtype, int32_t gated,
                           int32_t num_sms, dgl_plan_info* out) {
  if (!out) return DGL_ERR_ARG;
  if (dtype != DGL_DTYPE_BF16 && dtype != DGL_DTYPE_E4M3) return DGL_ERR_ARG;
  if (out_dtype != DGL_OUT_BF16 && out_dtype != DGL_OUT_F32) return DGL_ERR_ARG;
  if (m < 0 || n < 0 || K < 0 || (gated != 0 && gated != 1)) return DGL_ERR_ARG;
  if (m > INT32_MAX || 2 * n > INT32_MAX || K > INT32_MAX) return DGL_ERR_SHAPE;
  if (num_sms <= 0) {
    int dev = 0;
    DeviceState* ds = nullptr;
    const dgl_status st = get_device(&dev, &ds);
    if (st != DGL_OK) return st;
    num_sms = ds->num_sms;
  }
  choose_linear_plan(dtype, out_dtype, m, n, K, gated != 0, num_sms, out);
  return DGL_OK;
}

dgl_status dgl_tile_metrics(int64_t m, int64_t n, int32_t tile_m, int32_t tile_n, int32_t num_units,
                            dgl_plan_info* out) {
  if (!out || m < 0 || n < 0 || tile_m <= 0 || tile_n <= 0 || num_units <= 0) return DGL_ERR_ARG;
  *out = dgl_plan_info{};
  out->tile_m = tile_m;
  out->tile_n = tile_n;
  tile_metrics(m, n, tile_m, tile_n, num_units, out);
  return DGL_OK;
}

dgl_status dgl_device_status(void* stream) {
  int dev = 0;
  DeviceState* ds = nullptr;
  dgl_status st = get_device(&dev, &ds);
  if (st != DGL_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DGL_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, ds->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return DGL_ERR_CUDA;
  if (word != 0) {
    const int zero = 0;
    if (cudaMemcpy(ds->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return DGL_ERR_CUDA;
    return DGL_ERR_TIMEOUT;
  }
  return DGL_OK;
}

dgl_status dgl_gemm_noalloc(int32_t dtype, const void* A, const void* B, const float* sa, const float* sb, void* C,
                            int64_t M, int64_t N, int64_t K, int64_t m_valid, int64_t n_valid, int32_t out_dtype,
                            void* stream) {
  if (dtype != DGL_DTYPE_BF16 && dtype != DGL_DTYPE_E4M3) return DGL_ERR_ARG;
  Problem pr{dtype, out_dtype, A, B, dtype == DGL_DTYPE_E4M3 ? sa : nullptr,
             dtype == DGL_DTYPE_E4M3 ? sb : nullptr, C, M, N, K, m_valid, n_valid};
  dgl_status st = validate(pr);
  if (st != DGL_OK) return st;
  if (pr.m == 0 || pr.n == 0) return DGL_OK;
  int dev = 0;
  DeviceState* ds = nullptr;
  st = get_device(&dev, &ds);
  if (st != DGL_OK) return st;
  StaticScratch* sc = nullptr;
  st = noalloc_setup(dev, &sc);
  if (st != DGL_OK) return st;
  // the planner's path and tile; on the tcgen05 path the last, partial wave
  // is always split along K (when it has one)
  dgl_plan_info plan;
  choose_plan(pr.dtype, pr.out, pr.m, pr.n, pr.K, ds->num_sms, &plan);
  plan.stream_k = plan.path == DGL_PATH_TC ? 1 : 0;
  plan.grid = 0;
  plan.tile_k = 0;
  return run(pr, &plan, static_cast<cudaStream_t>(stream), sc);
}

const char* dgl_status_string(int32_t status) {
  switch (status) {
    case DGL_OK: return "ok";
    case DGL_ERR_ARG: return "invalid argument";
    case DGL_ERR_ALIGN: return "misaligned pointer or K not a multiple of 16 bytes";
    case DGL_ERR_SHAPE: return "extent out of range";
    case DGL_ERR_UNSUPPORTED: return "unsupported device or plan";
    case DGL_ERR_CUDA: return "CUDA error";
    case DGL_ERR_TIMEOUT: return "a kernel wait timed out";
    default: return "unknown status";
  }
}

int32_t dgl_version(void) { return 100; }

}  // extern "C"

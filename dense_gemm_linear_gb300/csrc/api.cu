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
#include <vector>

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

// Stream-K workspaces: fp32 partial tiles and one flag per partial slot, one
// workspace per (device, stream).  Launches on one stream run in order, so
// they can share it.  A contributor sets its flag to 1 once its partial is
// written; the worker that adds the partial clears it again after reading
// it, so every launch leaves the flags at zero (a CUDA graph replays the same
// launch parameters, which rules out a per-launch tag).  At most
// kWorkspacesPerDevice are kept per device: a new
// stream's workspace replaces the least recently used one (after the device
// has drained, since that stream's kernels may still read it), so a caller
// that makes a stream per request does not grow device memory without bound.
// dgl_shutdown() frees them all.
constexpr int kWorkspacesPerDevice = 4;
struct Workspace {
  int dev = -1;
  cudaStream_t stream = nullptr;
  float* ws = nullptr;
  size_t ws_bytes = 0;
  int* flags = nullptr;
  int nflags = 0;
  uint64_t last_use = 0;
};
std::vector<Workspace> g_workspaces;  // guarded by g_mu
uint64_t g_ws_clock = 0;

void free_workspace(Workspace& w) {
  if (w.ws) cudaFree(w.ws);
  if (w.flags) cudaFree(w.flags);
  w.ws = nullptr;
  w.flags = nullptr;
  w.ws_bytes = 0;
  w.nflags = 0;
}

// Whether (dev, stream) already has a workspace of at least bytes / nflags.
bool workspace_ready(int dev, cudaStream_t stream, size_t bytes, int nflags) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (const Workspace& x : g_workspaces)
    if (x.dev == dev && x.stream == stream) return x.ws && x.ws_bytes >= bytes && x.nflags >= nflags;
  return false;
}

dgl_status acquire_workspace(int dev, cudaStream_t stream, size_t bytes, int nflags, float** ws, int** flags) {
  std::lock_guard<std::mutex> lock(g_mu);
  Workspace* w = nullptr;
  int on_dev = 0;
  for (Workspace& x : g_workspaces) {
    if (x.dev != dev) continue;
    ++on_dev;
    if (x.stream == stream) w = &x;
  }
  if (!w) {
    if (on_dev >= kWorkspacesPerDevice) {
      // evict the device's least recently used workspace once its work is done
      size_t lru = g_workspaces.size();
      for (size_t i = 0; i < g_workspaces.size(); ++i)
        if (g_workspaces[i].dev == dev && (lru == g_workspaces.size() || g_workspaces[i].last_use < g_workspaces[lru].last_use))
          lru = i;
      if (cudaDeviceSynchronize() != cudaSuccess) return DGL_ERR_CUDA;
      free_workspace(g_workspaces[lru]);
      g_workspaces.erase(g_workspaces.begin() + static_cast<std::ptrdiff_t>(lru));
    }
    Workspace fresh;
    fresh.dev = dev;
    fresh.stream = stream;
    g_workspaces.push_back(fresh);
    w = &g_workspaces.back();
  }
  if (w->ws_bytes < bytes || w->nflags < nflags) {
    // growing frees the old buffers, which waits for work still using them
    free_workspace(*w);
    const size_t want = bytes > (size_t(24) << 20) ? bytes : (size_t(24) << 20);
    const int want_flags = nflags > 512 ? nflags : 512;
    if (cudaMalloc(reinterpret_cast<void**>(&w->ws), want) != cudaSuccess) {
      w->ws = nullptr;
      return DGL_ERR_CUDA;
    }
    if (cudaMalloc(reinterpret_cast<void**>(&w->flags), sizeof(int) * want_flags) != cudaSuccess) {
      w->flags = nullptr;
      free_workspace(*w);
      return DGL_ERR_CUDA;
    }
    w->ws_bytes = want;
    w->nflags = want_flags;
    if (cudaMemset(w->flags, 0, sizeof(int) * want_flags) != cudaSuccess) {
      free_workspace(*w);
      return DGL_ERR_CUDA;
    }
  }
  w->last_use = ++g_ws_clock;
  *ws = w->ws;
  *flags = w->flags;
  return DGL_OK;
}

// ---- scratch of dgl_gemm_noalloc: a fixed device array instead of cudaMalloc.
// Layout: DGL_NOALLOC_SCRATCH_BYTES of fp32 partial tiles, then one flag per
// partial slot (zero between launches).  Every device that loads the library
// holds it until exit.
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
};
StaticScratch g_noalloc[kMaxDevices];
std::mutex g_noalloc_mu;  // set-up of g_noalloc


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

// 3-D tensor map over a decode call's A ([m][K] row-major, K a whole number
// of 128-byte steps) as [K steps][m rows][128 bytes]: a box of 16 rows by
// `steps` K steps lands as `steps` consecutive 2 KB planes of 16 rows, rows
// past m and steps past K filled with zeros, with the 128-byte swizzle.
bool encode_decode_a_map(CUtensorMap* map, const void* base, bool e4m3, int64_t K, int64_t m, int steps) {
  const int64_t esize = e4m3 ? 1 : 2;
  const int64_t nk = K * esize / 128;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(128 / esize), static_cast<cuuint64_t>(m), static_cast<cuuint64_t>(nk)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(K * esize), 128};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / esize), 16, static_cast<cuuint32_t>(steps)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D tensor map over packed 4-bit codes, [rows][K / 2] bytes (element 2t in
// the low four bits of byte t), with a box of 128 elements by box_rows rows
// and the 128-byte swizzle.  The 16U4_ALIGN16B type lands each 16 elements
// (8 bytes) in a 16-byte unit of shared memory, the layout the kind::f8f6f4
// MMA reads a 4-bit operand from: a box row spans 128 bytes there, as an
// E4M3 row does.  Needs K a multiple of 128, a 32-byte-aligned base and a
// row pitch that is a multiple of 32 bytes.
bool encode_w4_map(CUtensorMap* map, const void* base, int64_t K, int64_t rows, int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
  cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
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

// 2-D tensor map over C [rows, cols] (row pitch ldc elements) for 32-column
// TMA stores of box_rows rows (32, or 16 for 64-row tiles) from the
// epilogue's swizzled staging tile.  Writes outside [0, cols) x [0, rows) are
// dropped.
bool encode_output_map(CUtensorMap* map, void* base, bool f32, int64_t cols, int64_t rows, int64_t ldc,
                       int box_rows) {
  const CUtensorMapDataType dt = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int64_t esize = f32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldc * esize)};
  cuuint32_t box[2] = {32, static_cast<cuuint32_t>(box_rows)};
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
  int box_rows, kind;  // kind: 0 bf16 operand, 1 E4M3 operand, 2 bf16 output, 3 fp32 output, 4 MN-major bf16,
                       // 5 packed 4-bit operand, 6 / 7 a decode call's 3-D bf16 / E4M3 A (box_rows: K steps)
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

bool cached_w4_map(CUtensorMap* map, const void* base, int64_t K, int64_t rows, int box_rows) {
  const MapKey key{base, K, rows, K / 2, box_rows, 5};
  return cached_map(map, key, [&](CUtensorMap* m) { return encode_w4_map(m, base, K, rows, box_rows); });
}

// B's map: E4M3 / bf16 codes, or packed 4-bit codes (w4).
bool cached_b_map(CUtensorMap* map, const void* base, bool e4m3, bool w4, int64_t K, int64_t rows, int box_rows,
                  int64_t pitch = 0) {
  return w4 ? cached_w4_map(map, base, K, rows, box_rows)
            : cached_operand_map(map, base, e4m3, K, rows, box_rows, pitch);
}

bool cached_operand_map_mn(CUtensorMap* map, const void* base, int64_t mn, int64_t K, int64_t pitch) {
  const MapKey key{base, mn, K, pitch, 64, 4};
  return cached_map(map, key, [&](CUtensorMap* m) { return encode_operand_map_mn(m, base, mn, K, pitch); });
}

bool cached_output_map(CUtensorMap* map, void* base, bool f32, int64_t cols, int64_t rows, int64_t ldc,
                       int box_rows = 32) {
  const MapKey key{base, cols, rows, ldc, box_rows, f32 ? 3 : 2};
  return cached_map(map, key,
                    [&](CUtensorMap* m) { return encode_output_map(m, base, f32, cols, rows, ldc, box_rows); });
}

// L2 prefetch before the wait for the previous kernel on the stream
// (measured on GB300, back to back, operands rotated through 3x L2):
//  * decode: a CTA prefetches its first ring's worth of B when its part is
//    at least twice the ring (1 and 16 x 11008 x 4096: 16.6 -> 14.6 and
//    17.1 -> 15.0 us); with parts about one ring long (16 x 4096 x 4096) any
//    prefetch measured slower (9.9 -> 10.2-11.8 us), since the ring's own
//    loads follow at once;
//  * tile kernel: the first ring of its first tile when K spans at least
//    four rings (4096^3 bf16 79.1 -> 77.9 us); never for short K, where the
//    ring's loads follow at once.
constexpr int kDecodeRingBytes = 196608;

// The E2M1 code of the kind::f8f6f4 instruction descriptor's A / B format
// fields (bits 7-9 / 10-12; E4M3 is 0).
constexpr uint32_t kIdescE2M1 = 5;

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
  // W4A8 (dgl_gemm_w4a8): dtype E4M3 for A, B holds packed E2M1 codes (K / 2
  // bytes a row)
  int w4 = 0;
  // programmatic dependent launch mode of the kernel (PDL_*; dgl_gemm_batch)
  int pdl_mode = PDL_SERIAL;
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
  // packed 4-bit B: whole 128-element boxes along K, a 32-byte-aligned base
  // (the tensor-map rules of the 16U4_ALIGN16B type)
  if (pr.w4 && (pr.K % 128 != 0 || !aligned(pr.B, 32))) return DGL_ERR_ALIGN;
  if (pr.K * esize > INT32_MAX) return DGL_ERR_SHAPE;
  if (pr.a_mn || pr.b_mn) {
    if (pr.dtype != DGL_DTYPE_BF16 || pr.gated || pr.act || pr.bias) return DGL_ERR_UNSUPPORTED;
  }
  // row pitches: at least the row's extent, and a multiple of 16 bytes (the TMA stride rule)
  const int64_t a_row = pr.a_mn ? pr.m : pr.K, b_row = pr.b_mn ? pr.n : pr.K;
  if (pr.lda == 0) pr.lda = a_row;
  if (pr.ldb == 0) pr.ldb = b_row;
  if (pr.lda < a_row || pr.ldb < b_row) return DGL_ERR_ARG;
  if ((pr.lda * esize) % 16 != 0 || (!pr.w4 && (pr.ldb * esize) % 16 != 0)) return DGL_ERR_ALIGN;
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
      // 64-row tiles read K-major operands only
      if (forced->tile_m == 64 && (pr.a_mn || pr.b_mn)) return DGL_ERR_UNSUPPORTED;
      if (linear && !tc_supported_epi_tile(forced->tile_m, forced->tile_n, pr.gated != 0)) return DGL_ERR_UNSUPPORTED;
      fill_tc_plan(pr.dtype, pr.out, pr.m, pr.gated ? 2 * pr.n : pr.n, pr.K, forced->tile_m, forced->tile_n,
                   ds->num_sms, &plan, forced->stream_k > 0 ? forced->stream_k : 0);
      plan.split_tail = forced->split_tail && !plan.stream_k && forced->tile_m != 64 ? 1 : 0;
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
    if (plan.tile_m == 64 && (pr.a_mn || pr.b_mn))
      fill_tc_plan(pr.dtype, pr.out, pr.m, pr.n, pr.K, 128, plan.tile_n, ds->num_sms, &plan, 0);
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
        !cached_b_map(&tb_lo, pr.B, e4m3, pr.w4, pr.K, pr.n, rows_lo) ||
        !cached_b_map(&tb_hi, pr.B, e4m3, pr.w4, pr.K, pr.n, rows_hi))
      return DGL_ERR_CUDA;
    DecodeParams p;
    // B's rows are the MMA's A operand here: E2M1 goes in the A format field
    p.idesc_or = pr.w4 ? kIdescE2M1 << 7 : 0u;
    p.b_tx_shift = pr.w4 ? 1 : 0;
    p.prefetch_planes = static_cast<int64_t>(rows_hi) * pr.K * esize >= 2 * kDecodeRingBytes
                            ? kDecodeRingBytes / (rows_hi * 128)
                            : 0;
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
    p.a3d = 0;
    if ((pr.K * esize) % 128 == 0) {
      const MapKey ak{pr.A, pr.K, pr.m, pr.K, ks, e4m3 ? 7 : 6};
      if (!cached_map(&ta, ak, [&](CUtensorMap* m) { return encode_decode_a_map(m, pr.A, e4m3, pr.K, pr.m, ks); }))
        return DGL_ERR_CUDA;
      p.a3d = 1;
    }
    p.group = g;
    p.ksteps = ks;
    p.b_plane_bytes = decode_plane_bytes(rows_hi, g);
    p.stage_bytes = decode_stage_bytes(rows_hi, ks, g);
    p.stages = decode_stages(rows_hi, ks, g);
    p.status = ds->status;
    p.bias = pr.bias;
    p.act = pr.act;
    p.pdl_mode = pr.pdl_mode;
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
               : cached_operand_map(&ta, pr.A, e4m3, pr.K, pr.m, plan.tile_m == 64 ? 64 : 128, pr.lda)) &&
      (pr.b_mn ? cached_operand_map_mn(&tb, pr.B, b_rows, pr.K, pr.ldb)
               : cached_b_map(&tb, pr.B, e4m3, pr.w4, pr.K, b_rows, plan.tile_n / cg, pr.ldb));
  if (!map_ok) return DGL_ERR_CUDA;
  // B with half-height boxes, for the half tiles of a split tail (else unused)
  CUtensorMap tbh = tb;
  if (plan.split_tail && !pr.b_mn && plan.tile_n == 256 &&
      !cached_b_map(&tbh, pr.B, e4m3, pr.w4, pr.K, b_rows, plan.tile_n / cg / 2, pr.ldb))
    return DGL_ERR_CUDA;
  const bool f32 = pr.out == DGL_OUT_F32;
  const bool c_tma = aligned(pr.C, 16) && (pr.N * (f32 ? 4 : 2)) % 16 == 0;
  std::memset(&tc, 0, sizeof(tc));
  if (c_tma && !cached_output_map(&tc, pr.C, f32, pr.n, pr.m, pr.N, plan.tile_m == 64 ? 16 : 32)) return DGL_ERR_CUDA;
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
  p.idesc_or = pr.w4 ? kIdescE2M1 << 10 : 0u;  // E2M1 in the B format field
  p.b_tx_shift = pr.w4 ? 1 : 0;
  p.prefetch_stages = p.num_kb >= 4 * plan.stages ? plan.stages : 0;
  p.pdl_mode = pr.pdl_mode;
  // A split schedule needs the stream's workspace.  A stream being captured
  // into a CUDA graph cannot have one allocated, so a captured call on a
  // stream without one runs the data-parallel schedule instead.
  bool split = plan.stream_k != 0;
  if (split && !fixed) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return DGL_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone &&
        !workspace_ready(dev, stream, sizeof(float) * 128 * static_cast<size_t>(plan.tile_n) * ds->num_sms,
                         ds->num_sms))
      split = false;
  }
  // grid counts CTAs; a pair per tile when cg == 2
  int grid = plan.grid > 0 ? plan.grid : p.num_tiles * cg;
  if (!split && grid > p.num_tiles * cg) grid = p.num_tiles * cg;
  if (grid > ds->num_sms) grid = ds->num_sms;
  grid = grid / cg * cg;
  if (grid < cg) grid = cg;
  p.workers = grid / cg;
  p.dp_tiles = p.num_tiles;
  p.sk_units = 0;
  p.sk_workers = p.workers;
  p.half_tiles = 0;
  p.ws = nullptr;
  p.flags = nullptr;
  if (plan.split_tail && !split && !pr.gated && plan.tile_n == 256 && p.num_tiles > p.workers) {
    // the last, partial wave as half tiles, one per worker
    const int tail = p.num_tiles % p.workers;
    if (tail > 0 && 2 * tail <= p.workers) {
      p.dp_tiles = p.num_tiles - tail;
      p.half_tiles = 2 * tail;
    }
  }
  if (split && p.num_tiles % p.workers != 0) {
    p.dp_tiles = p.num_tiles / p.workers * p.workers;
    p.sk_units = static_cast<int64_t>(p.num_tiles - p.dp_tiles) * p.num_kb;
    // stream_k = S >= 2: each tail tile's k-stages in S equal ranges, one per
    // worker (tail x S workers), instead of all workers sharing them
    const int tail = p.num_tiles - p.dp_tiles;
    if (plan.stream_k >= 2 && static_cast<int64_t>(tail) * plan.stream_k <= p.workers)
      p.sk_workers = tail * plan.stream_k;
    const size_t slot_floats = static_cast<size_t>(128) * plan.tile_n;
    const size_t bytes = sizeof(float) * slot_floats * static_cast<size_t>(grid);
    if (fixed) {
      // the caller's problem needs more partial tiles than the array holds
      if (bytes > fixed->ws_bytes || grid > fixed->nflags) return DGL_ERR_SHAPE;
      p.ws = fixed->ws;
      p.flags = fixed->flags;
    } else {
      const dgl_status wst = acquire_workspace(dev, stream, bytes, grid, &p.ws, &p.flags);
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
dgl_status validate_mxfp4(Problem& pr, const uint8_t* sfa, const uint8_t* sfb) {
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
  return DGL_OK;
}

dgl_status run_mxfp4(Problem pr, const uint8_t* sfa, const uint8_t* sfb, cudaStream_t stream) {
  const dgl_status vst = validate_mxfp4(pr, sfa, sfb);
  if (vst != DGL_OK) return vst;
  if (pr.m == 0 || pr.n == 0) return DGL_OK;
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
  p.pdl_mode = pr.pdl_mode;
  const bool row_staging = !c_tma && !f32;
  return launch_tc_mxfp4(pr.out, row_staging, ta, tb, tc, p, grid, stream) == cudaSuccess ? DGL_OK : DGL_ERR_CUDA;
}

// First use on a device: look up the array's device address and clear its
// flags (synchronous; later calls enqueue work only).
// Whether the stream-K split of a plan fits the array on a device of num_sms
// SMs: one 128 x tile_n fp32 slot and one flag per CTA of the grid.  On 152
// SMs every plan fits (at most 152 slots of 128 KB).
bool noalloc_fits(const Problem& pr, const dgl_plan_info& plan, int num_sms) {
  if (plan.path != DGL_PATH_TC ||
      !stream_k_eligible(pr.m, pr.n, pr.K, pr.dtype, plan.tile_m, plan.tile_n, num_sms))
    return true;
  const int cg = plan.cta_group == 2 ? 2 : 1;
  const int64_t grid = static_cast<int64_t>(num_sms / cg) * cg;
  const int64_t bytes = static_cast<int64_t>(sizeof(float)) * 128 * plan.tile_n * grid;
  return bytes <= static_cast<int64_t>(DGL_NOALLOC_SCRATCH_BYTES) && grid <= kNoallocFlags;
}

// Its own lock: the synchronous set-up must not hold up other threads' calls,
// which take g_mu.
dgl_status noalloc_setup(int dev, StaticScratch** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
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

dgl_status dgl_gemm_w4a8(const void* A, const void* B, const float* sa, const float* sb, void* C, int64_t M,
                         int64_t N, int64_t K, int64_t m_valid, int64_t n_valid, int32_t out_dtype, void* stream) {
  Problem pr{DGL_DTYPE_E4M3, out_dtype, A, B, sa, sb, C, M, N, K, m_valid, n_valid};
  pr.w4 = 1;
  return run(pr, nullptr, static_cast<cudaStream_t>(stream));
}

dgl_status dgl_gemm_mxfp4(const void* A, const void* B, const uint8_t* sfa, const uint8_t* sfb, void* C, int64_t M,
                          int64_t N, int64_t K, int64_t m_valid, int64_t n_valid, int32_t out_dtype, void* stream) {
  Problem pr{DGL_DTYPE_MXFP4, out_dtype, A, B, nullptr, nullptr, C, M, N, K, m_valid, n_valid};
  return run_mxfp4(pr, sfa, sfb, static_cast<cudaStream_t>(stream));
}

dgl_status dgl_gemm_batch(const dgl_gemm_desc* items, int32_t count, void* stream) {
  if (count < 0 || (count > 0 && !items)) return DGL_ERR_ARG;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto problem = [](const dgl_gemm_desc& d) {
    const bool e4m3 = d.dtype == DGL_DTYPE_E4M3 || d.dtype == DGL_DTYPE_W4A8;
    Problem pr{e4m3 ? DGL_DTYPE_E4M3 : d.dtype, d.out_dtype, d.A, d.B,
               e4m3 ? static_cast<const float*>(d.scale_a) : nullptr,
               e4m3 ? static_cast<const float*>(d.scale_b) : nullptr, d.C, d.M, d.N, d.K, d.m_valid, d.n_valid};
    pr.w4 = d.dtype == DGL_DTYPE_W4A8 ? 1 : 0;
    return pr;
  };
  // every item is checked before any is enqueued
  for (int32_t i = 0; i < count; ++i) {
    const dgl_gemm_desc& d = items[i];
    Problem pr = problem(d);
    dgl_status st = DGL_ERR_ARG;
    if (d.dtype == DGL_DTYPE_MXFP4)
      st = validate_mxfp4(pr, static_cast<const uint8_t*>(d.scale_a), static_cast<const uint8_t*>(d.scale_b));
    else if (d.dtype == DGL_DTYPE_BF16 || d.dtype == DGL_DTYPE_E4M3 || d.dtype == DGL_DTYPE_W4A8)
      st = validate(pr);
    if (st != DGL_OK) return st;
  }
  // The first kernel waits for the work before the batch and only then lets
  // the next launch; the later ones read their operands at once and wait for
  // their predecessor before writing C.  A zero fill (K == 0) is an ordinary
  // launch, after all earlier work, so it too may head the chain.
  bool head = true;
  for (int32_t i = 0; i < count; ++i) {
    const dgl_gemm_desc& d = items[i];
    Problem pr = problem(d);
    const int64_t m = pr.m == 0 ? pr.M : pr.m, n = pr.n == 0 ? pr.N : pr.n;
    if (m == 0 || n == 0) continue;
    pr.pdl_mode = head ? PDL_BATCH_HEAD : PDL_BATCH_NEXT;
    const dgl_status st =
        d.dtype == DGL_DTYPE_MXFP4
            ? run_mxfp4(pr, static_cast<const uint8_t*>(d.scale_a), static_cast<const uint8_t*>(d.scale_b), s)
            : run(pr, nullptr, s);
    if (st != DGL_OK) return st;
    head = false;
  }
  return DGL_OK;
}

dgl_status dgl_gemm_planned(int32_t dtype, const void* A, const void* B, const float* sa, const float* sb, void* C,
                            int64_t M, int64_t N, int64_t K, int64_t m_valid, int64_t n_valid, int32_t out_dtype,
                            const dgl_plan_info* plan, void* stream) {
  if (!plan) return DGL_ERR_ARG;
  const bool w4 = dtype == DGL_DTYPE_W4A8;
  if (w4) dtype = DGL_DTYPE_E4M3;
  Problem pr{dtype, out_dtype, A, B, dtype == DGL_DTYPE_E4M3 ? sa : nullptr,
             dtype == DGL_DTYPE_E4M3 ? sb : nullptr, C, M, N, K, m_valid, n_valid};
  pr.w4 = w4 ? 1 : 0;
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
  if (dtype != DGL_DTYPE_BF16 && dtype != DGL_DTYPE_E4M3 && dtype != DGL_DTYPE_MXFP4 && dtype != DGL_DTYPE_W4A8)
    return DGL_ERR_ARG;
  if (dtype == DGL_DTYPE_W4A8) dtype = DGL_DTYPE_E4M3;  // the E4M3 tiles and decode path
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
    // A kernel that gave up may have left partial-tile flags set: clear every
    // flag of this device once its work has drained, so no later launch takes
    // a stale partial for a fresh one.
    if (cudaDeviceSynchronize() != cudaSuccess) return DGL_ERR_CUDA;
    {
      std::lock_guard<std::mutex> lock(g_mu);
      for (const Workspace& w : g_workspaces)
        if (w.dev == dev && w.flags && cudaMemset(w.flags, 0, sizeof(int) * w.nflags) != cudaSuccess)
          return DGL_ERR_CUDA;
    }
    {
      std::lock_guard<std::mutex> lock(g_noalloc_mu);
      if (g_noalloc[dev].ready && cudaMemset(g_noalloc[dev].flags, 0, sizeof(int) * g_noalloc[dev].nflags) != cudaSuccess)
        return DGL_ERR_CUDA;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) return DGL_ERR_CUDA;
    // a tile kernel that found its shared memory misaligned did nothing
    return (word & ~STATUS_SMEM_ALIGN) != 0 ? DGL_ERR_TIMEOUT : DGL_ERR_UNSUPPORTED;
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
  // the planner's path and tile; on the tcgen05 path a partial last wave is
  // split along K when stream-K applies to it
  dgl_plan_info plan;
  choose_plan(pr.dtype, pr.out, pr.m, pr.n, pr.K, ds->num_sms, &plan);
  // checked before the set-up, so a refused call enqueues nothing
  if (!noalloc_fits(pr, plan, ds->num_sms)) return DGL_ERR_SHAPE;
  StaticScratch* sc = nullptr;
  st = noalloc_setup(dev, &sc);
  if (st != DGL_OK) return st;
  plan.stream_k = plan.path == DGL_PATH_TC ? 1 : 0;
  plan.grid = 0;
  plan.tile_k = 0;
  return run(pr, &plan, static_cast<cudaStream_t>(stream), sc);
}

dgl_status dgl_shutdown(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DGL_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DGL_ERR_UNSUPPORTED;
  dgl_status st = DGL_OK;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    bool any = false;
    for (const Workspace& w : g_workspaces) any = any || w.dev == dev;
    // the device's queued kernels may still read a workspace
    if (any && cudaDeviceSynchronize() != cudaSuccess) st = DGL_ERR_CUDA;
    for (size_t i = g_workspaces.size(); i-- > 0;) {
      if (g_workspaces[i].dev != dev) continue;
      free_workspace(g_workspaces[i]);
      g_workspaces.erase(g_workspaces.begin() + static_cast<std::ptrdiff_t>(i));
    }
    for (auto it = g_plans.begin(); it != g_plans.end();) {
      if (it->first.dev == dev)
        it = g_plans.erase(it);
      else
        ++it;
    }
  }
  {
    // encoded tensor maps hold only addresses and extents; dropping them all
    // means none outlives the buffers it was made for
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (MapSlot& s : g_map_cache) s.valid = false;
  }
  return st;
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

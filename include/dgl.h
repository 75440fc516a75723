/*
 * dgl.h -- C ABI of the GB300 (sm_103a) dense linear-layer GEMM library.
 *
 * The operation.  Every compute entry point evaluates, for the valid region
 * 0 <= i < m_valid, 0 <= j < n_valid,
 *
 *     C[i, j] = sum_{k < K} A[i, k] * B[j, k]                   (bf16 inputs)
 *     C[i, j] = (sa[i] * sb[j]) applied to that sum              (E4M3 inputs)
 *
 * with fp32 accumulation.  This is a linear layer Y = X W^T flattened to one
 * GEMM: A = X_flat [M = B*L tokens, K = d_model], B = W [N = d_ff, K]
 * ("GEMM analysis in TraceLens", sections "Linear layers in LLMs",
 * "Flattening for GEMM" and "Linear layer: Y = X @ W^T", which is the BLAS
 * (T, N) call on row-major data).  The operand orientation C[M,N] = A[M,K] x
 * B[N,K]^T, and the epilogue value = acc * scale_a * scale_b, follow the
 * "Gemm Optimization" guide (sections 1.1 "Three-Level Tiling" and 7.1
 * "Direct Store").  m_valid / n_valid are the real extents behind a tiled
 * problem, as in FlyDSL pull request 1303 (RDNA3 WMMA GEMM): the caller sizes
 * the problem in whole tiles and these two arguments say how many rows and
 * columns of the last tile hold data; passing 0 selects the full extent, the
 * old behaviour.
 *
 * Layout (all row-major, last dimension contiguous -- flattening is free only
 * when it is, "GEMM analysis in TraceLens", section "Edge cases"):
 *   A  at least m_valid rows of K elements, row pitch K elements.
 *   B  at least n_valid rows of K elements, row pitch K elements.
 *   C  M rows, row pitch N elements (so N is C's leading dimension).  Only
 *      the valid region [0, m_valid) x [0, n_valid) is written; every other
 *      element of C is left untouched.
 *   sa m_valid fp32 scales (row i of A), sb n_valid fp32 scales (row j of B).
 * Element types: bf16 (A, B), OCP E4M3 "e4m3fn" (A, B of dgl_gemm_fp8),
 * fp32 scales; C is bf16 (rounded to nearest even) or fp32 by `out_dtype`.
 *
 * Memory and ownership: A, B, C, sa, sb are DEVICE pointers owned by the
 * caller, on the current CUDA device.  The library never copies to or from the
 * host.  It keeps a small per-device plan cache, a cache of encoded tensor
 * maps and, for plans with stream_k = 1, a per-(device, stream) workspace of
 * fp32 partial tiles (at least 24 MB), allocated with cudaMalloc on the first
 * such call on that stream.  At most four such workspaces are kept per
 * device: a call on a fifth stream first waits for the device to drain, then
 * frees the least recently used one.  dgl_shutdown() frees them all.  A call
 * made while its stream is being captured into a CUDA graph never allocates:
 * if the stream has no workspace yet it runs the data-parallel schedule
 * instead (make one call on that stream before capturing to keep the split
 * schedule).  Every launch leaves the workspace's flags cleared, so a
 * captured graph may be replayed.  Other calls that allocate or free a
 * workspace must not be made while another stream of the device is being
 * captured.  Calls are asynchronous
 * with respect to the host: work is enqueued on `stream` (a cudaStream_t;
 * NULL = the legacy default stream) and buffers must stay valid until it
 * completes.
 *
 * Errors: arguments are validated on the host before any launch; a failed
 * check returns an error code and enqueues nothing.  Nothing is printed and
 * nothing is thrown.  Kernel waits are bounded: a wait that times out sets a
 * per-device status word that dgl_device_status() reports.  There is no CPU
 * fallback; a device that is not sm_103 returns DGL_ERR_UNSUPPORTED.
 */
#ifndef DGL_H_
#define DGL_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DGL_OK = 0,
  DGL_ERR_ARG = -1,         /* null pointer, bad enum, negative extent, m_valid > M, n_valid > N */
  DGL_ERR_ALIGN = -2,       /* A/B/scales not 16/4-byte aligned, K not a multiple of 16 bytes */
  DGL_ERR_SHAPE = -3,       /* an extent beyond 2^31 - 1 */
  DGL_ERR_UNSUPPORTED = -4, /* device is not sm_103, or a forced plan the library cannot run */
  DGL_ERR_CUDA = -5,        /* a CUDA runtime/driver call failed */
  DGL_ERR_TIMEOUT = -6      /* a kernel's bounded wait gave up (see dgl_device_status) */
} dgl_status;

typedef enum { DGL_OUT_BF16 = 0, DGL_OUT_F32 = 1 } dgl_out_t;
typedef enum { DGL_DTYPE_BF16 = 0, DGL_DTYPE_E4M3 = 1, DGL_DTYPE_MXFP4 = 2, DGL_DTYPE_W4A8 = 3 } dgl_dtype_t;
typedef enum { DGL_PATH_TC = 0, DGL_PATH_DECODE = 1, DGL_PATH_EMPTY = 2 } dgl_path_t;
/* Activations of dgl_linear: GELU(x) = x * Phi(x) (Phi the standard normal
 * distribution function, the exact erf form); SiLU(x) = x * sigma(x) (sigma
 * the logistic function). */
typedef enum { DGL_ACT_NONE = 0, DGL_ACT_GELU = 1, DGL_ACT_SILU = 2 } dgl_act_t;
/* Operand storage of dgl_gemm_bf16_ex: K-major rows hold K contiguous
 * elements (A [m][K], B [n][K]); MN-major rows hold M (or N) contiguous
 * elements (A [K][m], B [K][n]). */
typedef enum { DGL_K_MAJOR = 0, DGL_MN_MAJOR = 1 } dgl_major_t;

/*
 * A launch plan: the path, the tile of the tile ladder, and the cost-model
 * quantities behind the choice.  tile_eff, wq_eff and dim_eff are the tile-
 * and wave-quantisation efficiencies of "GEMM analysis in TraceLens"
 * (section "GEMM dimension efficiency": tile_eff = M N / (M_pad N_pad),
 * wq_eff = tiles / (ceil(tiles / units) units), dim_eff = their product).
 */
typedef struct {
  int32_t path;       /* dgl_path_t */
  int32_t tile_m;     /* rows of C per tile (tcgen05 path: 64, 128, or 256 for a CTA pair) */
  int32_t tile_n;     /* columns of C per tile (tcgen05 path: 64, 128 or 256; 224 on a CTA pair) */
  int32_t tile_k;     /* K elements per pipeline stage (64 bf16, 128 E4M3) */
  int32_t stages;     /* shared-memory ring depth */
  int32_t cta_group;  /* CTAs sharing one MMA: 1, or 2 (a CTA pair, tile_m 256) */
  int32_t grid;       /* CTAs launched (persistent: at most one per SM) */
  int32_t num_tiles;  /* output tiles (tcgen05 path) or parts of B's rows (decode path) */
  double tile_eff;
  double wq_eff;
  double dim_eff;
  double est_us;      /* cost-model estimate of the kernel time, microseconds */
  int32_t stream_k;   /* 1: tiles of the last, partial wave are split along K across all workers; */
                      /* S >= 2: each such tile's k-stages in S equal ranges on S workers (a split-K tail, */
                      /*    the planner's choice for long K when that wave fills at most half the workers) */
  int32_t split_tail; /* 1: the last, partial wave's tiles (tile_n 256) run as two half tiles each, */
                      /*    when that wave fills at most half the workers (not with stream_k or gated); */
                      /*    the planner sets it only for K of at most 16 k-blocks of 128 bytes */
  int32_t k_group;    /* decode path: 128-byte K steps stacked into one 128-row MMA operand (1, 2, 4, */
                      /*    8 or 16: parts of at most 128 / k_group rows); 1 on the tcgen05 tile path */
} dgl_plan_info;

/*
 * bf16 GEMM.  A [m_valid, K] bf16, B [n_valid, K] bf16, C [M, ldc = N].
 * M, N: C's rows and row pitch (elements); m_valid <= M, n_valid <= N, 0 = full.
 * K: inner extent; K * 2 bytes must be a multiple of 16 (K % 8 == 0).
 * A, B 16-byte aligned; C aligned to its element size.
 * out_dtype: DGL_OUT_BF16 or DGL_OUT_F32.  stream: cudaStream_t.
 * M == 0 or N == 0 is an empty product (DGL_OK, nothing enqueued); K == 0
 * writes zeros to the valid region (the empty sum).
 */
dgl_status dgl_gemm_bf16(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                         int64_t m_valid, int64_t n_valid, int32_t out_dtype, void* stream);

/*
 * E4M3 GEMM with per-row scales sa on A and per-column scales sb on B
 * (fp32, 4-byte aligned, m_valid and n_valid entries):
 *   C[i, j] = (acc * sa[i]) * sb[j], acc = fp32 sum of A[i, k] * B[j, k].
 * K must be a multiple of 16.  Otherwise as dgl_gemm_bf16.
 */
dgl_status dgl_gemm_fp8(const void* A, const void* B, const float* sa, const float* sb, void* C, int64_t M,
                        int64_t N, int64_t K, int64_t m_valid, int64_t n_valid, int32_t out_dtype, void* stream);

/*
 * Either GEMM with a caller-chosen plan instead of the planner's choice: the
 * forced-tile sweep of FlyDSL pull request 1303, whose tests run each tile of
 * both ladders on a shape that no tile divides.
 * dtype: dgl_dtype_t: bf16 (sa/sb ignored), E4M3 or W4A8 (the operands of
 * dgl_gemm_w4a8).  plan->path, tile_m, tile_n,
 * stream_k, split_tail and grid are honoured (grid <= 0 picks one), and for the decode
 * path tile_k (K elements per ring stage: a multiple of 128 bytes and of
 * k_group such steps, 0 = pick);
 * other fields are ignored.  A plan the library has no kernel for returns
 * DGL_ERR_UNSUPPORTED.
 */
dgl_status dgl_gemm_planned(int32_t dtype, const void* A, const void* B, const float* sa, const float* sb,
                            void* C, int64_t M, int64_t N, int64_t K, int64_t m_valid, int64_t n_valid,
                            int32_t out_dtype, const dgl_plan_info* plan, void* stream);

/*
 * Block-scaled FP4 GEMM (MXFP4).  The "Gemm Optimization" guide's bandwidth
 * formulas (section 8.2, "FP4 (MXFP4)") count half a byte per element of A
 * and of B and one scale byte per 32 elements of K for every row of each;
 * the format read into that name is OCP Microscaling MXFP4: E2M1 elements and
 * one E8M0 scale (2^(e - 127); 0xFF is NaN) per block of 32 consecutive
 * elements of a row along K.
 *   C[i, j] = sum_k 2^(sfa[i][k/32] - 127) a(i, k) * 2^(sfb[j][k/32] - 127) b(j, k)
 * accumulated in fp32 on the tensor cores (tcgen05 kind::mxf4), then
 * rounded to bf16 (nearest even) or kept in fp32.
 * A: m_valid rows of K / 2 bytes, B: n_valid rows of K / 2 bytes; element 2t
 * of a row in the low four bits of byte t.  sfa: m_valid rows of K / 32
 * bytes, sfb: n_valid rows of K / 32 bytes (unaligned is fine).
 * C, M, N, m_valid, n_valid, out_dtype and the never-written region outside
 * [0, m_valid) x [0, n_valid) as dgl_gemm_bf16.  K: a multiple of 32 (whole
 * blocks; the K / 2-byte rows are then whole 16-byte units).  A, B 16-byte
 * aligned.  Errors: DGL_ERR_ARG (null pointers, extents), DGL_ERR_ALIGN
 * (K not a multiple of 32, A or B not 16-byte aligned, C not aligned to
 * its element), DGL_ERR_SHAPE (extents past int32).  Every problem, small
 * m included, runs on 128 x 256 tiles (the decode path is bf16 / E4M3 only).
 * Results whose block-scale products leave fp32's range are not specified;
 * the parity tests keep scales within 2^-20 .. 2^20.
 */
dgl_status dgl_gemm_mxfp4(const void* A, const void* B, const uint8_t* sfa, const uint8_t* sfb, void* C, int64_t M,
                          int64_t N, int64_t K, int64_t m_valid, int64_t n_valid, int32_t out_dtype, void* stream);

/*
 * 8-bit activations times 4-bit weights (W4A8).  The "Gemm Optimization"
 * guide's bandwidth formulas (section 8.2) count, for 4-bit weights, one byte
 * per element of A, half a byte per element of B, a bf16 C and (M + N) fp32
 * scales.  Read on GB300, whose tensor cores take E4M3 and E2M1 operands in
 * one kind::f8f6f4 instruction: A holds E4M3 codes with a per-row scale sa,
 * B holds E2M1 codes (values 0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6) two
 * to a byte, element 2t in the low four bits of byte t, with a per-row scale
 * sb (one per column of C):
 *   C[i, j] = (acc * sa[i]) * sb[j],  acc = fp32 sum of e4m3(A[i, k]) e2m1(B[j, k])
 * A: m_valid rows of K bytes (16-byte aligned).  B: n_valid rows of K / 2
 * bytes (32-byte aligned).  K: a multiple of 128.  sa, sb, C, M, N, m_valid,
 * n_valid, out_dtype and the never-written region as dgl_gemm_fp8, whose
 * tiles and decode path (m_valid <= 16) it shares.  Errors: DGL_ERR_ALIGN for
 * K not a multiple of 128 or B not 32-byte aligned; otherwise as dgl_gemm_fp8.
 */
dgl_status dgl_gemm_w4a8(const void* A, const void* B, const float* sa, const float* sb, void* C, int64_t M,
                         int64_t N, int64_t K, int64_t m_valid, int64_t n_valid, int32_t out_dtype, void* stream);

/*
 * Size in bytes of the fixed device array that dgl_gemm_noalloc uses for its
 * fp32 partial tiles: 20 MiB, one 128 x 256 fp32 tile for each of 160 CTAs.
 */
#define DGL_NOALLOC_SCRATCH_BYTES (20u * 1024u * 1024u)

/*
 * GEMM that allocates no device memory.  No page behind this library
 * describes it: it exists for callers that cannot call cudaMalloc while they
 * run, such as a framework that hands every byte of device memory out from
 * its own pool (an allocation outside the pool fails or breaks the pool's
 * accounting) or a serving loop that forbids allocation after start-up
 * (cudaMalloc may block on the whole device).
 *
 * It computes what dgl_gemm_bf16 (dtype = DGL_DTYPE_BF16; sa and sb ignored)
 * or dgl_gemm_fp8 (dtype = DGL_DTYPE_E4M3) compute, with the same arguments,
 * layouts, validation and error codes.  On the tcgen05 path, when the last
 * wave of tiles is partial and each worker (CTA or CTA pair) gets at least
 * four 128-byte k-stages of it, those tiles are split along K across all
 * workers (stream-K); the partial tiles go through a static device array of
 * DGL_NOALLOC_SCRATCH_BYTES plus 160 flags that the library holds on every
 * device that loads it, until the process exits.  A problem whose split would
 * need more partial tiles than the array holds (more than
 * DGL_NOALLOC_SCRATCH_BYTES, or more than 160 CTAs: possible only on a device
 * with more than 160 SMs) returns DGL_ERR_SHAPE and enqueues nothing.  Other
 * partial-wave shapes (a short tail), problems without a partial last wave,
 * and those on the decode path (m_valid <= 16) run as dgl_gemm_bf16 /
 * dgl_gemm_fp8 would and do not touch the array.
 *
 * Device memory: the array belongs to the library's CUDA module, whose memory
 * the driver commits when the module is loaded: by the first dgl_* call that
 * touches a device (modules load lazily by default), or when the library is
 * loaded if CUDA_MODULE_LOADING=EAGER.  A caller whose own pool reserves the
 * device's memory must make one dgl_* call on each device before the pool
 * takes it.
 *
 * Set-up: the first call on a device (the current device) looks the array's
 * address up and clears its flags, synchronously; make that first call
 * before any stream capture.  Later calls only enqueue work.
 * The array is shared by every call on a device and keeps what the last call
 * left in it: partial tiles (never read before they are rewritten) and its
 * flags, which every call leaves cleared.  Calls whose kernels overlap on the GPU,
 * for example on two streams, race on it: order them, or use dgl_gemm_bf16 /
 * dgl_gemm_fp8.
 */
dgl_status dgl_gemm_noalloc(int32_t dtype, const void* A, const void* B, const float* sa, const float* sb,
                            void* C, int64_t M, int64_t N, int64_t K, int64_t m_valid, int64_t n_valid,
                            int32_t out_dtype, void* stream);

/*
 * One GEMM of a batch (dgl_gemm_batch).  The fields are the arguments of
 * dgl_gemm_bf16 / dgl_gemm_fp8 / dgl_gemm_w4a8 / dgl_gemm_mxfp4, chosen by
 * dtype (DGL_DTYPE_BF16, _E4M3, _W4A8 or _MXFP4):
 *   scale_a, scale_b: E4M3 and W4A8: the fp32 per-row scales sa (m_valid
 *     entries) and sb (n_valid entries); MXFP4: the E8M0 scale bytes sfa
 *     [m_valid][K / 32] and sfb [n_valid][K / 32]; bf16: unused (NULL).
 * Layouts, alignment rules and the meaning of M, N, m_valid and n_valid are
 * those of the matching single call.
 */
typedef struct dgl_gemm_desc {
  int32_t dtype;
  int32_t out_dtype;
  const void* A;
  const void* B;
  const void* scale_a;
  const void* scale_b;
  void* C;
  int64_t M, N, K, m_valid, n_valid;
} dgl_gemm_desc;

/*
 * A batch of GEMMs, enqueued in order on one stream: what `count` single
 * calls would compute, with the kernels overlapped further.  Each kernel after
 * the first reads its operands while its predecessor is still running
 * (programmatic dependent launch) and waits for the predecessor only before
 * it writes C.  This is the running of independent GEMMs back to back (a
 * ragged-shape sweep, the projections of a layer that share no output), where
 * one kernel's operand loads then hide the previous kernel's last tiles.
 *
 * Contract: no item's A, B or scales may overlap the C of an earlier item of
 * the same batch (an item may not consume an earlier item's result).  Items may
 * share inputs, and may write the same C (the later one wins).  Work enqueued
 * on the stream before the batch is complete before any item reads its
 * operands; work enqueued after the batch sees every item's C, as after single
 * calls.
 *
 * items: host array of `count` descriptors, read during the call only.
 * Every item is checked before any is enqueued: an invalid one returns its
 * status (DGL_ERR_ARG, _ALIGN, _SHAPE) and nothing is enqueued.  An error while
 * enqueueing item i (DGL_ERR_CUDA, DGL_ERR_UNSUPPORTED) returns that status,
 * with items 0 .. i - 1 enqueued.  count == 0 is DGL_OK.  Empty items
 * (m_valid or n_valid resolving to 0) enqueue nothing; K == 0 items write zeros.
 */
dgl_status dgl_gemm_batch(const dgl_gemm_desc* items, int32_t count, void* stream);

/*
 * bf16 GEMM with either operand stored K-major or MN-major and explicit row
 * pitches: the three GEMMs of a linear layer's training step ("GEMM analysis
 * in TraceLens", sections "Backward pass GEMMs" and "How PyTorch calls BLAS"):
 *   forward  Y  = X W^T   A = X  [m][K]   K-major,  B = W [n][K]  K-major
 *   backward dX = dY W    A = dY [m][K]   K-major,  B = W [K][n]  MN-major
 *   backward dW = dY^T X  A = dY [K][m]   MN-major, B = X [K][n]  MN-major
 * C[i, j] = sum_k A(i, k) B(j, k) for i < m, j < n, fp32 accumulation; C is
 * [m][ldc] (ldc >= n, 0 = n).  lda / ldb: row pitches in elements (0 = the
 * packed pitch: K for K-major, m or n for MN-major); each a multiple of 8
 * (16 bytes) and at least the row's extent.  A, B 16-byte aligned.  Returns
 * DGL_ERR_ALIGN for a pitch that breaks the 16-byte rule.  plan: NULL or as
 * dgl_gemm_planned (tcgen05 path only; MN-major operands never take the
 * decode path).  Otherwise as dgl_gemm_bf16.
 */
dgl_status dgl_gemm_bf16_ex(int32_t a_major, int32_t b_major, const void* A, int64_t lda, const void* B, int64_t ldb,
                           void* C, int64_t ldc, int64_t m, int64_t n, int64_t K, int32_t out_dtype,
                           const dgl_plan_info* plan, void* stream);

/*
 * A linear layer: the GEMM above with its epilogue fused into the kernel
 * (Funlib GEMM issue, section "Investigate later optimizations": fused bias
 * and activation to cut intermediate memory traffic).  The forward operation
 * is Y = X W^T + b with b of length d_ff ("GEMM analysis in TraceLens",
 * section "Backward pass GEMMs"; the trace's aten::addmm), followed in a
 * feed-forward block by an activation (Funlib GEMM issue, "Description":
 * XW1 -> GELU -> XW2).  The LLaMA MLP's up and gate projections of one input
 * ("GEMM analysis in TraceLens", "Real-world example: LLaMA-2 7B") fuse into
 * one call with gated = 1.
 *   gated = 0:  C[i, j] = act(acc(i, j) + bias[j])
 *   gated = 1:  C[i, j] = act(acc(i, j) + bias[j]) * (acc(i, n + j) + bias[n + j])
 * where acc(i, r) is sum_k A[i, k] * B[r, k] (times sa[i] * sb[r] for E4M3)
 * in fp32, and n = n_valid.  A gated layer's B holds 2 n rows: the gate
 * projection's n rows, then the up projection's n rows; sb and bias then hold
 * 2 n entries in the same order.  bias (fp32, 4-byte aligned) may be NULL.
 * act: dgl_act_t.  plan: NULL for the library's choice, else as
 * dgl_gemm_planned (a gated layer needs tile_m 256; tile_n 128 or 256).
 * Layout, scales, validation and errors otherwise as dgl_gemm_bf16 /
 * dgl_gemm_fp8.  Problems with m_valid <= 16 take the decode path unless
 * gated; gated layers always run on CTA-pair tiles.
 */
dgl_status dgl_linear(int32_t dtype, const void* A, const void* B, const float* sa, const float* sb,
                      const float* bias, void* C, int64_t M, int64_t N, int64_t K, int64_t m_valid, int64_t n_valid,
                      int32_t out_dtype, int32_t act, int32_t gated, const dgl_plan_info* plan, void* stream);

/*
 * The plan the library would use for a problem of m x n x K (valid extents)
 * on a device with num_sms SMs (num_sms <= 0: query the current device).
 * Pure host logic when num_sms > 0: needs no GPU.
 * Rule: m <= 16 takes the decode path; otherwise the tcgen05 tile ladder is
 * screened by padded output area (rejecting a tile whose padded area exceeds
 * 1.25x the real one unless none passes, as in FlyDSL pull request 1303's
 * autotuner) and the survivor with the lowest cost-model time is chosen.
 * dtype DGL_DTYPE_MXFP4 has one tile: 128 x 256 (tile_k 256 elements).
 * dtype DGL_DTYPE_W4A8 is planned as DGL_DTYPE_E4M3 (the same tiles).
 */
dgl_status dgl_plan(int32_t dtype, int64_t m, int64_t n, int64_t K, int32_t out_dtype, int32_t num_sms,
                    dgl_plan_info* out);

/*
 * The plan dgl_linear would use (gated: a layer whose B holds 2 n rows).
 * Pure host logic when num_sms > 0.
 */
dgl_status dgl_plan_linear(int32_t dtype, int64_t m, int64_t n, int64_t K, int32_t out_dtype, int32_t gated,
                           int32_t num_sms, dgl_plan_info* out);

/*
 * Tile- and wave-quantisation metrics of an m x n output on tile_m x tile_n
 * tiles spread over num_units parallel units ("GEMM analysis in TraceLens",
 * section "How it's calculated").  Fills num_tiles, tile_eff, wq_eff and
 * dim_eff of *out (other fields zero).  Pure host logic.
 */
dgl_status dgl_tile_metrics(int64_t m, int64_t n, int32_t tile_m, int32_t tile_n, int32_t num_units,
                            dgl_plan_info* out);

/*
 * Release what the library holds on the current device: wait for the device's
 * queued work, free every stream-K workspace, and drop the cached plans and
 * tensor maps.  The caller owns every other buffer (the Funlib GEMM issue,
 * "Support device-resident tensors": each allocation has an owner that frees
 * it); this gives the library's own allocation an explicit end.  Later calls
 * rebuild what they need.  The static array of dgl_gemm_noalloc is not
 * freed (it lives as long as the library is loaded).  Must not race with
 * other threads' calls on this device, nor run while a stream of the device
 * is being captured.  Returns DGL_ERR_CUDA if the synchronisation reported an
 * error (the state is released anyway), else DGL_OK.
 */
dgl_status dgl_shutdown(void);

/*
 * Synchronise `stream`, then report and clear the current device's status
 * word: DGL_ERR_TIMEOUT if any kernel's bounded wait gave up since the last
 * call (the device is then drained and every partial-tile flag of the
 * library on it cleared), DGL_ERR_UNSUPPORTED if a tile kernel found its
 * dynamic shared memory without the 1024-byte alignment it declares and
 * exited without work (not seen on GB300), DGL_ERR_CUDA if synchronisation
 * failed, else DGL_OK.
 */
dgl_status dgl_device_status(void* stream);

/* Static description of a status code (never NULL). */
const char* dgl_status_string(int32_t status);

/* Library ABI version (major * 100 + minor). */
int32_t dgl_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DGL_H_ */

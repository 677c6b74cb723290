/*
 * qmuon -- quantized Muon optimizer step for one NVIDIA GB300 (sm_103a).
 *
 * C ABI.  Every pointer argument is either a host pointer (H) or a device
 * pointer (D), as marked.  All device memory is owned by the caller except
 * the small metadata tables a qmuon_plan owns.  Every entry that takes a
 * `stream` (a cudaStream_t passed as void*, NULL = legacy default stream)
 * only enqueues work on it and returns; results are ready when the stream
 * reaches that point.  Every entry validates its arguments on the host first
 * and launches nothing when validation fails; no entry aborts or throws
 * (a failed host allocation returns QMUON_ERR_OUT_OF_MEMORY).
 *
 * Layouts: tensors are dense, row-major and contiguous.  q8 codes and
 * gradients must start on a 16-byte boundary; absmax on a 4-byte boundary.
 * A tensor has rows*cols elements, split into 256-element quantization
 * blocks in flat order; the last block may be partial.
 *
 * Concurrency: calls that share a workspace must not overlap on the GPU
 * (enqueue them on one stream).  The steps of one plan (qmuon_step,
 * qmuon_step_from_host, qmuon_step_prepare) share the plan's Newton-Schulz
 * tables: make them from one host thread at a time and enqueue them on one
 * stream.  Distinct plans/workspaces are independent.
 */
#ifndef QMUON_H_
#define QMUON_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define QMUON_API __attribute__((visibility("default")))
#else
#define QMUON_API
#endif

#define QMUON_BLOCK 256          /* elements per quantization block          */
#define QMUON_SCALE_BLOCK 32     /* elements per MXFP8 carrier scale (a row) */

typedef enum {
  QMUON_OK = 0,
  QMUON_ERR_INVALID_ARGUMENT = 1,   /* NULL/misaligned pointer, bad size or enum */
  QMUON_ERR_MISALIGNED_SEGMENT = 2, /* norm segment not on 256-element blocks   */
  QMUON_ERR_UNSUPPORTED = 3,        /* valid request the library does not serve  */
  QMUON_ERR_WORKSPACE_TOO_SMALL = 4,
  QMUON_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed         */
  QMUON_ERR_TIMEOUT = 6,            /* a kernel's bounded wait expired (see qmuon_sync_status) */
  QMUON_ERR_OUT_OF_MEMORY = 7       /* host memory for a plan's or a call's tables could not be allocated */
} qmuon_status;

typedef enum { QMUON_Q8_INT8 = 0, QMUON_Q8_UINT8 = 1 } qmuon_q8_kind;
typedef enum { QMUON_BF16 = 0, QMUON_FP16 = 1, QMUON_FP32 = 2 } qmuon_dtype;

/* One optimizer tensor (a matrix of momentum state).
 *   q8     D  rows*cols codes: int8 q, or uint8 q+128 (offset binary)
 *   absmax D  ceil(rows*cols/256) fp32 block maxima
 *   grad   D  rows*cols gradient elements of the plan's dtype; IN: gradient,
 *             OUT: the new momentum m (update entries) or the orthogonalised
 *             update U (qmuon_step)
 * State format: "Quantized Muon Momentum", section "What Exists". */
typedef struct {
  void* q8;
  float* absmax;
  void* grad;
  int64_t rows;
  int64_t cols;
} qmuon_tensor;

/* A run of one tensor's flat elements that belongs to a norm group
 * ("Quantized Muon Momentum", section "Grouped QKV And Sharding").
 * `start` must be a multiple of 256 and `start + length` a multiple of 256
 * or the tensor's element count; otherwise QMUON_ERR_MISALIGNED_SEGMENT.
 * Group ids are dense in [0, n_groups).  A block may belong to at most one
 * segment; blocks in no segment are updated but not summed. */
typedef struct {
  int32_t tensor_index;
  int32_t group_id;
  int64_t start;
  int64_t length;
} qmuon_norm_segment;

typedef struct qmuon_plan qmuon_plan;

/* Build a reusable plan over `n_tensors` tensors (H array, copied).
 *   segments/n_segments  H  norm groups for qmuon_update_multi_normalize_groups;
 *                           NULL/0 = one group per tensor (n_groups must then
 *                           equal n_tensors, or be 0 to mean that)
 *   tile_r, tile_c          MuonBP block tiling used by qmuon_step's block
 *                           steps: every tensor is cut into tile_r x tile_c
 *                           tiles of (rows/tile_r) x (cols/tile_c), so rows
 *                           and cols must divide (else
 *                           QMUON_ERR_INVALID_ARGUMENT); tiles must be whole
 *                           256-element blocks (else
 *                           QMUON_ERR_MISALIGNED_SEGMENT): with tile_c > 1,
 *                           cols and the tile width are multiples of 256;
 *                           with tile_c == 1 and tile_r > 1, each tile's
 *                           element count is a multiple of 256
 *   out                  H  receives the plan (freed by qmuon_plan_destroy)
 * Tensors may be empty (rows or cols 0; their pointers are not used), but the
 * plan must hold between 1 and 2^31 - 1 quantization blocks in all
 * (QMUON_ERR_INVALID_ARGUMENT otherwise).  The plan uploads its tables once
 * (one H2D copy) to the current device and is tied to that device.
 * Allocates device memory (small tables) only. */
QMUON_API qmuon_status qmuon_plan_create(const qmuon_tensor* tensors, int32_t n_tensors,
                               qmuon_q8_kind q8_kind, qmuon_dtype grad_dtype,
                               const qmuon_norm_segment* segments, int32_t n_segments,
                               int32_t n_groups, int32_t tile_r, int32_t tile_c,
                               qmuon_plan** out);
QMUON_API void qmuon_plan_destroy(qmuon_plan* plan);

/* Counts a caller needs to size outputs: the plan's segment groups, the
 * full-step groups (one per tensor) and block-step groups (tiles). */
QMUON_API qmuon_status qmuon_plan_info(const qmuon_plan* plan, int64_t* n_blocks, int32_t* n_groups,
                             int32_t* n_full_groups, int32_t* n_block_groups);

/* Which entry a workspace is sized for. */
typedef enum { QMUON_WS_UPDATE = 0, QMUON_WS_STEP = 1 } qmuon_ws_kind;

/* Bytes of device workspace the entry needs (0 on a NULL plan or an unknown
 * kind).  The workspace is scratch: its contents between calls are
 * unspecified, except that it must not be shared by calls in flight at the
 * same time. */
QMUON_API size_t qmuon_workspace_size(const qmuon_plan* plan, qmuon_ws_kind which);

/* The blockwise 8-bit momentum update over every tensor of the plan in one
 * launch ("Quantized Muon Momentum", section "Algorithm", steps 1-9):
 * dequantize, m = beta*old + (1-beta)*grad in fp32, m written over grad,
 * new absmax, symmetric nearest requantization to [-127, 127], and the
 * per-group sum of m*m reduced across the grid in the same launch.
 *   normalize_mode  0: no normalisation (sums/inverse norms still written to
 *                      the non-NULL outputs)
 *                   1: in place -- every grouped block of grad is then
 *                      scaled by its group's inverse norm (second pass)
 *                   2: deferred -- inverse norms only, for a later
 *                      qmuon_newton_schulz_batched (group_inv_norm required)
 *   group_sumsq     D  [n_groups] fp32 sum of m*m per group, or NULL
 *   group_inv_norm  D  [n_groups] fp32 1/(sqrt(sum)+1e-7), or NULL
 *   ws, ws_bytes    D  workspace of qmuon_workspace_size(plan, QMUON_WS_UPDATE)
 * The arithmetic is exactly the fp32 operation order above, one rounding per
 * operation (no FMA contraction), so q8 codes and absmax are reproducible
 * bit for bit; sums are accumulated in fp64 across blocks.  Non-finite
 * momenta: NaN lanes are ignored by the absmax (a block of NaN only gets 0),
 * a NaN product quantises to code 0, and an infinity makes its block's absmax
 * infinite and every code of that block 0. */
QMUON_API qmuon_status qmuon_update_multi_normalize_groups(const qmuon_plan* plan, float beta,
                                                 int32_t normalize_mode, float* group_sumsq,
                                                 float* group_inv_norm, void* ws,
                                                 size_t ws_bytes, void* stream);

/* qmuon_update_multi_normalize_groups with stochastic requantisation (the
 * page, section "Known Limitations", lists stochastic rounding as not yet
 * implemented; this is the reading taken): with x = fl(m * (127/absmax)),
 *   q = clamp(floor(x + u), -127, 127)   (a NaN product gives 0)
 * where u = (w >> 8) * 2^-24 and w is word (e mod 4) of Philox4x32-10
 * (Salmon et al., SC'11; 10 rounds) with
 *   key     = (seed mod 2^32, seed >> 32)
 *   counter = (e/4 mod 2^32, e/2^34, tensor index in the plan, step mod 2^32)
 * for element e (flat index) of the tensor.  E[q] = x up to 2^-24, so the
 * dequantised state is unbiased.  Everything else, arguments and errors
 * included, is as in qmuon_update_multi_normalize_groups. */
QMUON_API qmuon_status qmuon_update_multi_normalize_groups_sr(const qmuon_plan* plan, float beta,
                                                    int32_t normalize_mode, uint64_t seed, int64_t step,
                                                    float* group_sumsq, float* group_inv_norm, void* ws,
                                                    size_t ws_bytes, void* stream);

/* Count non-finite momenta: every update launch through this plan (the
 * update entries, the carrier over the plan, qmuon_step and
 * qmuon_step_from_host) adds to *counter, with an atomic add, the number of
 * 256-element blocks whose fp32 sum of m*m is not finite (a NaN or an
 * infinity in m, or squares that overflow fp32).  Such a block's codes
 * follow the rules of qmuon_update_multi_normalize_groups but no longer
 * represent its momentum, and its group's norm is not meaningful.
 * The caller zeroes and reads the counter.
 *   counter  D  one uint32, 4-byte aligned, or NULL to stop counting
 * Host-only: changes no device state.  QMUON_ERR_INVALID_ARGUMENT on a NULL
 * plan or a misaligned counter. */
QMUON_API qmuon_status qmuon_plan_set_nonfinite_counter(qmuon_plan* plan, uint32_t* counter);

/* Make qmuon_step requantise stochastically (enable = 1; 0 restores nearest
 * rounding), as qmuon_update_multi_normalize_groups_sr does with this seed
 * and step = the step's t.  Host-only: changes no device state.
 * QMUON_ERR_INVALID_ARGUMENT on a NULL plan or enable not 0/1. */
QMUON_API qmuon_status qmuon_plan_set_stochastic_rounding(qmuon_plan* plan, int32_t enable, uint64_t seed);

/* How qmuon_step_from_host moves host gradients into the plan's buffers:
 *   QMUON_INGEST_PULL (the default): gradients in page-locked host memory
 *     that the device can address, 16-byte aligned, are read by a small
 *     kernel's own loads over the host link (about 19 CTAs on 152 SMs); any
 *     other gradient is copied with cudaMemcpyAsync;
 *   QMUON_INGEST_COPY: every gradient is copied with cudaMemcpyAsync.
 * Both move about 211 GB/s on GB300.  Copy-engine transfers were seen to
 * stall for 70-120 ms every ~510 ms on some hosts, which the pull does not;
 * the pull's host reads, in turn, slow Newton-Schulz kernels running beside
 * them (a MuonBP block step by about 2.8 ms while it runs).  Host-only:
 * changes no device state.  QMUON_ERR_INVALID_ARGUMENT on a NULL plan or an
 * unknown mode.  The pages have no counterpart. */
#define QMUON_INGEST_PULL 0
#define QMUON_INGEST_COPY 1
QMUON_API qmuon_status qmuon_plan_set_host_ingest(qmuon_plan* plan, int32_t mode);

/* Workspace bytes of qmuon_update_mxfp8_carrier for a rows x cols tensor. */
QMUON_API size_t qmuon_carrier_workspace_size(int64_t rows, int64_t cols);

/* q8 state + grad -> q8 state + normalised rowwise MXFP8 carrier
 * ("Quantized Muon Momentum", section "Wave18B MXFP8 Carrier Probe").
 *   tensor     H  one tensor (q8/absmax D, updated in place; grad D, READ ONLY)
 *   payload    D  rows x cols uint8 E4M3 codes of m / 2^(scale-127)
 *   scale_inv  D  rows x (cols/32) uint8 E8M0 exponents: the smallest power
 *                 of two with amax/2^(e-127) <= 448 per 32 row elements
 *   inv_norm   D  one fp32, 1/(sqrt(sum m*m)+1e-7)
 * cols must be a multiple of 32 (else QMUON_ERR_UNSUPPORTED). */
QMUON_API qmuon_status qmuon_update_mxfp8_carrier(const qmuon_tensor* tensor, qmuon_q8_kind q8_kind,
                                        qmuon_dtype grad_dtype, float beta, uint8_t* payload,
                                        uint8_t* scale_inv, float* inv_norm, void* ws,
                                        size_t ws_bytes, void* stream);

/* The carrier of every tensor of a plan in one launch (one norm group per
 * tensor, as in qmuon_step's full steps):
 *   payloads    H  n_tensors device pointers (D): tensor i's rows x cols E4M3
 *                  codes (16-byte aligned)
 *   scale_invs  H  n_tensors device pointers (D): tensor i's rows x (cols/32)
 *                  E8M0 exponents
 *   inv_norms   D  n_tensors fp32: 1/(sqrt(sum m*m)+1e-7) per tensor
 *   group_sumsq D  n_tensors fp32 sums of m*m, or NULL
 *   ws, ws_bytes D workspace of qmuon_workspace_size(plan, QMUON_WS_UPDATE);
 *                  the call copies its tensor table into it (no allocation)
 * Every non-empty tensor needs cols % 32 == 0 (else QMUON_ERR_UNSUPPORTED).
 * Gradients are read only; codes, scales, q8 and absmax equal those of
 * qmuon_update_mxfp8_carrier on each tensor alone. */
QMUON_API qmuon_status qmuon_update_mxfp8_carrier_multi(const qmuon_plan* plan, float beta,
                                              uint8_t* const* payloads, uint8_t* const* scale_invs,
                                              float* inv_norms, float* group_sumsq, void* ws,
                                              size_t ws_bytes, void* stream);

/* ---- 4-bit GRASP momentum state ("4-bit-Muon-GRASP", the update
 * equations and the grid quantisation on that page) ----
 * The momentum of a rows x cols matrix is a rank-8 factor P R^T plus a
 * residual, every piece grid-quantised: in each block an entry x is coded as
 * q = clamp(rint(x * L / min(r, c)), -L, L) with r, c the block's maxima of
 * |x| over the entry's row and column (stored in fp32) and L = 7 (residual,
 * 64 x 64 blocks) or 127 (P, R: blocks of 64 rows by all 8 columns).  Layouts
 * (row-major, all device memory, in/out):
 *   res       rows x cols/2 bytes: 4-bit codes q + 8, column 2c in the low nibble
 *   res_rmax  [cols/64][rows]     res_cmax [ceil(rows/64)][cols]
 *   p         rows x 8 int8       p_rmax [rows]   p_cmax [ceil(rows/64)][8]
 *   r         cols x 8 int8       r_rmax [cols]   r_cmax [ceil(cols/64)][8]
 *   grad      rows x cols bf16: g_t in, M_t out (round to nearest even)
 * A first step starts from a zero residual and P and a seeded R (the power
 * iteration's warm start). */
#define QMUON_GRASP_RANK 8
#define QMUON_GRASP_BLOCK 64
typedef struct {
  int64_t rows, cols;            /* rows >= 8 (else QMUON_ERR_INVALID_ARGUMENT: a rank-8 factor needs 8 rows),
                                    cols % 64 == 0 (else QMUON_ERR_UNSUPPORTED) */
  uint8_t* res;
  float* res_rmax;
  float* res_cmax;
  int8_t* p;
  float* p_rmax;
  float* p_cmax;
  int8_t* r;
  float* r_rmax;
  float* r_cmax;
  void* grad;
} qmuon_grasp_matrix;

/* Workspace bytes of qmuon_grasp_step for these matrices: 0 for a NULL array,
 * n <= 0, or any shape qmuon_grasp_step rejects (the state pointers are not
 * looked at, so the size can be asked for before the state is allocated). */
QMUON_API size_t qmuon_grasp_workspace_size(const qmuon_grasp_matrix* matrices, int32_t n);

/* One GRASP momentum step of n matrices (H array of descriptors):
 *   M_{t-1} = res + P R^T, M_t = mu M_{t-1} + g_t (fp32, one rounding per
 *   operation, the rank sum left to right), stored in bf16 over g_t;
 *   Q = ColNorm(R_{t-1}), P_t = orth(M_t Q) (thin QR, positive diagonal),
 *   R_t = M_t^T P_t, res_t = M_t - P_t R_t^T, all from the stored M_t;
 *   res_t, P_t, R_t are grid-quantised into the state.
 * Asynchronous on `stream`; M_t Q of rank below 8 records
 * QMUON_ERR_INVALID_ARGUMENT in the workspace header (qmuon_sync_status)
 * and leaves R and the residual unchanged. */
QMUON_API qmuon_status qmuon_grasp_step(const qmuon_grasp_matrix* matrices, int32_t n, float mu, void* ws,
                                        size_t ws_bytes, void* stream);

/* Input of one Newton-Schulz problem. */
typedef enum { QMUON_NS_BF16 = 0, QMUON_NS_MXFP8 = 1 } qmuon_ns_input;

/* One matrix to orthogonalise.
 *   x          D  bf16 rows x cols, row stride ld elements (ld >= cols,
 *                 ld % 8 == 0, x 16-byte aligned); IN: M, OUT: NS(inv*M)
 *                 (MXFP8 input: OUT only)
 *   inv_norm   D  fp32 scalar applied to the input, or NULL for 1
 *   input      QMUON_NS_BF16, or QMUON_NS_MXFP8 with payload/scale_inv:
 *   payload    D  rows x cols E4M3 codes (row stride cols), cols % 32 == 0,
 *                 16-byte aligned -- the carrier of qmuon_update_mxfp8_carrier
 *   scale_inv  D  rows x (cols/32) E8M0 bytes
 * An MXFP8 problem is expanded exactly (E4M3 times a power of two fits in
 * bf16) into x, which then receives the result; inv_norm is the carrier's. */
typedef struct {
  void* x;
  int64_t rows;
  int64_t cols;
  int64_t ld;
  const float* inv_norm;
  int32_t input;
  int32_t reserved;
  const uint8_t* payload;
  const uint8_t* scale_inv;
} qmuon_ns_problem;

/* Workspace bytes for qmuon_newton_schulz_batched on these problems: 0 for a
 * NULL array, n_problems <= 0, or any shape, stride or input kind the batched
 * call rejects (pointers are not looked at). */
QMUON_API size_t qmuon_ns_workspace_size(const qmuon_ns_problem* problems, int32_t n_problems);

/* Quintic Newton-Schulz on a batch of independent matrices, in place:
 * per iteration A = X X^T, B = b*A + c*A*A, X <- a*X + B*X (three products,
 * "NVIDIA impulsa optimizadores avanzados ... con Megatron", section
 * "Newton-Schulz distribuido"; the first two are symmetric, section "SYRK y
 * reducción fusionada").  A matrix with rows > cols is processed as its
 * transpose.  tcgen05 tensor cores, bf16 operands, fp32 accumulation.
 *   problems  H  n_problems entries (copied)
 *   iters     >= 1
 *   coeffs    H  (a, b, c) */
QMUON_API qmuon_status qmuon_newton_schulz_batched(const qmuon_ns_problem* problems, int32_t n_problems,
                                         int32_t iters, const float coeffs[3], void* ws,
                                         size_t ws_bytes, void* stream);

/* One MuonBP quantized Muon step over every tensor of the plan ("MuonBP:
 * Faster Muon via Block-Periodic Orthogonalization", section "整体框架"):
 * the momentum update of qmuon_update_multi_normalize_groups, then, when
 * t mod P == 0 (a full step; P == 1 is plain Muon), Newton-Schulz on each
 * whole matrix with one norm group per tensor and W <- W - eta_full*U;
 * otherwise (a block step; P == 0 means never full, i.e. BlockMuon)
 * Newton-Schulz on every tile of the plan's tiling, each with its own norm,
 * and W <- W - eta_block*U.  U (bf16) is left in each grad buffer.
 *   t          1-based step index
 *   weights    H  n_tensors device pointers (D) to fp32 rows x cols master
 *                 weights, updated in place
 *   group_sumsq D [n groups of this step] fp32 sums of m*m, or NULL
 * Once qmuon_step_prepare has built the plan's tables for these weights and
 * this workspace (and one step has run in the process), a step is a
 * workspace memset and kernel launches on `stream`, so it can be captured
 * into a CUDA graph.  The step index is fixed in the captured launches: a
 * captured period of P steps (t = 1 .. P) replays as any later period, with
 * nearest requantisation (stochastic requantisation would replay the same
 * random numbers). */
QMUON_API qmuon_status qmuon_step(const qmuon_plan* plan, int64_t t, int32_t P, float beta,
                        float eta_full, float eta_block, float* const* weights,
                        const float coeffs[3], int32_t iters, float* group_sumsq, void* ws,
                        size_t ws_bytes, void* stream);

/* Largest tensor (elements) qmuon_update_normalize_noalloc accepts. */
#define QMUON_NOALLOC_MAX_ELEMS ((int64_t)1 << 31)

/* The momentum update of one tensor with one norm group, for callers that
 * must not allocate device memory at this point -- for example a C caller
 * with no device allocator at hand, or code inside a framework whose caching
 * allocator owns the device's memory, where a side cudaMalloc could fail,
 * fragment that pool or escape its accounting, and where cudaMalloc/cudaFree
 * may also synchronise the device.  It needs no plan and no workspace and
 * calls neither cudaMalloc nor cudaFree: its scratch (the last-CTA ticket and
 * one partial sum per CTA, about 64 KB) is a static array compiled into the
 * library, which every GPU that loads the library holds until the process
 * exits.  The arithmetic and outputs are those of
 * qmuon_update_multi_normalize_groups on a plan holding this single tensor
 * with normalize_mode 2.  The pages have no counterpart: this entry exists
 * for integration only.
 *   tensor     H  q8/absmax D, updated in place; grad D, IN gradient, OUT m
 *   sumsq      D  one fp32, sum of m*m over the tensor, or NULL
 *   inv_norm   D  one fp32, 1/(sqrt(sum)+1e-7), or NULL
 * Tensors above QMUON_NOALLOC_MAX_ELEMS elements are rejected with
 * QMUON_ERR_INVALID_ARGUMENT (qmuon_last_error says why).  The first call on
 * a device looks up the array's device address with that device current;
 * make that first call before any stream capture begins.  Every call uses the
 * same array (the call clears what must start at zero), so calls that may
 * overlap on the GPU -- on different streams or from different threads --
 * race on it; enqueue them in order on one stream.
 * A failure the kernel detects on the GPU (a bounded wait that expired,
 * QMUON_ERR_TIMEOUT) cannot be returned by this asynchronous call: it is kept
 * in the static array, carried over by later calls (the first one is kept),
 * and reported by qmuon_noalloc_sync_status.  A call's outputs are valid only
 * if the next qmuon_noalloc_sync_status returns QMUON_OK. */
QMUON_API qmuon_status qmuon_update_normalize_noalloc(const qmuon_tensor* tensor, qmuon_q8_kind q8_kind,
                                                      qmuon_dtype grad_dtype, float beta, float* sumsq,
                                                      float* inv_norm, void* stream);

/* Waits for `stream`, then reads the status that the kernels of
 * qmuon_update_normalize_noalloc recorded in the static array of the current
 * device since the last read, and clears it.  Returns QMUON_OK, the recorded
 * status (qmuon_last_error names the kernel's site), or QMUON_ERR_CUDA if the
 * stream or the read failed.  It synchronises the calling thread and
 * allocates nothing.  The pages have no counterpart. */
QMUON_API qmuon_status qmuon_noalloc_sync_status(void* stream);

/* Writes `status` (a failure code, QMUON_ERR_INVALID_ARGUMENT ..
 * QMUON_ERR_OUT_OF_MEMORY) and `site` into the static array's pending status
 * on the current device, as a kernel would record them, so that a caller can
 * test its handling of a failure reported through qmuon_noalloc_sync_status
 * without making a kernel fail.  Synchronous; allocates nothing.  Returns
 * QMUON_ERR_INVALID_ARGUMENT for QMUON_OK or an unknown code (nothing
 * written).  The pages have no counterpart. */
QMUON_API qmuon_status qmuon_noalloc_inject_status(qmuon_status status, uint32_t site);

/* qmuon_step fed from host memory: the step's gradients are copied in, the
 * step runs, and its group sums are copied out, all enqueued without
 * blocking the caller.  The copies into the plan's gradient buffers go on
 * copy_stream and start once this plan's previous qmuon_step_from_host has
 * finished with those buffers; the step runs on `stream` once the copies
 * have landed.  With the plan's default ingest mode (qmuon_plan_set_host_ingest),
 * a gradient in page-locked host memory that the device can address
 * (cudaHostAlloc, or cudaHostRegister with cudaHostRegisterMapped), 16-byte
 * aligned, is read by a kernel's own loads over the host link; any other is
 * moved by cudaMemcpyAsync (qmuon_counters host_pulled_bytes and
 * host_copied_bytes count the two).  A caller that alternates two plans over the same q8 state
 * (the same q8/absmax pointers, different gradient buffers) therefore
 * overlaps step t+1's host->device copies with step t's kernels.  The
 * arithmetic and device outputs are those of qmuon_step.
 *   host_grads        H  n_tensors host pointers, each rows x cols bf16 in
 *                        row-major order (page-locked memory lets the copy
 *                        run asynchronously; pageable memory makes
 *                        cudaMemcpyAsync stage it before returning)
 *   host_group_sumsq  H  [n groups of this step kind] fp32, written when the
 *                        step completes on `stream`; NULL skips the read-back
 *   group_sumsq       D  as for qmuon_step (NULL: workspace scratch)
 *   copy_stream       stream of the host->device copies; NULL = `stream`
 *                     (no overlap)
 * Anything else that reads or writes the plan's gradient buffers must be
 * ordered against these calls by the caller.  Returns
 * QMUON_ERR_INVALID_ARGUMENT for a NULL host_grads or a NULL entry in it
 * (for a non-empty tensor). */
QMUON_API qmuon_status qmuon_step_from_host(const qmuon_plan* plan, int64_t t, int32_t P, float beta,
                                            float eta_full, float eta_block, float* const* weights,
                                            const float coeffs[3], int32_t iters,
                                            const void* const* host_grads, float* host_group_sumsq,
                                            float* group_sumsq, void* ws, size_t ws_bytes, void* stream,
                                            void* copy_stream);

/* Build, ahead of time, the Newton-Schulz problem tables qmuon_step needs for
 * both step kinds with these weights and this workspace (tensor maps and
 * tile lists; one synchronous upload each).  Optional: qmuon_step builds them
 * on first use and rebuilds them when the weights or workspace change, with
 * the upload enqueued on its stream behind the steps already there; preparing
 * keeps that host work out of the steps that follow, and must precede any
 * stream capture of them.  When tables already exist and change, this call
 * first waits for the device to finish every earlier launch, since earlier
 * steps may still be reading them.  Arguments as for qmuon_step. */
QMUON_API qmuon_status qmuon_step_prepare(const qmuon_plan* plan, float* const* weights, void* ws,
                                          size_t ws_bytes);

/* Synchronise `stream` and report a kernel-side error recorded in `ws`
 * (QMUON_ERR_TIMEOUT when a bounded wait expired), then clear it. */
QMUON_API qmuon_status qmuon_sync_status(void* ws, void* stream);

/* ---------------------------------------------------------------------------
 * Path and dtype audit.  "Quantized Muon Momentum", §Wave18B MXFP8 Carrier
 * Probe, checks a run with counters: calls of the carrier update and the
 * dtypes of the tensors it read and wrote (uint8 payload and scales, fp32
 * inverse norm, the gradient's dtype), and whether a bf16 path was taken.
 * The library keeps the same kind of tallies for every entry point that
 * computes, process-wide: a caller can check which paths ran, for example
 * that Newton-Schulz was fed from MXFP8 carriers and how many bytes of bf16
 * the carrier expansion wrote on the way (ns_bf16_handoff_bytes; the
 * expansion is the bf16 hand-off that the page's probe still needs).
 *
 * A call adds to the tallies once it has enqueued all of its work and is
 * about to return QMUON_OK; a call that fails adds nothing.  They count what
 * was enqueued, not what the GPU has finished.  Additions are relaxed atomic
 * ones, so calls from several threads are all counted.  Per-tensor fields
 * add one per non-empty tensor per call.
 * ------------------------------------------------------------------------- */
typedef struct qmuon_counters {
  uint64_t update_calls;            /* qmuon_update_multi_normalize_groups(_sr), qmuon_update_normalize_noalloc */
  uint64_t update_sr_calls;         /*   of those, with stochastic requantisation */
  uint64_t carrier_calls;           /* qmuon_update_mxfp8_carrier(_multi) */
  uint64_t ns_calls;                /* qmuon_newton_schulz_batched */
  uint64_t step_block_calls;        /* qmuon_step and qmuon_step_from_host, block steps */
  uint64_t step_full_calls;         /*   full steps */
  uint64_t step_sr_calls;           /*   steps with stochastic requantisation */
  uint64_t step_host_fed_calls;     /*   steps through qmuon_step_from_host */
  uint64_t grasp_calls;             /* qmuon_grasp_step */
  uint64_t grad_bf16_tensors;       /* gradients read by update, carrier, step and GRASP calls, by dtype */
  uint64_t grad_fp16_tensors;
  uint64_t grad_fp32_tensors;
  uint64_t state_int8_tensors;      /* 8-bit blockwise states updated (update, carrier and step calls) */
  uint64_t state_uint8_tensors;
  uint64_t carrier_payload_u8_tensors;   /* E4M3 payloads written (uint8) */
  uint64_t carrier_scale_u8_tensors;     /* E8M0 scale arrays written (uint8) */
  uint64_t carrier_inv_norm_f32_values;  /* fp32 inverse norms written by carrier calls */
  uint64_t ns_bf16_problems;        /* Newton-Schulz problems read as bf16 (batched calls and steps) */
  uint64_t ns_mxfp8_problems;       /* Newton-Schulz problems read from MXFP8 carriers */
  uint64_t ns_bf16_handoff_bytes;   /* bf16 bytes the carrier expansion wrote as Newton-Schulz input */
  uint64_t weight_f32_tensors;      /* fp32 master weights updated by steps */
  uint64_t grasp_matrices;          /* matrices whose 4-bit state qmuon_grasp_step updated */
  uint64_t host_pulled_bytes;       /* host-fed gradient bytes read by the device's own loads (page-locked memory) */
  uint64_t host_copied_bytes;       /* host-fed gradient bytes moved by cudaMemcpyAsync (other host memory) */
} qmuon_counters;

/* Copies the tallies into `out`: the first min(out_bytes, sizeof(qmuon_counters))
 * bytes, so a caller built against an older, shorter struct still reads its
 * own fields.  Returns QMUON_ERR_INVALID_ARGUMENT for a NULL `out`.  Host
 * only; no CUDA call. */
QMUON_API qmuon_status qmuon_get_counters(qmuon_counters* out, size_t out_bytes);

/* Sets every tally to zero.  Host only; no CUDA call. */
QMUON_API void qmuon_reset_counters(void);

/* Detail of the last non-OK status returned on the calling thread (which
 * call failed and the CUDA error string), or "" if none.  The pointer stays
 * valid until the next qmuon call on this thread. */
QMUON_API const char* qmuon_last_error(void);

/* Static description of a status code (never NULL). */
QMUON_API const char* qmuon_status_string(qmuon_status status);

/* Library version, e.g. "qmuon 0.1 sm_103a". */
QMUON_API const char* qmuon_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QMUON_H_ */

// Internal declarations shared by the qmuon translation units (not part of
// the public C ABI in include/qmuon.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <exception>
#include <new>

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "qmuon.h"

namespace qm {

// An NVTX range named after a C-ABI entry, open for the entry's host work and
// launches (visible to nsys/ncu; a no-op call when no tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

constexpr int kBlock = QMUON_BLOCK;   // elements per quantization block
constexpr int kUpdThreads = 256;      // 8 warps = 16 half-warps, one block per half-warp
constexpr int kMaxChunk = 2048;       // quantization blocks per CTA (shared-memory bound)
constexpr double kEps = 1e-7;         // added to the Frobenius norm

// Workspace header: the first kWsHeader bytes of every workspace.
struct WsHeader {
  unsigned int error;      // 0 = ok, else a qmuon_status recorded by a kernel
  unsigned int error_info; // where it happened (kernel-specific)
  unsigned int ticket;     // last-CTA counter of the update kernel (self-resetting)
  unsigned int pad[61];
};
constexpr size_t kWsHeader = sizeof(WsHeader);
static_assert(kWsHeader == 256, "workspace header is 256 bytes");

// One tensor as the update kernel sees it (device table entry).
struct UpdTensor {
  void* q8;
  float* absmax;
  void* grad;
  uint8_t* payload;     // carrier only
  uint8_t* scale;       // carrier only
  int64_t numel;
  int64_t block_begin;  // global index of the tensor's first quantization block
  int32_t index;        // the tensor's index in its plan (stochastic rounding's counter)
};

// Group layout of one launch: which norm group every block feeds, how the
// grid's CTAs map onto (CTA, group) partial-sum slots, and the per-group list
// of slots for the final deterministic reduction.  With block_group null the
// launch has one group holding every block and one slot per CTA.
struct GroupLayout {
  int32_t n_groups = 0;
  int32_t n_slots = 0;
  const int32_t* block_group = nullptr;     // [nb_total], -1 = no group
  const int32_t* cta_slot_begin = nullptr;  // [grid+1]
  const int32_t* slot_group = nullptr;      // [n_slots], ascending within a CTA
  const int32_t* grp_ptr = nullptr;         // [n_groups+1]
  const int32_t* grp_slots = nullptr;       // slots of each group, CTA order
};

struct UpdLaunch {
  const UpdTensor* tensors;   // device table, or null: use `single`
  const int64_t* tensor_begin;  // device [n_tensors+1] block_begin, last = nb_total
  UpdTensor single;           // the only tensor when `tensors` is null
  int32_t n_tensors;
  int64_t nb_total;
  int64_t chunk;              // blocks per CTA
  int32_t grid;
  float beta;
  GroupLayout layout;         // n_groups == 0: no reduction
  double* partials;           // workspace [n_slots]
  WsHeader* header;           // workspace header
  float* group_sumsq;         // D or null
  float* group_inv;           // D or null
  // stochastic requantisation: Philox4x32-10 key (seed) and the step word of its counter
  int32_t sr;
  uint32_t sr_key0, sr_key1, sr_step;
  // D: blocks whose sum of m*m is not finite are counted here, or null
  unsigned int* nonfinite;
};

// Update launch geometry: whole waves of resident CTAs, at most kMaxChunk
// blocks per CTA and at least 16 (one per half-warp).  Every entry that
// launches the update kernel takes its grid and chunk from here, so that the
// per-CTA partial sums are formed over the same blocks in the same order.
inline void update_geometry(int64_t nb, int sms, int per_sm, int32_t* grid, int64_t* chunk) {
  const int64_t wave = (int64_t)(sms > 1 ? sms : 1) * (per_sm > 1 ? per_sm : 1);
  int64_t g;
  if (nb <= wave * 16) {
    g = (nb + 15) / 16;
    if (g < 1) g = 1;
  } else {
    const int64_t waves = (nb + wave * kMaxChunk - 1) / (wave * kMaxChunk);
    g = wave * waves;
  }
  int64_t c = (nb + g - 1) / g;
  if (c < 1) c = 1;
  g = (nb + c - 1) / c;
  if (g < 1) g = 1;
  *grid = (int32_t)g;
  *chunk = c;
}

// Record the detail of a failure for qmuon_last_error() (api.cu); returns
// QMUON_ERR_CUDA (or `status`) for convenient `return set_error(...)`.
qmuon_status set_error(const char* where, cudaError_t e, qmuon_status status = QMUON_ERR_CUDA);
qmuon_status set_error_msg(const char* msg, qmuon_status status);
qmuon_status set_error_what(const char* where, const char* what, qmuon_status status);

// Runs the body of a C-ABI entry so that no C++ exception leaves the library:
// a host allocation that fails (std::bad_alloc, e.g. for the tables of a huge
// plan) returns QMUON_ERR_OUT_OF_MEMORY, any other exception
// QMUON_ERR_INVALID_ARGUMENT, with the detail kept for qmuon_last_error().
template <class Body>
qmuon_status no_throw(const char* where, Body&& body) noexcept {
  try {
    return body();
  } catch (const std::bad_alloc&) {
    return set_error_what(where, "host memory allocation failed", QMUON_ERR_OUT_OF_MEMORY);
  } catch (const std::exception& e) {
    return set_error_what(where, e.what(), QMUON_ERR_INVALID_ARGUMENT);
  } catch (...) {
    return set_error_what(where, "unexpected exception", QMUON_ERR_INVALID_ARGUMENT);
  }
}

// Path and dtype tallies behind qmuon_get_counters (api.cu), one per field
// of qmuon_counters, in the struct's order.
enum Tally {
  T_UPDATE_CALLS, T_UPDATE_SR_CALLS, T_CARRIER_CALLS, T_NS_CALLS, T_STEP_BLOCK_CALLS, T_STEP_FULL_CALLS,
  T_STEP_SR_CALLS, T_STEP_HOST_FED_CALLS, T_GRASP_CALLS, T_GRAD_BF16, T_GRAD_FP16, T_GRAD_FP32, T_STATE_INT8,
  T_STATE_UINT8, T_CARRIER_PAYLOAD_U8, T_CARRIER_SCALE_U8, T_CARRIER_INV_NORM_F32, T_NS_BF16_PROBLEMS,
  T_NS_MXFP8_PROBLEMS, T_NS_BF16_HANDOFF_BYTES, T_WEIGHT_F32, T_GRASP_MATRICES, T_HOST_PULLED_BYTES,
  T_HOST_COPIED_BYTES, T_COUNT
};
static_assert(sizeof(qmuon_counters) == T_COUNT * sizeof(uint64_t), "one tally per qmuon_counters field");
void tally(Tally t, uint64_t v = 1);
// One tensor read as a gradient of `dt` and one 8-bit state of `q8` updated.
void tally_grad_state(qmuon_dtype dt, qmuon_q8_kind q8, uint64_t tensors);

// Host-side launchers (update.cu).  Return a cudaError_t from the launch.
cudaError_t launch_update(const UpdLaunch& L, qmuon_q8_kind q8, qmuon_dtype dt, bool carrier,
                          cudaStream_t stream);
cudaError_t launch_scale_groups(const UpdLaunch& L, qmuon_dtype dt, const float* inv,
                                cudaStream_t stream);
int update_blocks_per_sm(qmuon_q8_kind q8, qmuon_dtype dt, bool carrier);

}  // namespace qm

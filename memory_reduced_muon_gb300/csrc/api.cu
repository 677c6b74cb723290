// C-ABI entry points of qmuon (declared in include/qmuon.h).
//
// Host side only: argument validation (before any CUDA call), plan tables,
// workspace carving and launches.  Every device computation happens in the
// kernels of update.cu and ns_gemm.cu.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <memory>
#include <new>
#include <vector>

#include "qm_internal.h"
#include "qm_ns.h"

using namespace qm;

namespace {

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline int64_t nblocks(int64_t numel) { return (numel + kBlock - 1) / kBlock; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool valid_q8(int v) { return v == QMUON_Q8_INT8 || v == QMUON_Q8_UINT8; }
inline bool valid_dtype(int v) { return v == QMUON_BF16 || v == QMUON_FP16 || v == QMUON_FP32; }

// Host copy of one group layout (uploaded into the plan's device table).
struct HostLayout {
  int32_t n_groups = 0;
  std::vector<int32_t> block_group;     // [nb]
  std::vector<int32_t> cta_slot_begin;  // [grid+1]
  std::vector<int32_t> slot_group;      // [n_slots]
  std::vector<int32_t> grp_ptr;         // [n_groups+1]
  std::vector<int32_t> grp_slots;       // [n_slots]
};

// Slots: for every CTA, one per distinct group among its blocks (ascending).
void build_slots(HostLayout& L, int32_t grid, int64_t chunk, int64_t nb) {
  L.cta_slot_begin.assign(grid + 1, 0);
  L.slot_group.clear();
  std::vector<std::vector<int32_t>> per_group(L.n_groups);
  std::vector<int32_t> seen;
  for (int32_t c = 0; c < grid; ++c) {
    L.cta_slot_begin[c] = (int32_t)L.slot_group.size();
    const int64_t b0 = (int64_t)c * chunk, b1 = std::min(nb, b0 + chunk);
    seen.clear();
    for (int64_t b = b0; b < b1; ++b) {
      const int32_t g = L.block_group[b];
      if (g >= 0 && (seen.empty() || seen.back() != g)) seen.push_back(g);
    }
    std::sort(seen.begin(), seen.end());
    seen.erase(std::unique(seen.begin(), seen.end()), seen.end());
    for (int32_t g : seen) {
      per_group[g].push_back((int32_t)L.slot_group.size());
      L.slot_group.push_back(g);
    }
  }
  L.cta_slot_begin[grid] = (int32_t)L.slot_group.size();
  L.grp_ptr.assign(L.n_groups + 1, 0);
  L.grp_slots.clear();
  for (int32_t g = 0; g < L.n_groups; ++g) {
    L.grp_ptr[g] = (int32_t)L.grp_slots.size();
    L.grp_slots.insert(L.grp_slots.end(), per_group[g].begin(), per_group[g].end());
  }
  L.grp_ptr[L.n_groups] = (int32_t)L.grp_slots.size();
}

thread_local char g_last_error[512] = "";

}  // namespace

qmuon_status qm::set_error(const char* where, cudaError_t e, qmuon_status status) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", where, cudaGetErrorString(e),
                cudaGetErrorName(e));
  return status;
}

qmuon_status qm::set_error_msg(const char* msg, qmuon_status status) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s", msg);
  return status;
}

qmuon_status qm::set_error_what(const char* where, const char* what, qmuon_status status) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", where, what);
  return status;
}

namespace {
std::atomic<uint64_t> g_tally[T_COUNT];
}  // namespace

void qm::tally(Tally t, uint64_t v) { g_tally[t].fetch_add(v, std::memory_order_relaxed); }

void qm::tally_grad_state(qmuon_dtype dt, qmuon_q8_kind q8, uint64_t tensors) {
  tally(dt == QMUON_BF16 ? T_GRAD_BF16 : dt == QMUON_FP16 ? T_GRAD_FP16 : T_GRAD_FP32, tensors);
  tally(q8 == QMUON_Q8_INT8 ? T_STATE_INT8 : T_STATE_UINT8, tensors);
}

extern "C" qmuon_status qmuon_get_counters(qmuon_counters* out, size_t out_bytes) {
  if (!out) return QMUON_ERR_INVALID_ARGUMENT;
  uint64_t v[T_COUNT];
  for (int i = 0; i < T_COUNT; ++i) v[i] = g_tally[i].load(std::memory_order_relaxed);
  std::memcpy(out, v, std::min(out_bytes, sizeof(v)));
  return QMUON_OK;
}

extern "C" void qmuon_reset_counters(void) {
  for (int i = 0; i < T_COUNT; ++i) g_tally[i].store(0, std::memory_order_relaxed);
}

// ---------------------------------------------------------------------------
// the plan
// ---------------------------------------------------------------------------
struct qmuon_plan {
  int device = 0;
  int num_sms = 0;
  std::vector<qmuon_tensor> tensors;
  qmuon_q8_kind q8 = QMUON_Q8_INT8;
  qmuon_dtype dt = QMUON_BF16;
  int32_t tile_r = 1, tile_c = 1;
  int64_t nb_total = 0;
  std::vector<int64_t> tensor_begin;  // [n+1]
  int32_t grid = 0;
  int64_t chunk = 0;
  // layouts: 0 = segments (qmuon_update_multi_normalize_groups), 1 = one group
  // per tensor (full steps), 2 = tiles (block steps)
  GroupLayout layout[3];
  int32_t n_slots_max = 0;
  void* d_table = nullptr;            // one device allocation for every table
  UpdTensor* d_tensors = nullptr;
  int64_t* d_tensor_begin = nullptr;
  ns::StepTables* ns_full = nullptr;  // Newton-Schulz problem sets of qmuon_step
  ns::StepTables* ns_block = nullptr;
  bool sr = false;                    // qmuon_step requantises stochastically (counter step = t)
  uint64_t sr_seed = 0;
  unsigned int* nonfinite = nullptr;  // device counter of non-finite blocks, or null
  // qmuon_step_from_host: gradient buffers free again / host copies landed
  cudaEvent_t grads_free = nullptr;
  cudaEvent_t grads_copied = nullptr;
  bool grads_free_recorded = false;
  int32_t host_ingest = QMUON_INGEST_PULL;   // qmuon_plan_set_host_ingest
};

namespace {

// Host-fed gradients in page-locked host memory that the device can address
// are read by the SMs' own loads (host_pull_kernel) rather than copied by the
// copy engines (plan default, qmuon_plan_set_host_ingest).  Both move a step's
// 1.74 GB of bf16 gradients at about 211 GB/s on GB300, but copy-engine
// transfers of the same buffers showed periodic stalls of 70-120 ms every
// ~510 ms that SM loads did not.  The pull runs beside the previous step's
// kernels; its host reads slow them down, the more so the more CTAs issue
// them (a block step's Newton-Schulz products by about 7 ms with one CTA per
// SM, 2.8 ms with 16-19 CTAs), so it takes one 256-thread CTA per 8 SMs, each
// thread with four 16-byte loads in flight (about 300 KB in flight), which
// still moves the 1.74 GB in about 9.6 ms.
constexpr int kPullMax = 64;   // tensors per launch
struct HostPull {
  int32_t n;
  const uint4* src[kPullMax];   // device addresses of the page-locked host buffers
  uint4* dst[kPullMax];
  uint64_t n16[kPullMax];       // 16-byte units
};

__global__ void __launch_bounds__(256) host_pull_kernel(const __grid_constant__ HostPull p) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  const uint64_t t0 = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int j = 0; j < p.n; ++j) {
    const uint4* __restrict__ src = p.src[j];
    uint4* __restrict__ dst = p.dst[j];
    const uint64_t n = p.n16[j];
    uint64_t i = t0;
    // four independent 16-byte loads in flight per thread
    for (; i + 3 * stride < n; i += 4 * stride) {
      const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
      dst[i] = a;
      dst[i + stride] = b;
      dst[i + 2 * stride] = c;
      dst[i + 3 * stride] = d;
    }
    for (; i < n; i += stride) dst[i] = src[i];
  }
}

// The device address of `p` if it is page-locked host memory mapped into the
// device's address space, else null.
const void* device_view_of_host(const void* p) {
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return pa.type == cudaMemoryTypeHost ? pa.devicePointer : nullptr;
}

int sm_count_of_current_device() {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < 64 && cached[dev].load(std::memory_order_relaxed) > 0) return cached[dev].load(std::memory_order_relaxed);
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cached[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

uint64_t nonempty_tensors(const qmuon_plan* plan) {
  uint64_t k = 0;
  for (const qmuon_tensor& T : plan->tensors) k += (T.rows * T.cols != 0) ? 1 : 0;
  return k;
}

qmuon_status validate_tensor(const qmuon_tensor& t, qmuon_dtype dt) {
  if (t.rows < 0 || t.cols < 0) return QMUON_ERR_INVALID_ARGUMENT;
  if (t.rows > 0 && t.cols > (((int64_t)1 << 40) / t.rows)) return QMUON_ERR_INVALID_ARGUMENT;
  const int64_t n = t.rows * t.cols;
  if (n == 0) return QMUON_OK;
  if (!t.q8 || !t.absmax || !t.grad) return QMUON_ERR_INVALID_ARGUMENT;
  if (!aligned(t.q8, 16) || !aligned(t.grad, 16) || !aligned(t.absmax, 4)) return QMUON_ERR_INVALID_ARGUMENT;
  (void)dt;
  return QMUON_OK;
}

}  // namespace

extern "C" qmuon_status qmuon_plan_create(const qmuon_tensor* tensors, int32_t n_tensors,
                                          qmuon_q8_kind q8_kind, qmuon_dtype grad_dtype,
                                          const qmuon_norm_segment* segments, int32_t n_segments,
                                          int32_t n_groups, int32_t tile_r, int32_t tile_c,
                                          qmuon_plan** out) {
  qm::NvtxRange nvtx_range("qmuon_plan_create");
  return qm::no_throw("qmuon_plan_create", [&]() -> qmuon_status {
    // ---- host validation: nothing below touches CUDA until it all passes ----
    if (!out) return QMUON_ERR_INVALID_ARGUMENT;
    *out = nullptr;
    if (!tensors || n_tensors <= 0) return QMUON_ERR_INVALID_ARGUMENT;
    if (!valid_q8(q8_kind) || !valid_dtype(grad_dtype)) return QMUON_ERR_INVALID_ARGUMENT;
    if (tile_r < 1 || tile_c < 1) return QMUON_ERR_INVALID_ARGUMENT;
    if (n_segments < 0 || (n_segments > 0 && !segments)) return QMUON_ERR_INVALID_ARGUMENT;
    const bool per_tensor = (segments == nullptr || n_segments == 0);
    if (per_tensor && n_groups != 0 && n_groups != n_tensors) return QMUON_ERR_INVALID_ARGUMENT;
    if (!per_tensor && n_groups <= 0) return QMUON_ERR_INVALID_ARGUMENT;
    std::vector<int64_t> begin(n_tensors + 1, 0);
    for (int32_t i = 0; i < n_tensors; ++i) {
      const qmuon_status s = validate_tensor(tensors[i], grad_dtype);
      if (s != QMUON_OK) return s;
      begin[i + 1] = begin[i] + nblocks(tensors[i].rows * tensors[i].cols);
    }
    const int64_t nb = begin[n_tensors];
    if (nb == 0 || nb > ((int64_t)1 << 31) - 1) return QMUON_ERR_INVALID_ARGUMENT;
    // tiles of the MuonBP block steps must be whole 256-element runs
    for (int32_t i = 0; i < n_tensors; ++i) {
      const int64_t R = tensors[i].rows, C = tensors[i].cols;
      if (R * C == 0) continue;
      if (R % tile_r || C % tile_c) return QMUON_ERR_INVALID_ARGUMENT;
      if (tile_c > 1) {
        if (C % kBlock || (C / tile_c) % kBlock) return QMUON_ERR_MISALIGNED_SEGMENT;
      } else if (tile_r > 1) {
        if (((R / tile_r) * C) % kBlock) return QMUON_ERR_MISALIGNED_SEGMENT;
      }
    }

    std::unique_ptr<qmuon_plan> P(new qmuon_plan);
    P->tensors.assign(tensors, tensors + n_tensors);
    P->q8 = q8_kind;
    P->dt = grad_dtype;
    P->tile_r = tile_r;
    P->tile_c = tile_c;
    P->nb_total = nb;
    P->tensor_begin = begin;

    // ---- group layouts (host) ----
    HostLayout H[3];
    H[1].n_groups = n_tensors;
    H[1].block_group.resize(nb);
    for (int32_t i = 0; i < n_tensors; ++i)
      std::fill(H[1].block_group.begin() + begin[i], H[1].block_group.begin() + begin[i + 1], i);
    if (per_tensor) {
      H[0].n_groups = n_tensors;
      H[0].block_group = H[1].block_group;
    } else {
      H[0].n_groups = n_groups;
      H[0].block_group.assign(nb, -1);
      for (int32_t s = 0; s < n_segments; ++s) {
        const qmuon_norm_segment& g = segments[s];
        if (g.tensor_index < 0 || g.tensor_index >= n_tensors) return QMUON_ERR_INVALID_ARGUMENT;
        if (g.group_id < 0 || g.group_id >= n_groups) return QMUON_ERR_INVALID_ARGUMENT;
        const int64_t n = tensors[g.tensor_index].rows * tensors[g.tensor_index].cols;
        if (g.start < 0 || g.length <= 0 || g.start + g.length > n) return QMUON_ERR_INVALID_ARGUMENT;
        const int64_t end = g.start + g.length;
        if (g.start % kBlock || (end % kBlock && end != n)) return QMUON_ERR_MISALIGNED_SEGMENT;
        for (int64_t b = begin[g.tensor_index] + g.start / kBlock,
                     e = begin[g.tensor_index] + nblocks(end); b < e; ++b) {
          if (H[0].block_group[b] >= 0) return QMUON_ERR_INVALID_ARGUMENT;  // overlap
          H[0].block_group[b] = g.group_id;
        }
      }
    }
    {
      int32_t gbase = 0;
      H[2].block_group.assign(nb, -1);
      for (int32_t i = 0; i < n_tensors; ++i) {
        const int64_t R = tensors[i].rows, C = tensors[i].cols;
        if (R * C == 0) continue;
        const int64_t th = R / tile_r, tw = C / tile_c;
        for (int64_t r = 0; r < R; ++r)
          for (int64_t c0 = 0; c0 < C; c0 += tw) {
            const int32_t g = gbase + (int32_t)((r / th) * tile_c + c0 / tw);
            const int64_t e0 = r * C + c0, e1 = e0 + tw;
            for (int64_t b = e0 / kBlock; b < nblocks(e1); ++b) H[2].block_group[begin[i] + b] = g;
          }
        gbase += tile_r * tile_c;
      }
      H[2].n_groups = gbase;
    }

    // ---- device properties and geometry ----
    cudaError_t ce = cudaGetDevice(&P->device);
    if (ce != cudaSuccess) return set_error("qmuon_plan_create (cudaGetDevice)", ce);
    ce = cudaDeviceGetAttribute(&P->num_sms, cudaDevAttrMultiProcessorCount, P->device);
    if (ce != cudaSuccess) return set_error("qmuon_plan_create (SM count)", ce);
    const int per_sm = update_blocks_per_sm(q8_kind, grad_dtype, false);
    if (per_sm <= 0) return set_error_msg("qmuon_plan_create: occupancy query failed", QMUON_ERR_CUDA);
    update_geometry(nb, P->num_sms, per_sm, &P->grid, &P->chunk);
    for (auto& h : H) build_slots(h, P->grid, P->chunk, nb);

    // ---- one device allocation for every table, one H2D copy ----
    std::vector<UpdTensor> ut(n_tensors);
    for (int32_t i = 0; i < n_tensors; ++i) {
      ut[i].q8 = tensors[i].q8;
      ut[i].absmax = tensors[i].absmax;
      ut[i].grad = tensors[i].grad;
      ut[i].payload = nullptr;
      ut[i].scale = nullptr;
      ut[i].numel = tensors[i].rows * tensors[i].cols;
      ut[i].block_begin = begin[i];
      ut[i].index = i;
    }
    std::vector<unsigned char> blob;
    auto put = [&blob](const void* src, size_t bytes) {
      const size_t off = align_up(blob.size(), 256);
      blob.resize(off + bytes);
      if (bytes) std::memcpy(blob.data() + off, src, bytes);
      return off;
    };
    const size_t o_t = put(ut.data(), ut.size() * sizeof(UpdTensor));
    const size_t o_b = put(begin.data(), begin.size() * sizeof(int64_t));
    size_t o_l[3][5];
    for (int l = 0; l < 3; ++l) {
      o_l[l][0] = put(H[l].block_group.data(), H[l].block_group.size() * 4);
      o_l[l][1] = put(H[l].cta_slot_begin.data(), H[l].cta_slot_begin.size() * 4);
      o_l[l][2] = put(H[l].slot_group.data(), H[l].slot_group.size() * 4);
      o_l[l][3] = put(H[l].grp_ptr.data(), H[l].grp_ptr.size() * 4);
      o_l[l][4] = put(H[l].grp_slots.data(), H[l].grp_slots.size() * 4);
    }
    ce = cudaMalloc(&P->d_table, blob.size());
    if (ce != cudaSuccess) return set_error("qmuon_plan_create (cudaMalloc tables)", ce);
    ce = cudaMemcpy(P->d_table, blob.data(), blob.size(), cudaMemcpyHostToDevice);
    if (ce != cudaSuccess) {
      cudaFree(P->d_table);
      return set_error("qmuon_plan_create (upload tables)", ce);
    }
    unsigned char* base = static_cast<unsigned char*>(P->d_table);
    P->d_tensors = reinterpret_cast<UpdTensor*>(base + o_t);
    P->d_tensor_begin = reinterpret_cast<int64_t*>(base + o_b);
    for (int l = 0; l < 3; ++l) {
      GroupLayout& G = P->layout[l];
      G.n_groups = H[l].n_groups;
      G.n_slots = (int32_t)H[l].slot_group.size();
      G.block_group = reinterpret_cast<const int32_t*>(base + o_l[l][0]);
      G.cta_slot_begin = reinterpret_cast<const int32_t*>(base + o_l[l][1]);
      G.slot_group = reinterpret_cast<const int32_t*>(base + o_l[l][2]);
      G.grp_ptr = reinterpret_cast<const int32_t*>(base + o_l[l][3]);
      G.grp_slots = reinterpret_cast<const int32_t*>(base + o_l[l][4]);
      P->n_slots_max = std::max(P->n_slots_max, G.n_slots);
    }
    *out = P.release();
    return QMUON_OK;
  });
}

extern "C" void qmuon_plan_destroy(qmuon_plan* plan) {
  if (!plan) return;
  if (plan->d_table) cudaFree(plan->d_table);
  if (plan->grads_free) cudaEventDestroy(plan->grads_free);
  if (plan->grads_copied) cudaEventDestroy(plan->grads_copied);
  ns::destroy_step_tables(plan->ns_full);
  ns::destroy_step_tables(plan->ns_block);
  delete plan;
}

extern "C" qmuon_status qmuon_plan_info(const qmuon_plan* plan, int64_t* n_blocks, int32_t* n_groups,
                                        int32_t* n_full_groups, int32_t* n_block_groups) {
  if (!plan) return QMUON_ERR_INVALID_ARGUMENT;
  if (n_blocks) *n_blocks = plan->nb_total;
  if (n_groups) *n_groups = plan->layout[0].n_groups;
  if (n_full_groups) *n_full_groups = plan->layout[1].n_groups;
  if (n_block_groups) *n_block_groups = plan->layout[2].n_groups;
  return QMUON_OK;
}

namespace {

// Workspace carving: [header | partials | group sums | group inverse norms | NS]
struct UpdWs {
  WsHeader* header;
  double* partials;
  float* sumsq;
  float* inv;
  UpdTensor* table;         // per-call tensor table (multi-tensor carrier)
  unsigned char* ns;
  size_t ns_bytes;
};

size_t table_bytes(const qmuon_plan* p) { return align_up(std::max<size_t>(p->tensors.size(), 1) * sizeof(UpdTensor), 256); }

size_t update_ws_bytes(const qmuon_plan* p) {
  int32_t gmax = 0;
  for (const auto& l : p->layout) gmax = std::max(gmax, l.n_groups);
  return kWsHeader + align_up((size_t)std::max(p->n_slots_max, 1) * 8, 256) +
         2 * align_up((size_t)std::max(gmax, 1) * 4, 256) + table_bytes(p);
}

UpdWs carve(const qmuon_plan* p, void* ws, size_t ws_bytes) {
  int32_t gmax = 0;
  for (const auto& l : p->layout) gmax = std::max(gmax, l.n_groups);
  unsigned char* b = static_cast<unsigned char*>(ws);
  UpdWs w;
  w.header = reinterpret_cast<WsHeader*>(b);
  size_t off = kWsHeader;
  w.partials = reinterpret_cast<double*>(b + off);
  off += align_up((size_t)std::max(p->n_slots_max, 1) * 8, 256);
  w.sumsq = reinterpret_cast<float*>(b + off);
  off += align_up((size_t)std::max(gmax, 1) * 4, 256);
  w.inv = reinterpret_cast<float*>(b + off);
  off += align_up((size_t)std::max(gmax, 1) * 4, 256);
  w.table = reinterpret_cast<UpdTensor*>(b + off);
  off += table_bytes(p);
  w.ns = b + off;
  w.ns_bytes = ws_bytes > off ? ws_bytes - off : 0;
  return w;
}

UpdLaunch make_launch(const qmuon_plan* p, int layout, float beta, const UpdWs& w,
                      float* sumsq, float* inv) {
  UpdLaunch L{};
  L.tensors = p->d_tensors;
  L.tensor_begin = p->d_tensor_begin;
  L.n_tensors = (int32_t)p->tensors.size();
  L.nb_total = p->nb_total;
  L.chunk = p->chunk;
  L.grid = p->grid;
  L.beta = beta;
  L.layout = p->layout[layout];
  L.partials = w.partials;
  L.header = w.header;
  L.group_sumsq = sumsq;
  L.group_inv = inv;
  L.nonfinite = p->nonfinite;
  return L;
}

}  // namespace

extern "C" size_t qmuon_workspace_size(const qmuon_plan* plan, qmuon_ws_kind which) {
  if (!plan || (which != QMUON_WS_UPDATE && which != QMUON_WS_STEP)) return 0;
  size_t b = update_ws_bytes(plan);
  if (which == QMUON_WS_STEP) {
    const size_t a = ns::step_workspace_bytes(plan->tensors.data(), (int32_t)plan->tensors.size(), 1, 1);
    const size_t c = ns::step_workspace_bytes(plan->tensors.data(), (int32_t)plan->tensors.size(),
                                              plan->tile_r, plan->tile_c);
    b += std::max(a, c);
  }
  return b;
}

namespace {

void set_sr(UpdLaunch& L, bool on, uint64_t seed, int64_t step) {
  L.sr = on ? 1 : 0;
  L.sr_key0 = (uint32_t)seed;
  L.sr_key1 = (uint32_t)(seed >> 32);
  L.sr_step = (uint32_t)step;
}

qmuon_status update_groups(const qmuon_plan* plan, float beta, int32_t normalize_mode, float* group_sumsq,
                           float* group_inv_norm, void* ws, size_t ws_bytes, void* stream, bool sr,
                           uint64_t seed, int64_t step) {
  if (!plan || !ws) return QMUON_ERR_INVALID_ARGUMENT;
  if (normalize_mode < 0 || normalize_mode > 2) return QMUON_ERR_INVALID_ARGUMENT;
  if (normalize_mode == 2 && !group_inv_norm) return QMUON_ERR_INVALID_ARGUMENT;
  if (!aligned(ws, 256)) return QMUON_ERR_INVALID_ARGUMENT;
  if (ws_bytes < update_ws_bytes(plan)) return QMUON_ERR_WORKSPACE_TOO_SMALL;
  if ((group_sumsq && !aligned(group_sumsq, 4)) || (group_inv_norm && !aligned(group_inv_norm, 4)))
    return QMUON_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const UpdWs w = carve(plan, ws, ws_bytes);
  float* inv = group_inv_norm;
  if (normalize_mode == 1 && !inv) inv = w.inv;
  const bool reduce = group_sumsq || inv;
  UpdLaunch L = make_launch(plan, 0, beta, w, group_sumsq, inv);
  if (!reduce) L.layout.n_groups = 0;
  set_sr(L, sr, seed, step);
  cudaError_t e = cudaMemsetAsync(w.header, 0, kWsHeader, s);
  if (e == cudaSuccess) e = launch_update(L, plan->q8, plan->dt, false, s);
  if (e == cudaSuccess && normalize_mode == 1) e = launch_scale_groups(L, plan->dt, inv, s);
  if (e != cudaSuccess) return set_error("qmuon_update_multi_normalize_groups (launch)", e);
  tally(T_UPDATE_CALLS);
  if (sr) tally(T_UPDATE_SR_CALLS);
  tally_grad_state(plan->dt, plan->q8, nonempty_tensors(plan));
  return QMUON_OK;
}

}  // namespace

extern "C" qmuon_status qmuon_update_multi_normalize_groups(const qmuon_plan* plan, float beta,
                                                            int32_t normalize_mode,
                                                            float* group_sumsq, float* group_inv_norm,
                                                            void* ws, size_t ws_bytes, void* stream) {
  qm::NvtxRange nvtx_range("qmuon_update_multi_normalize_groups");
  return update_groups(plan, beta, normalize_mode, group_sumsq, group_inv_norm, ws, ws_bytes, stream, false, 0, 0);
}

extern "C" qmuon_status qmuon_update_multi_normalize_groups_sr(const qmuon_plan* plan, float beta,
                                                               int32_t normalize_mode, uint64_t seed, int64_t step,
                                                               float* group_sumsq, float* group_inv_norm,
                                                               void* ws, size_t ws_bytes, void* stream) {
  qm::NvtxRange nvtx_range("qmuon_update_multi_normalize_groups_sr");
  return update_groups(plan, beta, normalize_mode, group_sumsq, group_inv_norm, ws, ws_bytes, stream, true, seed,
                       step);
}

extern "C" qmuon_status qmuon_plan_set_nonfinite_counter(qmuon_plan* plan, uint32_t* counter) {
  if (!plan || (counter && (reinterpret_cast<uintptr_t>(counter) & 3))) return QMUON_ERR_INVALID_ARGUMENT;
  plan->nonfinite = reinterpret_cast<unsigned int*>(counter);
  return QMUON_OK;
}

extern "C" qmuon_status qmuon_plan_set_host_ingest(qmuon_plan* plan, int32_t mode) {
  if (!plan || (mode != QMUON_INGEST_PULL && mode != QMUON_INGEST_COPY)) return QMUON_ERR_INVALID_ARGUMENT;
  plan->host_ingest = mode;
  return QMUON_OK;
}

extern "C" qmuon_status qmuon_plan_set_stochastic_rounding(qmuon_plan* plan, int32_t enable, uint64_t seed) {
  if (!plan || (enable != 0 && enable != 1)) return QMUON_ERR_INVALID_ARGUMENT;
  plan->sr = enable != 0;
  plan->sr_seed = seed;
  return QMUON_OK;
}

extern "C" size_t qmuon_carrier_workspace_size(int64_t rows, int64_t cols) {
  if (rows <= 0 || cols <= 0) return kWsHeader;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int per_sm = std::max(1, update_blocks_per_sm(QMUON_Q8_INT8, QMUON_BF16, true));
  int32_t grid = 0;
  int64_t chunk = 0;
  update_geometry(nblocks(rows * cols), sms, per_sm, &grid, &chunk);
  return kWsHeader + align_up((size_t)grid * 8, 256);
}

extern "C" qmuon_status qmuon_update_mxfp8_carrier(const qmuon_tensor* tensor, qmuon_q8_kind q8_kind,
                                                   qmuon_dtype grad_dtype, float beta, uint8_t* payload,
                                                   uint8_t* scale_inv, float* inv_norm, void* ws,
                                                   size_t ws_bytes, void* stream) {
  qm::NvtxRange nvtx_range("qmuon_update_mxfp8_carrier");
  if (!tensor || !payload || !scale_inv || !inv_norm || !ws) return QMUON_ERR_INVALID_ARGUMENT;
  if (!valid_q8(q8_kind) || !valid_dtype(grad_dtype)) return QMUON_ERR_INVALID_ARGUMENT;
  const qmuon_status vs = validate_tensor(*tensor, grad_dtype);
  if (vs != QMUON_OK) return vs;
  const int64_t n = tensor->rows * tensor->cols;
  if (n == 0) return QMUON_ERR_INVALID_ARGUMENT;
  if (tensor->cols % QMUON_SCALE_BLOCK) return QMUON_ERR_UNSUPPORTED;
  if (!aligned(payload, 16) || !aligned(ws, 256) || !aligned(inv_norm, 4)) return QMUON_ERR_INVALID_ARGUMENT;
  int dev = 0, sms = 0;
  cudaError_t de = cudaGetDevice(&dev);
  if (de == cudaSuccess) de = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (de != cudaSuccess) return set_error("qmuon_update_mxfp8_carrier (device query)", de);
  const int per_sm = update_blocks_per_sm(q8_kind, grad_dtype, true);
  if (per_sm <= 0) return set_error_msg("qmuon_update_mxfp8_carrier: occupancy query failed", QMUON_ERR_CUDA);
  int32_t grid = 0;
  int64_t chunk = 0;
  update_geometry(nblocks(n), sms, per_sm, &grid, &chunk);
  if (ws_bytes < kWsHeader + align_up((size_t)grid * 8, 256)) return QMUON_ERR_WORKSPACE_TOO_SMALL;
  unsigned char* b = static_cast<unsigned char*>(ws);
  UpdLaunch L{};
  L.tensors = nullptr;
  L.single.q8 = tensor->q8;
  L.single.absmax = tensor->absmax;
  L.single.grad = tensor->grad;
  L.single.payload = payload;
  L.single.scale = scale_inv;
  L.single.numel = n;
  L.single.block_begin = 0;
  L.n_tensors = 1;
  L.nb_total = nblocks(n);
  L.chunk = chunk;
  L.grid = grid;
  L.beta = beta;
  L.layout.n_groups = 1;   // block_group == null: one group, one slot per CTA
  L.header = reinterpret_cast<WsHeader*>(b);
  L.partials = reinterpret_cast<double*>(b + kWsHeader);
  L.group_sumsq = nullptr;
  L.group_inv = inv_norm;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(L.header, 0, kWsHeader, s);
  if (e == cudaSuccess) e = launch_update(L, q8_kind, grad_dtype, true, s);
  if (e != cudaSuccess) return set_error("qmuon_update_mxfp8_carrier (launch)", e);
  tally(T_CARRIER_CALLS);
  tally_grad_state(grad_dtype, q8_kind, 1);
  tally(T_CARRIER_PAYLOAD_U8);
  tally(T_CARRIER_SCALE_U8);
  tally(T_CARRIER_INV_NORM_F32);
  return QMUON_OK;
}

extern "C" qmuon_status qmuon_update_mxfp8_carrier_multi(const qmuon_plan* plan, float beta, uint8_t* const* payloads,
                                                         uint8_t* const* scale_invs, float* inv_norms,
                                                         float* group_sumsq, void* ws, size_t ws_bytes,
                                                         void* stream) {
  qm::NvtxRange nvtx_range("qmuon_update_mxfp8_carrier_multi");
  return qm::no_throw("qmuon_update_mxfp8_carrier_multi", [&]() -> qmuon_status {
    if (!plan || !payloads || !scale_invs || !inv_norms || !ws) return QMUON_ERR_INVALID_ARGUMENT;
    if (!aligned(ws, 256) || !aligned(inv_norms, 4) || (group_sumsq && !aligned(group_sumsq, 4)))
      return QMUON_ERR_INVALID_ARGUMENT;
    if (ws_bytes < update_ws_bytes(plan)) return QMUON_ERR_WORKSPACE_TOO_SMALL;
    const int32_t n = (int32_t)plan->tensors.size();
    std::vector<UpdTensor> ut(n);
    for (int32_t i = 0; i < n; ++i) {
      const qmuon_tensor& T = plan->tensors[i];
      const int64_t numel = T.rows * T.cols;
      if (numel > 0) {
        if (T.cols % QMUON_SCALE_BLOCK) return QMUON_ERR_UNSUPPORTED;
        if (!payloads[i] || !scale_invs[i] || !aligned(payloads[i], 16)) return QMUON_ERR_INVALID_ARGUMENT;
      }
      ut[i].q8 = T.q8;
      ut[i].absmax = T.absmax;
      ut[i].grad = T.grad;
      ut[i].payload = payloads[i];
      ut[i].scale = scale_invs[i];
      ut[i].numel = numel;
      ut[i].block_begin = plan->tensor_begin[i];
      ut[i].index = i;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const UpdWs w = carve(plan, ws, ws_bytes);
    // one group per tensor (the plan's full-step layout): inverse norm i is tensor i's
    UpdLaunch L = make_launch(plan, 1, beta, w, group_sumsq, inv_norms);
    L.tensors = w.table;
    cudaError_t e = cudaMemcpyAsync(w.table, ut.data(), n * sizeof(UpdTensor), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(w.header, 0, kWsHeader, s);
    if (e == cudaSuccess) e = launch_update(L, plan->q8, plan->dt, true, s);
    // the pageable host table is staged by the copy before it returns
    if (e != cudaSuccess) return set_error("qmuon_update_mxfp8_carrier_multi (launch)", e);
    const uint64_t k = nonempty_tensors(plan);
    tally(T_CARRIER_CALLS);
    tally_grad_state(plan->dt, plan->q8, k);
    tally(T_CARRIER_PAYLOAD_U8, k);
    tally(T_CARRIER_SCALE_U8, k);
    tally(T_CARRIER_INV_NORM_F32, k);
    return QMUON_OK;
  });
}

// ---------------------------------------------------------------------------
// Newton-Schulz and the MuonBP step
// ---------------------------------------------------------------------------
extern "C" size_t qmuon_ns_workspace_size(const qmuon_ns_problem* problems, int32_t n_problems) {
  if (!problems || n_problems <= 0) return 0;
  for (int32_t i = 0; i < n_problems; ++i) {
    // a shape the batched call rejects has no workspace size (the pointers
    // may still be unset when the size is asked for)
    const qmuon_ns_problem& p = problems[i];
    if (p.rows <= 0 || p.cols <= 0 || p.rows > (1 << 30) || p.cols > (1 << 30) || p.ld < p.cols || p.ld % 8 ||
        p.cols % 8 || (p.input != QMUON_NS_BF16 && p.input != QMUON_NS_MXFP8) ||
        (p.input == QMUON_NS_MXFP8 && p.cols % 32))
      return 0;
  }
  return kWsHeader + ns::batch_workspace_bytes(problems, n_problems);
}

extern "C" qmuon_status qmuon_newton_schulz_batched(const qmuon_ns_problem* problems, int32_t n_problems,
                                                    int32_t iters, const float coeffs[3], void* ws,
                                                    size_t ws_bytes, void* stream) {
  qm::NvtxRange nvtx_range("qmuon_newton_schulz_batched");
  return qm::no_throw("qmuon_newton_schulz_batched", [&]() -> qmuon_status {
    if (!problems || n_problems <= 0 || iters < 1 || !coeffs || !ws) return QMUON_ERR_INVALID_ARGUMENT;
    if (!aligned(ws, 256)) return QMUON_ERR_INVALID_ARGUMENT;
    for (int32_t i = 0; i < n_problems; ++i) {
      const qmuon_status s = ns::validate_problem(problems[i]);
      if (s != QMUON_OK) return s;
    }
    if (ws_bytes < kWsHeader + ns::batch_workspace_bytes(problems, n_problems))
      return QMUON_ERR_WORKSPACE_TOO_SMALL;
    unsigned char* b = static_cast<unsigned char*>(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t me = cudaMemsetAsync(b, 0, kWsHeader, s);
    if (me != cudaSuccess) return set_error("qmuon_newton_schulz_batched (memset)", me);
    const qmuon_status rs = ns::run_batch(problems, n_problems, iters, coeffs, reinterpret_cast<WsHeader*>(b),
                                          b + kWsHeader, ws_bytes - kWsHeader, s);
    if (rs != QMUON_OK) return rs;
    tally(T_NS_CALLS);
    for (int32_t i = 0; i < n_problems; ++i) {
      const qmuon_ns_problem& p = problems[i];
      if (p.input == QMUON_NS_MXFP8) {
        tally(T_NS_MXFP8_PROBLEMS);
        tally(T_NS_BF16_HANDOFF_BYTES, (uint64_t)p.rows * (uint64_t)p.cols * 2u);
      } else {
        tally(T_NS_BF16_PROBLEMS);
      }
    }
    return QMUON_OK;
  });
}

extern "C" qmuon_status qmuon_step(const qmuon_plan* plan, int64_t t, int32_t P, float beta,
                                   float eta_full, float eta_block, float* const* weights,
                                   const float coeffs[3], int32_t iters, float* group_sumsq, void* ws,
                                   size_t ws_bytes, void* stream) {
  qm::NvtxRange nvtx_range("qmuon_step");
  return qm::no_throw("qmuon_step", [&]() -> qmuon_status {
    if (!plan || !weights || !coeffs || !ws || t < 1 || P < 0 || iters < 1) return QMUON_ERR_INVALID_ARGUMENT;
    if (!aligned(ws, 256)) return QMUON_ERR_INVALID_ARGUMENT;
    if (plan->dt != QMUON_BF16) return QMUON_ERR_UNSUPPORTED;
    const int32_t n = (int32_t)plan->tensors.size();
    for (int32_t i = 0; i < n; ++i) {
      const qmuon_tensor& T = plan->tensors[i];
      if (T.rows * T.cols == 0) continue;
      if (!weights[i] || !aligned(weights[i], 16)) return QMUON_ERR_INVALID_ARGUMENT;
      if (T.cols % 8) return QMUON_ERR_UNSUPPORTED;
    }
    if (ws_bytes < qmuon_workspace_size(plan, QMUON_WS_STEP)) return QMUON_ERR_WORKSPACE_TOO_SMALL;
    const bool full = (P != 0) && (t % P == 0);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const UpdWs w = carve(plan, ws, ws_bytes);
    qmuon_plan* mp = const_cast<qmuon_plan*>(plan);
    ns::StepTables*& tabs = full ? mp->ns_full : mp->ns_block;
    const qmuon_status ts = ns::ensure_step_tables(&tabs, plan->tensors.data(), n, full ? 1 : plan->tile_r,
                                                   full ? 1 : plan->tile_c, weights, w.inv, w.ns, w.ns_bytes,
                                                   true, s);
    if (ts != QMUON_OK) return ts;
    UpdLaunch L = make_launch(plan, full ? 1 : 2, beta, w, group_sumsq ? group_sumsq : w.sumsq, w.inv);
    set_sr(L, plan->sr, plan->sr_seed, t);
    cudaError_t e = cudaMemsetAsync(w.header, 0, kWsHeader, s);
    if (e == cudaSuccess) e = launch_update(L, plan->q8, plan->dt, false, s);
    if (e != cudaSuccess) return set_error("qmuon_step (update launch)", e);
    const qmuon_status rs = ns::run_step(tabs, iters, coeffs, full ? eta_full : eta_block, w.header, s);
    if (rs != QMUON_OK) return rs;
    const uint64_t k = nonempty_tensors(plan);
    tally(full ? T_STEP_FULL_CALLS : T_STEP_BLOCK_CALLS);
    if (plan->sr) tally(T_STEP_SR_CALLS);
    tally_grad_state(plan->dt, plan->q8, k);
    tally(T_NS_BF16_PROBLEMS, full ? k : k * (uint64_t)plan->tile_r * (uint64_t)plan->tile_c);
    tally(T_WEIGHT_F32, k);
    return QMUON_OK;
  });
}

extern "C" qmuon_status qmuon_step_from_host(const qmuon_plan* plan, int64_t t, int32_t P, float beta,
                                             float eta_full, float eta_block, float* const* weights,
                                             const float coeffs[3], int32_t iters,
                                             const void* const* host_grads, float* host_group_sumsq,
                                             float* group_sumsq, void* ws, size_t ws_bytes, void* stream,
                                             void* copy_stream) {
  qm::NvtxRange nvtx_range("qmuon_step_from_host");
  if (!plan || !host_grads) return QMUON_ERR_INVALID_ARGUMENT;
  if (plan->dt != QMUON_BF16) return QMUON_ERR_UNSUPPORTED;
  const int32_t n = (int32_t)plan->tensors.size();
  for (int32_t i = 0; i < n; ++i)
    if (plan->tensors[i].rows * plan->tensors[i].cols != 0 && !host_grads[i]) return QMUON_ERR_INVALID_ARGUMENT;
  qmuon_plan* mp = const_cast<qmuon_plan*>(plan);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStream_t cs = copy_stream ? static_cast<cudaStream_t>(copy_stream) : s;
  cudaError_t e = cudaSuccess;
  if (!mp->grads_free) e = cudaEventCreateWithFlags(&mp->grads_free, cudaEventDisableTiming);
  if (e == cudaSuccess && !mp->grads_copied) e = cudaEventCreateWithFlags(&mp->grads_copied, cudaEventDisableTiming);
  if (e != cudaSuccess) return set_error("qmuon_step_from_host (event create)", e);
  // the buffers are free once this plan's previous step has finished with them
  if (cs != s && mp->grads_free_recorded) e = cudaStreamWaitEvent(cs, mp->grads_free, 0);
  // page-locked, device-addressable, 16-byte aligned whole-vector buffers are
  // pulled by one kernel launch per kPullMax tensors; anything else is copied
  const int sms = plan->host_ingest == QMUON_INGEST_PULL ? sm_count_of_current_device() : 0;
  HostPull pull{};
  uint64_t pulled = 0, copied = 0;
  auto flush = [&]() -> cudaError_t {
    if (pull.n == 0) return cudaSuccess;
    host_pull_kernel<<<(unsigned)((sms + 7) / 8), 256, 0, cs>>>(pull);
    pull.n = 0;
    return cudaGetLastError();
  };
  for (int32_t i = 0; i < n && e == cudaSuccess; ++i) {
    const qmuon_tensor& T = plan->tensors[i];
    const size_t bytes = (size_t)(T.rows * T.cols) * sizeof(uint16_t);
    if (!bytes) continue;
    const void* dv = (sms > 0 && bytes % 16 == 0 && aligned(T.grad, 16)) ? device_view_of_host(host_grads[i]) : nullptr;
    if (dv && aligned(dv, 16)) {
      pull.src[pull.n] = static_cast<const uint4*>(dv);
      pull.dst[pull.n] = static_cast<uint4*>(T.grad);
      pull.n16[pull.n] = bytes / 16;
      ++pull.n;
      pulled += bytes;
      if (pull.n == kPullMax) e = flush();
    } else {
      e = cudaMemcpyAsync(T.grad, host_grads[i], bytes, cudaMemcpyHostToDevice, cs);
      copied += bytes;
    }
  }
  if (e == cudaSuccess) e = flush();
  if (e == cudaSuccess && cs != s) {
    e = cudaEventRecord(mp->grads_copied, cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, mp->grads_copied, 0);
  }
  if (e != cudaSuccess) return set_error("qmuon_step_from_host (gradient copies)", e);
  const qmuon_status st = qmuon_step(plan, t, P, beta, eta_full, eta_block, weights, coeffs, iters, group_sumsq,
                                     ws, ws_bytes, stream);
  if (st != QMUON_OK) return st;
  if (host_group_sumsq) {
    const bool full = (P != 0) && (t % P == 0);
    const int32_t ng = plan->layout[full ? 1 : 2].n_groups;
    const float* src = group_sumsq ? group_sumsq : carve(plan, ws, ws_bytes).sumsq;
    if (ng > 0) e = cudaMemcpyAsync(host_group_sumsq, src, (size_t)ng * sizeof(float), cudaMemcpyDeviceToHost, s);
  }
  if (e == cudaSuccess) e = cudaEventRecord(mp->grads_free, s);
  if (e != cudaSuccess) return set_error("qmuon_step_from_host (read-back)", e);
  mp->grads_free_recorded = true;
  tally(T_STEP_HOST_FED_CALLS);
  tally(T_HOST_PULLED_BYTES, pulled);
  tally(T_HOST_COPIED_BYTES, copied);
  return QMUON_OK;
}

extern "C" qmuon_status qmuon_step_prepare(const qmuon_plan* plan, float* const* weights, void* ws,
                                           size_t ws_bytes) {
  qm::NvtxRange nvtx_range("qmuon_step_prepare");
  return qm::no_throw("qmuon_step_prepare", [&]() -> qmuon_status {
    if (!plan || !weights || !ws || !aligned(ws, 256)) return QMUON_ERR_INVALID_ARGUMENT;
    if (plan->dt != QMUON_BF16) return QMUON_ERR_UNSUPPORTED;
    const int32_t n = (int32_t)plan->tensors.size();
    for (int32_t i = 0; i < n; ++i) {
      const qmuon_tensor& T = plan->tensors[i];
      if (T.rows * T.cols == 0) continue;
      if (!weights[i] || !aligned(weights[i], 16)) return QMUON_ERR_INVALID_ARGUMENT;
      if (T.cols % 8) return QMUON_ERR_UNSUPPORTED;
    }
    if (ws_bytes < qmuon_workspace_size(plan, QMUON_WS_STEP)) return QMUON_ERR_WORKSPACE_TOO_SMALL;
    const UpdWs w = carve(plan, ws, ws_bytes);
    qmuon_plan* mp = const_cast<qmuon_plan*>(plan);
    qmuon_status st = ns::ensure_step_tables(&mp->ns_full, plan->tensors.data(), n, 1, 1, weights, w.inv, w.ns,
                                             w.ns_bytes, false, nullptr);
    if (st != QMUON_OK) return st;
    return ns::ensure_step_tables(&mp->ns_block, plan->tensors.data(), n, plan->tile_r, plan->tile_c, weights, w.inv,
                                  w.ns, w.ns_bytes, false, nullptr);
  });
}

extern "C" qmuon_status qmuon_sync_status(void* ws, void* stream) {
  if (!ws || !aligned(ws, 256)) return QMUON_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return set_error("qmuon_sync_status (stream synchronize)", e);
  unsigned int err[2] = {0u, 0u};
  e = cudaMemcpy(err, ws, sizeof(err), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return set_error("qmuon_sync_status (read header)", e);
  if (err[0] != 0) {
    const unsigned int zero[2] = {0u, 0u};
    cudaMemcpy(ws, zero, sizeof(zero), cudaMemcpyHostToDevice);
    char msg[128];
    std::snprintf(msg, sizeof(msg), "kernel reported status %u at site 0x%x", err[0], err[1]);
    return set_error_msg(msg, (qmuon_status)err[0]);
  }
  return QMUON_OK;
}

extern "C" const char* qmuon_status_string(qmuon_status status) {
  switch (status) {
    case QMUON_OK: return "ok";
    case QMUON_ERR_INVALID_ARGUMENT: return "invalid argument";
    case QMUON_ERR_MISALIGNED_SEGMENT: return "norm segment not aligned to 256-element blocks";
    case QMUON_ERR_UNSUPPORTED: return "unsupported request";
    case QMUON_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case QMUON_ERR_CUDA: return "CUDA error";
    case QMUON_ERR_TIMEOUT: return "a kernel's bounded wait expired";
    case QMUON_ERR_OUT_OF_MEMORY: return "host memory allocation failed";
  }
  return "unknown status";
}

extern "C" const char* qmuon_version(void) { return "qmuon 0.1 sm_103a"; }

extern "C" const char* qmuon_last_error(void) { return g_last_error; }

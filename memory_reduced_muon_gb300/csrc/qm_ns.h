// Newton-Schulz engine internals (ns_gemm.cu), used by api.cu.
#pragma once

#include "qm_internal.h"

namespace qm {
namespace ns {

struct StepTables;  // device problem table of qmuon_step (full or block steps)

qmuon_status validate_problem(const qmuon_ns_problem& p);
size_t batch_workspace_bytes(const qmuon_ns_problem* probs, int32_t n);
qmuon_status run_batch(const qmuon_ns_problem* probs, int32_t n, int32_t iters, const float coeffs[3],
                       WsHeader* hdr, unsigned char* ws, size_t ws_bytes, cudaStream_t s);

size_t step_workspace_bytes(const qmuon_tensor* t, int32_t n, int32_t tile_r, int32_t tile_c);
// Builds (or keeps) the tables of one step kind.  A rebuild uploads them in
// the order of `s` when `ordered` (after the steps already enqueued there,
// which may still read the old tables); otherwise it waits for the device to
// finish every earlier launch and uploads them synchronously.
qmuon_status ensure_step_tables(StepTables** tabs, const qmuon_tensor* t, int32_t n, int32_t tile_r,
                                int32_t tile_c, float* const* weights, const float* inv,
                                unsigned char* ws, size_t ws_bytes, bool ordered, cudaStream_t s);
qmuon_status run_step(StepTables* tabs, int32_t iters, const float coeffs[3], float eta, WsHeader* hdr,
                      cudaStream_t s);
void destroy_step_tables(StepTables* t);

}  // namespace ns
}  // namespace qm

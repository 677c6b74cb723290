// 4-bit GRASP momentum state for sm_103a (qmuon_grasp_step).
//
// Implements the update of "4-bit-Muon-GRASP" (the page's equations): the
// momentum of every matrix is held as a rank-8 factor P R^T (8-bit) plus a
// residual (4-bit), each grid-quantised in 64 x 64 blocks (an entry is scaled
// by the smaller of its row and column maxima inside its block).  One step:
//   M_{t-1} = res + P R^T,  M_t = mu M_{t-1} + g_t  (stored in bf16 over g_t)
//   Q = ColNorm(R_{t-1}),  P_t = orth(M_t Q),  R_t = M_t^T P_t
//   res_t = M_t - P_t R_t^T,  then res_t, P_t, R_t are grid-quantised.
// The reconstruction and the momentum are computed in fp32 with one rounding
// per operation in a fixed order (the sum over the rank runs left to right);
// the power iteration accumulates in fp32, and orth is CholeskyQR2 in fp64
// (the orthonormal factor whose triangular factor has a positive diagonal).
// All matrices of a call share each launch:
//   grasp_colnorm   per matrix:     dequantised R and its column norms
//   grasp_pass1     per row strip:  reconstruct, momentum, store M_t,
//                                   Y = M_t Q = (M_t R_{t-1}) diag(1 / norms),
//                                   the strip's share of Y^T Y
//   grasp_chol      per matrix:     the Gram from the strips' shares, its Cholesky L
//   grasp_tsolve    per row strip:  rows times L^{-T}; first pass: P1 and its
//                                   shares of P1^T P1; second pass: P, quantised
//   grasp_pass2     per col strip:  R = M_t^T P, quantised
//   grasp_pass3     per tile:       residual, its 4-bit grid codes and maxima
// A strip (64 rows or 64 columns of one matrix) is one CTA's whole sum, so
// there are no partial sums and no atomics on results: they are deterministic.
// Grid steps use fl(min(r, c) / L) = min(fl(r / L), fl(c / L)) (division is
// monotonic), so divisions run per row and per column, not per entry.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstddef>
#include <cstring>
#include <type_traits>
#include <vector>

#include "qm_internal.h"

namespace qm {
namespace {

constexpr int kRank = QMUON_GRASP_RANK;   // 8
constexpr int kS = QMUON_GRASP_BLOCK;     // 64
constexpr int kThreads = 256;
constexpr int kNormCols = 1024;   // columns of R_{t-1} per CTA of the column-norm pass

// Device copy of one matrix's description plus its workspace slices.
struct GraspProb {
  qmuon_grasp_matrix m;
  int64_t nbr, nbc;          // row / column blocks
  int64_t ncc;               // chunks of kNormCols columns
  double* qpart;             // [ncc][8]    each chunk's sums of r_jl^2 (R_{t-1}); Q = R_{t-1} diag(1 / norms)
  float* rdeq;               // [cols][8]   R_{t-1} dequantised
  float* y;                  // [rows][8]   M_t Q
  float* p;                  // [rows][8]   P_t
  float* r;                  // [cols][8]   R_t
  double* p1;                // [rows][8]   first CholeskyQR pass: Y L1^{-T}
  double* gpart;             // [nbr][36]   each row strip's share of the Gram (lower triangle)
  double* L;                 // [8][8]      Cholesky factor of the current pass
};

struct GraspArgs {
  const GraspProb* probs;
  const int64_t* tile_start;  // [n + 1] prefix of pass 3's chunks (64 rows x 4 column blocks)
  const int64_t* rstrip_start;  // [n + 1] prefix of 64-row strips, problems in rorder
  const int64_t* cstrip_start;  // [n + 1] prefix of 64-column strips, problems in corder
  // The order in which the grid deals each kind of strip: longest first (a
  // row strip's length is its matrix's column count, a column strip's its row
  // count), so that the longest strips do not start last and run alone
  const int32_t* rorder;        // [n] problem at each position of the row-strip order
  const int32_t* corder;        // [n] problem at each position of the column-strip order
  int32_t n;
  float mu;
};

__device__ __forceinline__ int find_prob(const int64_t* start, int n, int64_t idx) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(start + mid) <= idx) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Grid dequantisation step of an entry: fl(min(rmax, cmax) / L).
__device__ __forceinline__ float grid_step(float rmax, float cmax, float L) {
  return __fdiv_rn(fminf(rmax, cmax), L);
}
// Grid quantisation factor fl(L / min(r, c)) = max(fl(L / r), fl(L / c)) for
// positive maxima (division is monotonic); 0 where a maximum is 0.
__device__ __forceinline__ float grid_factor(float inv_r, float inv_c) { return fmaxf(inv_r, inv_c); }
__device__ __forceinline__ float inv_level(float mx, float L) { return mx == 0.0f ? 0.0f : __fdiv_rn(L, mx); }
__device__ __forceinline__ int grid_code(float x, float sc, int L) {
  if (sc == 0.0f) return 0;
  const int q = __float2int_rn(__fmul_rn(x, sc));   // NaN converts to 0
  return q < -L ? -L : (q > L ? L : q);
}

// Two fp32 fused multiply-adds in one packed instruction, d = a * b + c per
// component, each rounded once exactly as fmaf rounds it.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n\t.reg .b64 pa, pb, pc, pd;\n\tmov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
      "mov.b64 pc, {%6, %7};\n\tfma.rn.f32x2 pd, pa, pb, pc;\n\tmov.b64 {%0, %1}, pd;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}

__device__ __forceinline__ float2 add2_rn(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 pa, pb, pd;\n\tmov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
      "add.rn.f32x2 pd, pa, pb;\n\tmov.b64 {%0, %1}, pd;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
// A packed multiply, each half rounded as __fmul_rn rounds it.  Its results
// feed scalar additions only: ptxas fuses a packed multiply whose single use
// is a packed addition into a packed FMA, which would round once instead of twice.
__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 pa, pb, pd;\n\tmov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
      "mul.rn.f32x2 pd, pa, pb;\n\tmov.b64 {%0, %1}, pd;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 sub2_rn(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 pa, pb, pd;\n\tmov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
      "sub.rn.f32x2 pd, pa, pb;\n\tmov.b64 {%0, %1}, pd;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
// Compensated (Neumaier) addition of a block's sum into a running total, on
// two independent sums at once: the strips add up to 224 blocks, and the
// orthogonalisation magnifies the error of Y when its columns are nearly
// parallel.  Knuth's TwoSum (additions and subtractions only, so no packed
// multiply can be fused into them) gives the exact rounding error of each
// addition, the same value as the magnitude-ordered Fast2Sum.
__device__ __forceinline__ void two_sum_add2(float2& sum, float2& comp, float2 v) {
  const float2 t = add2_rn(sum, v);
  const float2 bv = sub2_rn(t, sum);
  comp = add2_rn(comp, add2_rn(sub2_rn(sum, sub2_rn(t, bv)), sub2_rn(v, bv)));
  sum = t;
}

// Sum over the CTA of 8 fp64 values per thread, in a fixed order.
__device__ __forceinline__ void block_sum8(double (&v)[kRank], double* red /* [8 warps][8] */) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < kRank; ++c)
    for (int o = 16; o > 0; o >>= 1) v[c] += __shfl_xor_sync(0xffffffffu, v[c], o);
  __syncthreads();
  if (l == 0)
#pragma unroll
    for (int c = 0; c < kRank; ++c) red[w * kRank + c] = v[c];
  __syncthreads();
#pragma unroll
  for (int c = 0; c < kRank; ++c) {
    double s = 0.0;
    for (int i = 0; i < kThreads / 32; ++i) s += red[i * kRank + c];
    v[c] = s;
  }
}

// Dequantised 8-bit factor row (P or R): codes q[row][8], per-row max, per
// (row block, column) max.
__device__ __forceinline__ void factor_row(const int8_t* q, const float* rmax, const float* cmax, int64_t row,
                                           float (&out)[kRank]) {
  const float rm = __ldg(rmax + row);
  const float* cm = cmax + (row / kS) * kRank;
  const int2 raw = __ldg(reinterpret_cast<const int2*>(q + row * kRank));
  const int8_t* b = reinterpret_cast<const int8_t*>(&raw);
#pragma unroll
  for (int l = 0; l < kRank; ++l) out[l] = __fmul_rn((float)b[l], grid_step(rm, __ldg(cm + l), 127.0f));
}

// The step's kernels are launched as programmatic dependents of one another
// (launch_dep below): each first waits until every earlier grid of the stream
// has completed and its writes are visible, then lets the next kernel be
// scheduled, so that its launch overlaps this one's last wave.
__device__ __forceinline__ void grid_dep_sync() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// R_{t-1} dequantised and the inverse norms of its columns, one CTA per matrix
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) grasp_colnorm(GraspArgs a) {
  grid_dep_sync();
  __shared__ double red[kThreads / 32 * kRank];
  // CTA (c, k): matrix k's columns c * kNormCols .. + kNormCols
  const GraspProb& P = a.probs[blockIdx.y];
  if ((int64_t)blockIdx.x >= P.ncc) return;
  const int64_t cols = P.m.cols;
  const int64_t j0 = (int64_t)blockIdx.x * kNormCols;
  const int64_t j1 = cols < j0 + kNormCols ? cols : j0 + kNormCols;
  double ss[kRank] = {0, 0, 0, 0, 0, 0, 0, 0};
  // unrolled so that several rows' loads are in flight at once; the sums
  // still run over j in order
#pragma unroll 4
  for (int64_t j = j0 + threadIdx.x; j < j1; j += kThreads) {
    float r[kRank];
    factor_row(P.m.r, P.m.r_rmax, P.m.r_cmax, j, r);
    float4* dst = reinterpret_cast<float4*>(P.rdeq + j * kRank);
    dst[0] = make_float4(r[0], r[1], r[2], r[3]);
    dst[1] = make_float4(r[4], r[5], r[6], r[7]);
#pragma unroll
    for (int l = 0; l < kRank; ++l) ss[l] += (double)r[l] * (double)r[l];
  }
  block_sum8(ss, red);
  if (threadIdx.x < kRank) P.qpart[blockIdx.x * kRank + threadIdx.x] = ss[threadIdx.x];
}

// The CTA's share of Z^T Z in fp64 (36 lower-triangle entries, row-major
// (u, v <= u)): the rows are held by the lanes with `mine` set, every `stride`
// lanes apart; butterfly sums inside each warp, then the warps in order.
// Written to out[0..35].  Every thread of the CTA calls it.
__device__ __forceinline__ void gram_share(const double (&z)[kRank], bool mine, int stride, double (*red)[36],
                                           double* out) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  int k = 0;
#pragma unroll
  for (int u = 0; u < kRank; ++u)
#pragma unroll
    for (int v = 0; v <= u; ++v, ++k) {
      double g = mine ? z[u] * z[v] : 0.0;
      for (int o = stride; o < 32; o <<= 1) g += __shfl_xor_sync(0xffffffffu, g, o);
      if (l == 0) red[w][k] = g;
    }
  __syncthreads();
  if (threadIdx.x < 36) {
    double s = 0.0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += red[i][threadIdx.x];
    out[threadIdx.x] = s;
  }
}

// Grid quantisation of one 64-row block of an 8-column factor held in shared
// memory (x[row][8], rows r0 .. r0 + nvalid - 1 of the factor): codes, per-row
// maxima and the block's per-column maxima.  Every thread of the CTA calls it.
__device__ __forceinline__ void quantize_block8(const float (*x)[kRank], int nvalid, int64_t r0, int8_t* q,
                                                float* rmax, float* cmax_blk) {
  __shared__ float cm[kRank];
  if (threadIdx.x < kRank) {
    float m = 0.0f;
    for (int r = 0; r < nvalid; ++r) m = fmaxf(m, fabsf(x[r][threadIdx.x]));
    cm[threadIdx.x] = m;
    cmax_blk[threadIdx.x] = m;
  }
  __syncthreads();
  if ((int)threadIdx.x < nvalid) {
    const int r = threadIdx.x;
    float rm = 0.0f;
#pragma unroll
    for (int l = 0; l < kRank; ++l) rm = fmaxf(rm, fabsf(x[r][l]));
    rmax[r0 + r] = rm;
    const float ir = inv_level(rm, 127.0f);
    int8_t c[kRank];
#pragma unroll
    for (int l = 0; l < kRank; ++l) c[l] = (int8_t)grid_code(x[r][l], grid_factor(ir, inv_level(cm[l], 127.0f)), 127);
    *reinterpret_cast<int2*>(q + (r0 + r) * kRank) = *reinterpret_cast<const int2*>(c);
  }
}

// 16- and 8-byte asynchronous global -> shared copies; an invalid one
// writes zeros (source size 0) and reads nothing.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src, bool valid) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(d), "l"(src), "r"(valid ? 8 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// ---------------------------------------------------------------------------
// pass 1: one CTA per 64-row strip of a matrix, walking its column blocks in
// chunks of two (128 columns).  Each chunk's gradient tile, residual codes and
// dequantised R rows arrive in shared memory by asynchronous copies through a
// two-stage ring, one chunk ahead of the arithmetic; the rows' residual
// maxima and the columns' residual steps come by plain loads one chunk ahead
// too.  With nothing held in registers between chunks, three CTAs fit on an
// SM.  Thread t owns row t/4 of the strip and 16 consecutive columns
// (t % 4) * 16 of each block; Y for the strip's rows is complete when the
// walk ends.
// ---------------------------------------------------------------------------
constexpr int kChunk = 4;   // column blocks per chunk of pass 3
constexpr int kC1 = 2;      // column blocks per chunk of pass 1

// Shared rows of 8 floats for a chunk's columns.  The four 16-column groups a
// warp reads at once sit 16 * 8 = 128 floats apart, one bank apart modulo 32:
// each group of 16 columns is shifted by 4 more floats so that their float4
// reads fall in different banks.
__device__ __forceinline__ int sidx(int col, int l) { return col * kRank + (col >> 4) * 4 + l; }

// One stage of pass 1's ring.  Row strides are padded so that the rows a warp
// reads at once fall in different banks: 272 bytes for the gradient (8 rows x
// 4 column groups of 16 bf16 read as 16-byte halves), 96 bytes for the codes
// (4 rows x 4 groups of 8 bytes per half-warp).
constexpr int kP1GStride = kC1 * kS * 2 + 16;                  // bytes per gradient row
constexpr int kP1CStride = kC1 * kS / 2 + 32;                  // bytes per code row
constexpr int kP1RFloats = kC1 * kS * kRank + (kC1 * kS / 16) * 4;
struct P1Stage {
  unsigned char g[kS * kP1GStride];
  unsigned char codes[kS * kP1CStride];
  float r[kP1RFloats];
  float step_c[kC1 * kS];                                      // fl(cmax_j / 7) of the residual
};
static_assert(sizeof(P1Stage) % 16 == 0 && offsetof(P1Stage, codes) % 16 == 0 && offsetof(P1Stage, r) % 16 == 0,
              "pass 1 stage fields must stay 16-byte aligned");
constexpr int kP1Smem = 2 * (int)sizeof(P1Stage);

__global__ void __launch_bounds__(kThreads, 2) grasp_pass1(GraspArgs a) {
  grid_dep_sync();
  extern __shared__ __align__(16) unsigned char p1smem[];
  P1Stage* stage = reinterpret_cast<P1Stage*>(p1smem);
  const int pk = find_prob(a.rstrip_start, a.n, blockIdx.x);
  const GraspProb& P = a.probs[__ldg(a.rorder + pk)];
  const int64_t bi = blockIdx.x - __ldg(a.rstrip_start + pk);
  const int64_t rows = P.m.rows, cols = P.m.cols;
  const int t = threadIdx.x;
  const int ti = t >> 2, tj = (t & 3) * 16;
  const int64_t i = bi * kS + ti;
  const bool live = i < rows;
  const __nv_bfloat16* grad = static_cast<const __nv_bfloat16*>(P.m.grad);
  const int64_t nch = (P.nbc + kC1 - 1) / kC1;

  // chunk k's copies into stage k & 1 (NB blocks, a compile-time count so
  // the index arithmetic is shifts and masks): rows past the matrix read as zeros
  auto issue_nb = [&](auto nb_c, int64_t k) {
    constexpr int NB = decltype(nb_c)::value;
    P1Stage& st = stage[k & 1];
    const int64_t j0 = k * kC1 * kS;
    // gradient: 64 rows x NB * 8 segments of 16 bytes
#pragma unroll 1
    for (int q = 0; q < kS * NB * 8 / kThreads; ++q) {
      const int e = t + q * kThreads;
      const int row = e / (NB * 8), seg = e % (NB * 8);
      const bool ok = bi * kS + row < rows;
      cp_async16(st.g + row * kP1GStride + seg * 16, grad + (ok ? (bi * kS + row) * cols + j0 + seg * 8 : 0), ok);
    }
    // codes: 64 rows x NB * 4 pieces of 8 bytes (the code array is 8-byte aligned)
#pragma unroll 1
    for (int q = 0; q < kS * NB * 4 / kThreads; ++q) {
      const int e = t + q * kThreads;
      const int row = e / (NB * 4), seg = e % (NB * 4);
      const bool ok = bi * kS + row < rows;
      cp_async8(st.codes + row * kP1CStride + seg * 8,
                P.m.res + (ok ? (bi * kS + row) * (cols / 2) + j0 / 2 + seg * 8 : 0), ok);
    }
    // dequantised R rows of the chunk's columns: NB * 64 rows of 8 floats, in halves
    if (t < NB * kS * 2)
      cp_async16(&st.r[sidx(t >> 1, (t & 1) * 4)], P.rdeq + (j0 + (t >> 1)) * kRank + (t & 1) * 4, true);
  };
  auto issue = [&](int64_t k) {
    if (P.nbc - k * kC1 >= kC1) issue_nb(std::integral_constant<int, kC1>{}, k);
    else issue_nb(std::integral_constant<int, 1>{}, k);
  };
  static_assert(kC1 == 2 && kS * 4 % kThreads == 0 && kS * 2 * 2 <= kThreads,
                "pass 1's copy loops assume two-block chunks of 64 x 64 blocks and 256 threads");
  // chunk k's residual maxima of this thread's row, and of column t (plain loads)
  float rmax_next[kC1], cmax_next;
  auto fetch = [&](int64_t k) {
    const int64_t b0 = k * kC1;
    const int nb = (P.nbc - b0) < kC1 ? (int)(P.nbc - b0) : kC1;
#pragma unroll
    for (int c = 0; c < kC1; ++c) rmax_next[c] = (live && c < nb) ? __ldg(P.m.res_rmax + (b0 + c) * rows + i) : 0.0f;
    cmax_next = (t < nb * kS) ? __ldg(P.m.res_cmax + bi * cols + b0 * kS + t) : 0.0f;
  };

  float p[kRank];
  if (live) factor_row(P.m.p, P.m.p_rmax, P.m.p_cmax, i, p);
  float2 pp[kRank / 2];
#pragma unroll
  for (int l2 = 0; l2 < kRank / 2; ++l2) pp[l2] = make_float2(p[2 * l2], p[2 * l2 + 1]);
  float2 y2[kRank / 2], yc2[kRank / 2];
#pragma unroll
  for (int l2 = 0; l2 < kRank / 2; ++l2) y2[l2] = yc2[l2] = make_float2(0.0f, 0.0f);
  issue(0);
  cp_async_commit();
  fetch(0);
  for (int64_t k = 0; k < nch; ++k) {
    P1Stage& st = stage[k & 1];
    const int64_t b0 = k * kC1;
    const int nb = (P.nbc - b0) < kC1 ? (int)(P.nbc - b0) : kC1;
    // this chunk's column steps (its stage was last read two chunks ago,
    // before the barrier that ended that chunk) and row maxima
    if (t < nb * kS) st.step_c[t] = __fdiv_rn(cmax_next, 7.0f);
    float rmax[kC1];
#pragma unroll
    for (int c = 0; c < kC1; ++c) rmax[c] = rmax_next[c];
    if (k + 1 < nch) {
      issue(k + 1);   // into the other stage, free since the last chunk's closing barrier
      fetch(k + 1);
    }
    cp_async_commit();
    cp_async_wait<1>();   // chunk k's copies of this thread have landed
    __syncthreads();      // ... and every thread's, with the column steps
    if (live) {
#pragma unroll
      for (int c = 0; c < kC1; ++c) {
        if (c >= nb) break;
        const int64_t bj = b0 + c;
        const float step_r = __fdiv_rn(rmax[c], 7.0f);
        const int cb = c * kS + tj;   // column of the chunk
        const uint4 g0 = *reinterpret_cast<const uint4*>(st.g + ti * kP1GStride + cb * 2);
        const uint4 g1 = *reinterpret_cast<const uint4*>(st.g + ti * kP1GStride + cb * 2 + 16);
        const uint2 cwv = *reinterpret_cast<const uint2*>(st.codes + ti * kP1CStride + cb / 2);
        const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        // the residual codes as bytes: even elements' nibbles in lo, odd ones' in hi
        const uint32_t lo[2] = {cwv.x & 0x0F0F0F0Fu, cwv.y & 0x0F0F0F0Fu};
        const uint32_t hi[2] = {(cwv.x >> 4) & 0x0F0F0F0Fu, (cwv.y >> 4) & 0x0F0F0F0Fu};
        uint32_t out[8];
        float2 yb[kRank / 2];
#pragma unroll
        for (int l2 = 0; l2 < kRank / 2; ++l2) yb[l2] = make_float2(0.0f, 0.0f);
        // four elements at a time with the rank loop outside, so that four
        // independent reconstruction chains interleave; every sum keeps its
        // order (each element's over l, each Y sum's over the elements).  The
        // products of ranks l and l + 1 are one packed multiply, each half
        // rounded as fmul rounds it, and feed the scalar additions in order.
#pragma unroll
        for (int e0 = 0; e0 < 16; e0 += 4) {
          float2 rr[4][kRank / 2];
          float acc[4], m[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 r0 = *reinterpret_cast<const float4*>(&st.r[sidx(cb + e0 + j, 0)]);
            const float4 r1 = *reinterpret_cast<const float4*>(&st.r[sidx(cb + e0 + j, 4)]);
            rr[j][0] = make_float2(r0.x, r0.y);
            rr[j][1] = make_float2(r0.z, r0.w);
            rr[j][2] = make_float2(r1.x, r1.y);
            rr[j][3] = make_float2(r1.z, r1.w);
            acc[j] = 0.0f;
          }
#pragma unroll
          for (int l2 = 0; l2 < kRank / 2; ++l2)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 pr = mul2_rn(pp[l2], rr[j][l2]);
              acc[j] = __fadd_rn(__fadd_rn(acc[j], pr.x), pr.y);
            }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int e = e0 + j;
            // 2^23 + nibble, exactly, then the code's offset of 8 taken off (exact)
            const uint32_t src = (e & 1) ? hi[e >> 3] : lo[e >> 3];
            const float nib = __fsub_rn(__uint_as_float(__byte_perm(src, 0x4B000000u, 0x7650u | ((e & 7) >> 1))),
                                        8388616.0f);
            const float res = __fmul_rn(nib, fminf(step_r, st.step_c[cb + e]));
            const float mprev = __fadd_rn(res, acc[j]);
            const float g = __uint_as_float((e & 1) ? (gw[e >> 1] & 0xFFFF0000u) : (gw[e >> 1] << 16));
            m[j] = __fadd_rn(__fmul_rn(a.mu, mprev), g);
          }
          // M_t rounded to bf16 two elements at a time; Y takes the rounded values
          float mv[4];
#pragma unroll
          for (int jp = 0; jp < 2; ++jp) {
            const __nv_bfloat162 mb = __floats2bfloat162_rn(m[2 * jp], m[2 * jp + 1]);
            const uint32_t w = *reinterpret_cast<const uint32_t*>(&mb);
            out[(e0 >> 1) + jp] = w;
            mv[2 * jp] = __uint_as_float(w << 16);
            mv[2 * jp + 1] = __uint_as_float(w & 0xFFFF0000u);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int l2 = 0; l2 < kRank / 2; ++l2) yb[l2] = fma2(make_float2(mv[j], mv[j]), rr[j][l2], yb[l2]);
        }
#pragma unroll
        for (int l2 = 0; l2 < kRank / 2; ++l2) two_sum_add2(y2[l2], yc2[l2], yb[l2]);
        // M_t over the gradient (this chunk's gradient is already in shared memory)
        __nv_bfloat16* grow = static_cast<__nv_bfloat16*>(P.m.grad) + i * cols + bj * kS + tj;
        *reinterpret_cast<uint4*>(grow) = make_uint4(out[0], out[1], out[2], out[3]);
        *reinterpret_cast<uint4*>(grow + 8) = make_uint4(out[4], out[5], out[6], out[7]);
      }
    }
    __syncthreads();   // stage k & 1 is refilled by chunk k + 2's copies
  }
  cp_async_wait<0>();
  // 1 / (the column norms of R_{t-1}): the chunks' sums, added in chunk order
  __shared__ double s_qinv[kRank];
  if (t < kRank) {
    double v = 0.0;
    for (int64_t c = 0; c < P.ncc; ++c) v += __ldg(P.qpart + c * kRank + t);
    s_qinv[t] = v > 0.0 ? 1.0 / sqrt(v) : 0.0;
  }
  __syncthreads();
  float y[kRank];
#pragma unroll
  for (int l2 = 0; l2 < kRank / 2; ++l2) {
    y[2 * l2] = y2[l2].x + yc2[l2].x;
    y[2 * l2 + 1] = y2[l2].y + yc2[l2].y;
  }
  // the 4 threads of a row add their sums of M_t R_{t-1} (fixed order); the
  // column scaling of Q is applied once, in fp64
#pragma unroll
  for (int l = 0; l < kRank; ++l) {
    y[l] += __shfl_xor_sync(0xffffffffu, y[l], 1);
    y[l] += __shfl_xor_sync(0xffffffffu, y[l], 2);
    y[l] = (float)((double)y[l] * s_qinv[l]);
  }
  if ((t & 3) == 0 && live) {
    float4* dst = reinterpret_cast<float4*>(P.y + i * kRank);
    dst[0] = make_float4(y[0], y[1], y[2], y[3]);
    dst[1] = make_float4(y[4], y[5], y[6], y[7]);
  }
  // the strip's share of Y^T Y in fp64 (rows held by lanes 0, 4, ..., 28)
  __shared__ double red[kThreads / 32][36];
  double yd[kRank];
#pragma unroll
  for (int l = 0; l < kRank; ++l) yd[l] = live ? (double)y[l] : 0.0;
  gram_share(yd, (t & 3) == 0, 4, red, P.gpart + bi * 36);
}

// Cholesky of an 8 x 8 SPD matrix (lower factor, in place), one thread.
// Fully unrolled so that the matrix stays in registers; each column divides
// once (its diagonal's reciprocal, within one fp64 rounding of the quotients).
__device__ __forceinline__ bool chol8(double (&g)[kRank][kRank]) {
  bool ok = true;
#pragma unroll
  for (int j = 0; j < kRank; ++j) {
    double d = g[j][j];
#pragma unroll
    for (int k = 0; k < j; ++k) d -= g[j][k] * g[j][k];
    ok = ok && (d > 0.0);
    d = sqrt(ok ? d : 1.0);
    g[j][j] = d;
    const double inv = 1.0 / d;
#pragma unroll
    for (int i = j + 1; i < kRank; ++i) {
      double s = g[i][j];
#pragma unroll
      for (int k = 0; k < j; ++k) s -= g[i][k] * g[j][k];
      g[i][j] = s * inv;
    }
  }
  return ok;
}

// ---------------------------------------------------------------------------
// CholeskyQR2, in two passes of (grasp_chol, grasp_tsolve).  grasp_chol: the
// Gram as the sum of the row strips' shares (in strip order), its Cholesky
// factor L; one CTA per matrix.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(64) grasp_chol(GraspArgs a, WsHeader* hdr) {
  grid_dep_sync();
  __shared__ double sG[36];
  if (*reinterpret_cast<const volatile unsigned*>(&hdr->error) != 0u) return;
  const GraspProb& P = a.probs[blockIdx.x];
  if (threadIdx.x < 36) {
    double g = 0.0;
    for (int64_t b = 0; b < P.nbr; ++b) g += P.gpart[b * 36 + threadIdx.x];
    sG[threadIdx.x] = g;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double g[kRank][kRank];
#pragma unroll
    for (int u = 0; u < kRank; ++u)
#pragma unroll
      for (int v = 0; v < kRank; ++v) g[u][v] = (v <= u) ? sG[u * (u + 1) / 2 + v] : 0.0;
    if (!chol8(g)) {
      // rank-deficient M_t Q: no orthonormal factor
      if (atomicCAS(&hdr->error, 0u, (unsigned)QMUON_ERR_INVALID_ARGUMENT) == 0u) hdr->error_info = 0x2000u + blockIdx.x;
      return;
    }
#pragma unroll
    for (int u = 0; u < kRank; ++u)
#pragma unroll
      for (int v = 0; v < kRank; ++v) P.L[u * kRank + v] = g[u][v];
  }
}

// grasp_tsolve: one CTA per 64-row strip, one thread per row: z = L^{-1} x by
// forward substitution in fp64 (x the row of Y on the first pass, of P1 on the
// second).  First pass: z is P1's row, and the strip's share of P1^T P1 goes to
// the Gram shares.  Second pass: z rounded to fp32 is P's row, and the strip
// (one 64-row block of P) is grid-quantised.
template <int PASS>
__global__ void __launch_bounds__(64) grasp_tsolve(GraspArgs a, const WsHeader* hdr) {
  grid_dep_sync();
  __shared__ double sL[kRank][kRank];
  __shared__ double sInvD[kRank];         // 1 / L_uu
  __shared__ double sZZ[36][kS + 1];      // PASS 0: each row's products z_u z_v
  __shared__ float sx[kS][kRank];
  if (*reinterpret_cast<const volatile unsigned*>(&hdr->error) != 0u) return;
  const int pk = find_prob(a.rstrip_start, a.n, blockIdx.x);
  const GraspProb& P = a.probs[__ldg(a.rorder + pk)];
  const int64_t bi = blockIdx.x - __ldg(a.rstrip_start + pk);
  const int64_t rows = P.m.rows;
  sL[threadIdx.x >> 3][threadIdx.x & 7] = P.L[threadIdx.x];
  if (threadIdx.x < kRank) sInvD[threadIdx.x] = 1.0 / P.L[threadIdx.x * (kRank + 1)];
  __syncthreads();
  const int64_t i = bi * kS + threadIdx.x;
  const bool live = i < rows;
  // forward substitution; fp64 throughput is scarce here, so each row
  // multiplies by the diagonal's reciprocal (within one fp64 rounding of
  // the quotient) instead of dividing
  double z[kRank];
#pragma unroll
  for (int u = 0; u < kRank; ++u) {
    double s = 0.0;
    if (live) s = (PASS == 0) ? (double)P.y[i * kRank + u] : P.p1[i * kRank + u];
#pragma unroll
    for (int v = 0; v < u; ++v) s -= sL[u][v] * z[v];
    z[u] = live ? s * sInvD[u] : 0.0;
  }
  if (PASS == 0) {
    if (live)
#pragma unroll
      for (int l = 0; l < kRank; ++l) P.p1[i * kRank + l] = z[l];
    // the strip's share of Z^T Z: each row's 36 products, then one thread per
    // entry adds the 64 rows in order
    int k = 0;
#pragma unroll
    for (int u = 0; u < kRank; ++u)
#pragma unroll
      for (int v = 0; v <= u; ++v, ++k) sZZ[k][threadIdx.x] = z[u] * z[v];
    __syncthreads();
    if (threadIdx.x < 36) {
      double g = 0.0;
#pragma unroll 8
      for (int r = 0; r < kS; ++r) g += sZZ[threadIdx.x][r];
      P.gpart[bi * 36 + threadIdx.x] = g;
    }
  } else {
    const int nvalid = (rows - bi * kS) < kS ? (int)(rows - bi * kS) : kS;
    if (live) {
#pragma unroll
      for (int l = 0; l < kRank; ++l) {
        const float v = (float)z[l];
        P.p[i * kRank + l] = v;
        sx[threadIdx.x][l] = v;
      }
    }
    __syncthreads();
    quantize_block8(sx, nvalid, bi * kS, P.m.p, P.m.p_rmax, P.m.p_cmax + bi * kRank);
  }
}

// ---------------------------------------------------------------------------
// pass 2: R = M_t^T P, one CTA per 64-column strip of a matrix, walking its
// rows in chunks of 128.  Each chunk's M_t values (128 rows x 64 columns) and
// P rows arrive in shared memory by 16-byte asynchronous copies through a ring
// of kP2Stages stages, kP2Stages - 1 chunks ahead of the sums.  Thread t owns
// columns 2 (t % 32), 2 (t % 32) + 1 of the strip and rows 16 (t / 32) ... of
// each chunk; per-chunk sums are added with compensation, the 8 row groups in
// shared memory at the end, and the strip (one 64-row block of R) is
// grid-quantised.
// ---------------------------------------------------------------------------
constexpr int kP2Rows = 128;
constexpr int kP2Stages = 4;
constexpr int kP2StageBytes = kP2Rows * kS * 2 + kP2Rows * kRank * 4;   // M_t chunk + P rows
constexpr int kP2Smem = kP2Stages * kP2StageBytes + (kThreads / 32) * kS * kRank * 4;


__global__ void __launch_bounds__(kThreads, 2) grasp_pass2(GraspArgs a, const WsHeader* hdr) {
  grid_dep_sync();
  extern __shared__ __align__(16) unsigned char p2smem[];
  float (*part)[kS][kRank] = reinterpret_cast<float (*)[kS][kRank]>(p2smem + kP2Stages * kP2StageBytes);
  if (*reinterpret_cast<const volatile unsigned*>(&hdr->error) != 0u) return;
  const int pk = find_prob(a.cstrip_start, a.n, blockIdx.x);
  const GraspProb& P = a.probs[__ldg(a.corder + pk)];
  const int64_t bj = blockIdx.x - __ldg(a.cstrip_start + pk);
  const int64_t rows = P.m.rows, cols = P.m.cols;
  const int t = threadIdx.x;
  const int cp = t & 31, rg = t >> 5;   // column pair, row group (one per warp: P reads broadcast)
  const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(P.m.grad);
  const int64_t nch = (rows + kP2Rows - 1) / kP2Rows;
  // chunk c into stage c % kP2Stages: rows past the matrix are zero-filled
  auto load = [&](int64_t c) {
    unsigned char* st = p2smem + (c % kP2Stages) * kP2StageBytes;
    const int64_t r0 = c * kP2Rows;
#pragma unroll
    for (int k = 0; k < kP2Rows * kS * 2 / 16 / kThreads; ++k) {
      const int e = t + k * kThreads;
      const int row = e >> 3, seg = e & 7;
      const bool ok = r0 + row < rows;
      cp_async16(st + row * (kS * 2) + seg * 16, g + (ok ? (r0 + row) * cols : 0) + bj * kS + seg * 8, ok);
    }
    {
      const int row = t >> 1, half = t & 1;
      const bool ok = r0 + row < rows;
      cp_async16(st + kP2Rows * kS * 2 + row * (kRank * 4) + half * 16, P.p + (ok ? (r0 + row) * kRank : 0) + half * 4,
                 ok);
    }
  };
#pragma unroll
  for (int c = 0; c < kP2Stages - 1; ++c) {
    if (c < nch) load(c);
    cp_async_commit();
  }
  // sums of the thread's two columns as packed pairs (column 2 cp in .x,
  // 2 cp + 1 in .y): each component rounds as fmaf and as the scalar
  // compensated sum would
  float2 acc[kRank], accc[kRank];
#pragma unroll
  for (int l = 0; l < kRank; ++l) acc[l] = accc[l] = make_float2(0.0f, 0.0f);
  for (int64_t c = 0; c < nch; ++c) {
    if (c + kP2Stages - 1 < nch) load(c + kP2Stages - 1);
    cp_async_commit();
    cp_async_wait<kP2Stages - 1>();   // chunk c has landed (this thread's copies)
    __syncthreads();                  // ... and every thread's
    const unsigned char* st = p2smem + (c % kP2Stages) * kP2StageBytes;
    const uint32_t* sm = reinterpret_cast<const uint32_t*>(st);
    const float (*sp)[kRank] = reinterpret_cast<const float (*)[kRank]>(st + kP2Rows * kS * 2);
    float2 ab[kRank];
#pragma unroll
    for (int l = 0; l < kRank; ++l) ab[l] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int r = 0; r < kP2Rows / (kThreads / 32); ++r) {
      const int li = rg * (kP2Rows / (kThreads / 32)) + r;
      const uint32_t w = sm[li * (kS / 2) + cp];
      const float2 m = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
      float pr[kRank];
      *reinterpret_cast<float4*>(pr) = *reinterpret_cast<const float4*>(&sp[li][0]);
      *reinterpret_cast<float4*>(pr + 4) = *reinterpret_cast<const float4*>(&sp[li][4]);
#pragma unroll
      for (int l = 0; l < kRank; ++l) ab[l] = fma2(m, make_float2(pr[l], pr[l]), ab[l]);
    }
    // compensated sums over the chunks (TwoSum's error term is the exact
    // rounding error of each addition)
#pragma unroll
    for (int l = 0; l < kRank; ++l) two_sum_add2(acc[l], accc[l], ab[l]);
    __syncthreads();   // the stage is refilled by the next iteration's copies
  }
  cp_async_wait<0>();
#pragma unroll
  for (int l = 0; l < kRank; ++l) {
    part[rg][2 * cp][l] = acc[l].x + accc[l].x;
    part[rg][2 * cp + 1][l] = acc[l].y + accc[l].y;
  }
  __syncthreads();
  __shared__ float sx[kS][kRank];
  if (t < kS) {
    float sum[kRank];
#pragma unroll
    for (int l = 0; l < kRank; ++l) {
      float v = part[0][t][l];
      for (int w = 1; w < kThreads / 32; ++w) v += part[w][t][l];
      sum[l] = v;
      sx[t][l] = v;
    }
    float4* dst = reinterpret_cast<float4*>(P.r + (bj * kS + t) * kRank);
    dst[0] = make_float4(sum[0], sum[1], sum[2], sum[3]);
    dst[1] = make_float4(sum[4], sum[5], sum[6], sum[7]);
  }
  __syncthreads();
  // the strip is one 64-row block of R: its grid quantisation
  quantize_block8(sx, kS, bj * kS, P.m.r, P.m.r_rmax, P.m.r_cmax + bj * kRank);
}

// ---------------------------------------------------------------------------
// pass 3: residual M_t - P_t R_t^T and its 4-bit grid codes, one CTA of 128
// threads per 64-row x 256-column chunk (four 64 x 64 blocks).  The chunk's
// M_t values come into shared memory by asynchronous copies when the CTA
// starts, one commit group per block.  Thread t owns rows 4 (t / 8) ...
// 4 (t / 8) + 3 of the chunk and the 8 consecutive columns 8 (t % 8) of each
// block, so each column's R row read from shared memory serves four rows.
// Per block: the row maxima by shuffles over the row's 8 threads, the column
// maxima by a shuffle over the 4 row quads a warp holds and then the 4 warps'
// values in shared memory.
// ---------------------------------------------------------------------------
// Shared rows of 8 floats for the chunk's 256 columns, padded so that the
// eight columns a warp reads at once (8 apart) fall in different banks.
constexpr int kPadStride8 = kChunk * kS * kRank + (kChunk * kS / 8) * 4;
__device__ __forceinline__ int sidx8(int col, int l) { return col * kRank + (col >> 3) * 4 + l; }

constexpr int kP3Threads = 128;
constexpr int kP3Warps = kP3Threads / 32;
struct P3Smem {
  unsigned char m[kChunk][kS][kS * 2];   // the chunk's M_t (bf16), block by block
  float r[kPadStride8];                  // R_t rows of the chunk's columns
  float wmax[kP3Warps][kS];              // per-warp column maxima of a block
  float inv_c[kS];                       // fl(7 / cmax_j)
};
static_assert(offsetof(P3Smem, r) % 16 == 0, "pass 3 shared fields must stay 16-byte aligned");
constexpr int kP3Smem = (int)sizeof(P3Smem);

__global__ void __launch_bounds__(kP3Threads, 4) grasp_pass3(GraspArgs a, const WsHeader* hdr) {
  grid_dep_sync();
  extern __shared__ __align__(16) unsigned char p3smem[];
  P3Smem& S = *reinterpret_cast<P3Smem*>(p3smem);
  if (*reinterpret_cast<const volatile unsigned*>(&hdr->error) != 0u) return;
  const int pi = find_prob(a.tile_start, a.n, blockIdx.x);
  const GraspProb& P = a.probs[pi];
  const int64_t nchunk = (P.nbc + kChunk - 1) / kChunk;
  const int64_t local = blockIdx.x - __ldg(a.tile_start + pi);
  const int64_t bi = local / nchunk, b0 = (local % nchunk) * kChunk;
  const int nb = (P.nbc - b0) < kChunk ? (int)(P.nbc - b0) : kChunk;
  const int64_t rows = P.m.rows, cols = P.m.cols;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int rq = t >> 3, cg = t & 7;
  const int64_t i0 = bi * kS + 4 * rq;
  bool live[4];
#pragma unroll
  for (int h = 0; h < 4; ++h) live[h] = i0 + h < rows;
  const __nv_bfloat16* grad = static_cast<const __nv_bfloat16*>(P.m.grad);
  // the chunk's M_t: block c is commit group c (64 rows x 8 segments of 16
  // bytes, 4 per thread); rows past the matrix read as zeros
#pragma unroll
  for (int c = 0; c < kChunk; ++c) {
    if (c < nb) {
#pragma unroll
      for (int q = 0; q < kS * 8 / kP3Threads; ++q) {
        const int e = t + q * kP3Threads;
        const int row = e >> 3, seg = e & 7;
        const bool ok = bi * kS + row < rows;
        cp_async16(&S.m[c][row][seg * 16], grad + (ok ? (bi * kS + row) * cols + (b0 + c) * kS + seg * 8 : 0), ok);
      }
    }
    cp_async_commit();
  }
  for (int e = t; e < nb * kS * kRank / 4; e += kP3Threads)
    *reinterpret_cast<float4*>(&S.r[sidx8(e >> 1, (e & 1) * 4)]) =
        __ldg(reinterpret_cast<const float4*>(P.r + b0 * kS * kRank) + e);
  float p[4][kRank];
#pragma unroll
  for (int h = 0; h < 4; ++h)
#pragma unroll
    for (int l = 0; l < kRank; ++l) p[h][l] = live[h] ? P.p[(i0 + h) * kRank + l] : 0.0f;
#pragma unroll
  for (int c = 0; c < kChunk; ++c) {
    if (c >= nb) break;
    const int64_t bj = b0 + c;
    // block c's copies (commit groups 0..c) have landed, for every thread
    if (c == 0) cp_async_wait<kChunk - 1>();
    else if (c == 1) cp_async_wait<kChunk - 2>();
    else if (c == 2) cp_async_wait<kChunk - 3>();
    else cp_async_wait<0>();
    __syncthreads();
    float res[4][8];
    float cmx[8];
    uint4 mw[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) mw[h] = *reinterpret_cast<const uint4*>(&S.m[c][4 * rq + h][cg * 16]);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int cb = c * kS + 8 * cg + k;
      float rr[kRank];
      *reinterpret_cast<float4*>(rr) = *reinterpret_cast<const float4*>(&S.r[sidx8(cb, 0)]);
      *reinterpret_cast<float4*>(rr + 4) = *reinterpret_cast<const float4*>(&S.r[sidx8(cb, 4)]);
      // the rows' dot products P_i . R_j, row pairs at once, each in the order of fmaf's chain
      float2 a01 = make_float2(0.0f, 0.0f), a23 = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int l = 0; l < kRank; ++l) {
        a01 = fma2(make_float2(p[0][l], p[1][l]), make_float2(rr[l], rr[l]), a01);
        a23 = fma2(make_float2(p[2][l], p[3][l]), make_float2(rr[l], rr[l]), a23);
      }
      const float acc[4] = {a01.x, a01.y, a23.x, a23.y};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float v = 0.0f;
        if (live[h]) {
          const uint32_t w = (k >> 1) == 0 ? mw[h].x : (k >> 1) == 1 ? mw[h].y : (k >> 1) == 2 ? mw[h].z : mw[h].w;
          const float m = __uint_as_float((k & 1) ? (w & 0xFFFF0000u) : (w << 16));
          v = m - acc[h];
        }
        res[h][k] = v;
      }
      // fmaxf skips a NaN; a set of NaNs alone gives NaN, which the maxima
      // against zero further down drop, as a running maximum from zero would
      cmx[k] = fmaxf(fmaxf(fabsf(res[0][k]), fabsf(res[1][k])), fmaxf(fabsf(res[2][k]), fabsf(res[3][k])));
    }
    // row maxima over the block's 64 columns, reduced and scattered over the
    // 8 threads of a row quad: after the exchanges across lanes 4, 2 and 1
    // apart, thread cg holds the maximum of row hr = 2 (cg >> 2 & 1) + (cg >> 1 & 1)
    float rmh[4];
#pragma unroll
    for (int h = 0; h < 4; ++h)
      rmh[h] = fmaxf(fmaxf(fmaxf(fabsf(res[h][0]), fabsf(res[h][1])), fmaxf(fabsf(res[h][2]), fabsf(res[h][3]))),
                     fmaxf(fmaxf(fabsf(res[h][4]), fabsf(res[h][5])), fmaxf(fabsf(res[h][6]), fabsf(res[h][7]))));
    const bool hi2 = (cg & 4) != 0, hi1 = (cg & 2) != 0;
    float k0 = hi2 ? rmh[2] : rmh[0], k1 = hi2 ? rmh[3] : rmh[1];
    k0 = fmaxf(k0, __shfl_xor_sync(0xffffffffu, hi2 ? rmh[0] : rmh[2], 4));
    k1 = fmaxf(k1, __shfl_xor_sync(0xffffffffu, hi2 ? rmh[1] : rmh[3], 4));
    float rk = hi1 ? k1 : k0;
    rk = fmaxf(rk, __shfl_xor_sync(0xffffffffu, hi1 ? k0 : k1, 2));
    rk = fmaxf(rk, __shfl_xor_sync(0xffffffffu, rk, 1));
    rk = fmaxf(rk, 0.0f);
    const int hr = (hi2 ? 2 : 0) + (hi1 ? 1 : 0);
    if ((cg & 1) == 0 && i0 + hr < rows) P.m.res_rmax[bj * rows + i0 + hr] = rk;
    const float irr = inv_level(rk, 7.0f);
    float ir[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) ir[h] = __shfl_sync(0xffffffffu, irr, (h >> 1) * 4 + (h & 1) * 2, 8);
    // column maxima: lanes l, l ^ 8, l ^ 16, l ^ 24 hold the same columns of the warp's 16 rows
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float v = cmx[k];
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
      if (lane < 8) S.wmax[warp][8 * cg + k] = v;
    }
    __syncthreads();
    int inf_c = 0;
    if (t < kS) {
      float cm = 0.0f;
#pragma unroll
      for (int w = 0; w < kP3Warps; ++w) cm = fmaxf(cm, S.wmax[w][t]);
      P.m.res_cmax[bi * cols + bj * kS + t] = cm;
      const float icm = inv_level(cm, 7.0f);
      S.inv_c[t] = icm;
      inf_c = icm == INFINITY;
    }
    const bool any_inf_c = __syncthreads_or(inf_c) != 0;
    float ic[8];
    *reinterpret_cast<float4*>(ic) = *reinterpret_cast<const float4*>(&S.inv_c[8 * cg]);
    *reinterpret_cast<float4*>(ic + 4) = *reinterpret_cast<const float4*>(&S.inv_c[8 * cg + 4]);
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      if (!live[h]) continue;
      const int64_t i = i0 + h;
      uint32_t cw;
      if (!any_inf_c && ir[h] != INFINITY) {
        // Every factor fl(7 / min(r, c)) is finite and |x| <= min(r, c), so
        // fl(x * factor) <= 7 (1 + 2^-24) in magnitude: each code is already in
        // [-7, 7] (a NaN converts to 0), and the codes are packed by a
        // multiply-add chain modulo 2^32, offset by 8 per nibble at the end.
        uint32_t acc = 0u;
#pragma unroll
        for (int k = 7; k >= 0; --k)
          acc = acc * 16u + (uint32_t)__float2int_rn(__fmul_rn(res[h][k], grid_factor(ir[h], ic[k])));
        cw = acc + 0x88888888u;
      } else {
        cw = 0u;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int q = grid_code(res[h][k], grid_factor(ir[h], ic[k]), 7);
          cw |= (uint32_t)(q + 8) << (4 * k);
        }
      }
      *reinterpret_cast<uint32_t*>(P.m.res + i * (cols / 2) + (bj * kS + 8 * cg) / 2) = cw;
    }
    __syncthreads();   // wmax and inv_c are rewritten by the next block
  }
  cp_async_wait<0>();
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t prob_scratch_bytes(const qmuon_grasp_matrix& m) {
  const size_t nbr = (size_t)(m.rows + kS - 1) / kS;
  const size_t ncc = (size_t)(m.cols + kNormCols - 1) / kNormCols;
  return 2 * align_up((size_t)m.cols * kRank * 4, 256) + align_up(ncc * kRank * 8, 256) +
         2 * align_up((size_t)m.rows * kRank * 4, 256) +
         align_up((size_t)m.rows * kRank * 8, 256) + align_up(nbr * 36 * 8, 256) + align_up(kRank * kRank * 8, 256);
}

// A launch that may start while the stream's previous kernel finishes: the
// kernel itself waits for that kernel (grid_dep_sync) before it reads anything.
template <typename... KArgs, typename... Args>
cudaError_t launch_dep(void (*kern)(KArgs...), dim3 grid, unsigned block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

size_t table_bytes(int32_t n) {
  return align_up((size_t)n * sizeof(GraspProb), 256) + 3 * align_up((size_t)(n + 1) * 8, 256) +
         2 * align_up((size_t)n * 4, 256);
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

qmuon_status validate(const qmuon_grasp_matrix& m) {
  // a rank-8 orthonormal factor needs at least 8 rows
  if (m.rows < kRank || m.cols <= 0 || m.rows > (1 << 28) || m.cols > (1 << 28)) return QMUON_ERR_INVALID_ARGUMENT;
  if (m.cols % kS) return QMUON_ERR_UNSUPPORTED;
  if (!m.res || !m.res_rmax || !m.res_cmax || !m.p || !m.p_rmax || !m.p_cmax || !m.r || !m.r_rmax || !m.r_cmax ||
      !m.grad)
    return QMUON_ERR_INVALID_ARGUMENT;
  if (!aligned_to(m.res, 8) || !aligned_to(m.p, 8) || !aligned_to(m.r, 8) || !aligned_to(m.grad, 16) ||
      !aligned_to(m.res_rmax, 4) || !aligned_to(m.res_cmax, 4) || !aligned_to(m.p_rmax, 4) ||
      !aligned_to(m.p_cmax, 4) || !aligned_to(m.r_rmax, 4) || !aligned_to(m.r_cmax, 4))
    return QMUON_ERR_INVALID_ARGUMENT;
  return QMUON_OK;
}

}  // namespace
}  // namespace qm

extern "C" size_t qmuon_grasp_workspace_size(const qmuon_grasp_matrix* matrices, int32_t n) {
  using namespace qm;
  if (!matrices || n <= 0) return 0;
  size_t b = kWsHeader + table_bytes(n);
  for (int32_t i = 0; i < n; ++i) {
    // a shape qmuon_grasp_step rejects has no workspace size (the pointers
    // may still be unset when the size is asked for)
    const qmuon_grasp_matrix& m = matrices[i];
    if (m.rows < kRank || m.cols <= 0 || m.cols % kS || m.rows > (1 << 28) || m.cols > (1 << 28)) return 0;
    b += prob_scratch_bytes(m);
  }
  return b;
}

extern "C" qmuon_status qmuon_grasp_step(const qmuon_grasp_matrix* matrices, int32_t n, float mu, void* ws,
                                         size_t ws_bytes, void* stream) {
  qm::NvtxRange nvtx_range("qmuon_grasp_step");
  return qm::no_throw("qmuon_grasp_step", [&]() -> qmuon_status {
    using namespace qm;
    if (!matrices || n <= 0 || !ws || !aligned_to(ws, 256)) return QMUON_ERR_INVALID_ARGUMENT;
    for (int32_t i = 0; i < n; ++i) {
      const qmuon_status s = validate(matrices[i]);
      if (s != QMUON_OK) return s;
    }
    if (ws_bytes < qmuon_grasp_workspace_size(matrices, n)) return QMUON_ERR_WORKSPACE_TOO_SMALL;
    unsigned char* b = static_cast<unsigned char*>(ws);
    WsHeader* hdr = reinterpret_cast<WsHeader*>(b);
    unsigned char* table = b + kWsHeader;
    unsigned char* scratch = table + table_bytes(n);
    std::vector<GraspProb> hp(n);
    std::vector<int64_t> ts(n + 1, 0), rs(n + 1, 0), cs(n + 1, 0);
    for (int32_t i = 0; i < n; ++i) {
      GraspProb& P = hp[i];
      std::memset(&P, 0, sizeof(P));
      P.m = matrices[i];
      P.nbr = (P.m.rows + kS - 1) / kS;
      P.nbc = P.m.cols / kS;
      auto carve = [&](size_t bytes) {
        float* p = reinterpret_cast<float*>(scratch);
        scratch += align_up(bytes, 256);
        return p;
      };
      P.ncc = (P.m.cols + kNormCols - 1) / kNormCols;
      P.qpart = reinterpret_cast<double*>(carve((size_t)P.ncc * kRank * 8));
      P.rdeq = carve((size_t)P.m.cols * kRank * 4);
      P.y = carve((size_t)P.m.rows * kRank * 4);
      P.p = carve((size_t)P.m.rows * kRank * 4);
      P.r = carve((size_t)P.m.cols * kRank * 4);
      P.p1 = reinterpret_cast<double*>(carve((size_t)P.m.rows * kRank * 8));
      P.gpart = reinterpret_cast<double*>(carve((size_t)P.nbr * 36 * 8));
      P.L = reinterpret_cast<double*>(carve(kRank * kRank * 8));
      ts[i + 1] = ts[i] + P.nbr * ((P.nbc + kChunk - 1) / kChunk);   // pass 3: 64 x 256 chunks (all alike)
    }
    // row strips longest (most columns) first, column strips longest (most rows) first
    std::vector<int32_t> ro(n), co(n);
    for (int32_t i = 0; i < n; ++i) ro[i] = co[i] = i;
    std::stable_sort(ro.begin(), ro.end(), [&](int32_t x, int32_t y) { return hp[x].m.cols > hp[y].m.cols; });
    std::stable_sort(co.begin(), co.end(), [&](int32_t x, int32_t y) { return hp[x].m.rows > hp[y].m.rows; });
    for (int32_t k = 0; k < n; ++k) {
      rs[k + 1] = rs[k] + hp[ro[k]].nbr;
      cs[k + 1] = cs[k] + hp[co[k]].nbc;
    }
    GraspArgs a{};
    a.probs = reinterpret_cast<const GraspProb*>(table);
    unsigned char* pre = table + align_up((size_t)n * sizeof(GraspProb), 256);
    a.tile_start = reinterpret_cast<const int64_t*>(pre);
    a.rstrip_start = reinterpret_cast<const int64_t*>(pre + align_up((size_t)(n + 1) * 8, 256));
    a.cstrip_start = reinterpret_cast<const int64_t*>(pre + 2 * align_up((size_t)(n + 1) * 8, 256));
    a.rorder = reinterpret_cast<const int32_t*>(pre + 3 * align_up((size_t)(n + 1) * 8, 256));
    a.corder = reinterpret_cast<const int32_t*>(pre + 3 * align_up((size_t)(n + 1) * 8, 256) +
                                                align_up((size_t)n * 4, 256));
    a.n = n;
    a.mu = mu;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(hdr, 0, kWsHeader, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(table, hp.data(), (size_t)n * sizeof(GraspProb), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(const_cast<int64_t*>(a.tile_start), ts.data(), (size_t)(n + 1) * 8, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(const_cast<int64_t*>(a.rstrip_start), rs.data(), (size_t)(n + 1) * 8, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(const_cast<int64_t*>(a.cstrip_start), cs.data(), (size_t)(n + 1) * 8, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(const_cast<int32_t*>(a.rorder), ro.data(), (size_t)n * 4, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(const_cast<int32_t*>(a.corder), co.data(), (size_t)n * 4, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return set_error("qmuon_grasp_step (upload)", e);
    const int64_t tiles = ts[n];
    if (tiles > (int64_t)0x7FFFFFFF) return QMUON_ERR_UNSUPPORTED;
    // the opt-in belongs to the current device, so it is made on every call
    cudaError_t attr = cudaFuncSetAttribute(grasp_pass2, cudaFuncAttributeMaxDynamicSharedMemorySize, kP2Smem);
    if (attr == cudaSuccess)
      attr = cudaFuncSetAttribute(grasp_pass1, cudaFuncAttributeMaxDynamicSharedMemorySize, kP1Smem);
    if (attr == cudaSuccess)
      attr = cudaFuncSetAttribute(grasp_pass3, cudaFuncAttributeMaxDynamicSharedMemorySize, kP3Smem);
    if (attr != cudaSuccess) return set_error("qmuon_grasp_step (shared memory attribute)", attr);
    int64_t ncc_max = 1;
    for (int32_t i = 0; i < n; ++i) ncc_max = hp[i].ncc > ncc_max ? hp[i].ncc : ncc_max;
    e = launch_dep(grasp_colnorm, dim3((unsigned)ncc_max, (unsigned)n), kThreads, 0, s, a);
    if (e == cudaSuccess) e = launch_dep(grasp_pass1, (unsigned)rs[n], kThreads, kP1Smem, s, a);
    if (e == cudaSuccess) e = launch_dep(grasp_chol, (unsigned)n, 64, 0, s, a, hdr);
    if (e == cudaSuccess) e = launch_dep(grasp_tsolve<0>, (unsigned)rs[n], 64, 0, s, a, (const WsHeader*)hdr);
    if (e == cudaSuccess) e = launch_dep(grasp_chol, (unsigned)n, 64, 0, s, a, hdr);
    if (e == cudaSuccess) e = launch_dep(grasp_tsolve<1>, (unsigned)rs[n], 64, 0, s, a, (const WsHeader*)hdr);
    if (e == cudaSuccess) e = launch_dep(grasp_pass2, (unsigned)cs[n], kThreads, kP2Smem, s, a, (const WsHeader*)hdr);
    if (e == cudaSuccess) e = launch_dep(grasp_pass3, (unsigned)tiles, kP3Threads, kP3Smem, s, a, (const WsHeader*)hdr);
    // the pageable host tables are staged by the copies above before they return
    if (e != cudaSuccess) return set_error("qmuon_grasp_step (launch)", e);
    tally(T_GRASP_CALLS);
    tally(T_GRASP_MATRICES, (uint64_t)n);
    tally(T_GRAD_BF16, (uint64_t)n);
    return QMUON_OK;
  });
}

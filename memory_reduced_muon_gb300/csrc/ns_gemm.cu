// Quintic Newton-Schulz orthogonalisation on tcgen05 tensor cores (sm_103a).
//
// One iteration is three matrix products ("NVIDIA impulsa optimizadores
// avanzados ... con Megatron", section "Newton-Schulz distribuido"):
//   G_GRAM   A = s1 * X X^T            (s1 = inv^2 on the first iteration)
//   G_POLY   B = a I + b A + c A A
//   G_UPDATE X <- s3 * (B X)           (s3 = inv on the first iteration;
//                                       the last one may also apply W -= eta U)
// The a X term of the quintic rides in B's diagonal: a X + (b A + c A A) X =
// (a I + b A + c A A) X, so the update is one plain product and never reads X
// outside its operand pipeline.  A matrix stored with more rows than columns
// (S, n x m) is orthogonalised as its transpose without moving data: A = S^T S
// and S <- S B, since (B X)^T = X^T B for the symmetric B.  Operands are bf16,
// accumulation fp32 in tensor memory.
//
// Kernel: a persistent CTA pair (cta_group::2, one cluster) per two SMs runs
// the 256 x 256 output tiles the host scheduled for it, over every problem of
// the batch.  10 warps per CTA: warp 0 issues TMA loads (64 x 64 bf16 boxes,
// 128-byte swizzle) into a shared-memory ring, warp 1 allocates 512 TMEM
// columns (two accumulators) and, in the leader CTA, issues tcgen05.mma
// (M=256, N=256, K=16) from one thread; warps 2-9 read the accumulator back
// with tcgen05.ld and run the fused epilogue.  K-major and MN-major operands
// are both read straight from the row-major buffers; the instruction
// descriptor says which.  Every mbarrier wait is bounded: on expiry it records
// QMUON_ERR_TIMEOUT in the workspace header and the CTA winds down instead of
// hanging.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <utility>
#include <vector>

#include "qm_ns.h"

namespace qm {
namespace ns {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kEpiWarps = 8;                      // epilogue warps: two per TMEM lane quarter
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 64 + kEpiThreads;        // warp 0 TMA, warp 1 MMA, warps 2.. epilogue
constexpr uint32_t kBox = 64 * 64 * 2;          // one TMA box: 64 x 64 bf16 = 8 KB
constexpr uint32_t kStageA = 2 * kBox;          // 128 rows (or columns) x 64
constexpr uint32_t kStageB = 4 * kBox;          // 256 x 64
constexpr uint32_t kStageBytes = kStageA + kStageB;
constexpr uint32_t kTmemCols = 512;             // two 128 x 256 fp32 accumulators
constexpr uint32_t kStageOutBytes = 128 * 128 * 2;   // epilogue staging: two 64-column steps (Gram) or 8 x 4 KB warp boxes
constexpr uint32_t kUSlotBytes = 2 * kBox;           // G_UPDATE_W: 128 x 64 output columns of one step
constexpr uint32_t kWChunkBytes = 128 * 32 * 4;      // G_UPDATE_W: 128 rows x 32 fp32 weights (one TMA box)

// Shared memory per product kind and CTA group.  One CTA (CG = 1) owns a
// 128 x 256 output tile and loads all of A (128 rows) and B (256 rows) per
// stage (48 KB); a CTA pair (CG = 2) owns 256 x 256, each CTA loading its
// 128 rows of A and half of B (32 KB per stage per CTA).  The polynomial and
// update products stage their output per epilogue warp (4 KB each, one
// 32 x 64 TMA box at a time), the Gram in two buffers of one 64-column step
// each; the updates that also move the weights keep two output slots of one
// step each and a ring of weight chunks, two per step (one per column half),
// two steps deep (kind 3, for short K loops where the weights bound the tile)
// or one step deep with a fifth operand stage (kind 4, for long K loops).
__host__ __device__ constexpr uint32_t stage_bytes_of(int cg) { return cg == 2 ? 4 * kBox : kStageBytes; }
__host__ __device__ constexpr int w_depth_of(int kind) { return kind == 3 ? 2 : 1; }
__host__ __device__ constexpr int stages_of(int kind, int cg) {
  return cg == 2 ? (kind == 3 ? 4 : kind == 4 ? 5 : 6) : (kind >= 3 ? 2 : 4);
}
__host__ __device__ constexpr uint32_t side_bytes_of(int kind, int cg) {
  return kind >= 3 ? 2 * kUSlotBytes + 2 * w_depth_of(kind) * kWChunkBytes : kStageOutBytes;
}
__host__ __device__ constexpr size_t smem_bytes_of(int kind, int cg) {
  return (size_t)stages_of(kind, cg) * stage_bytes_of(cg) + side_bytes_of(kind, cg) + 1024 + 256;
}

static_assert(smem_bytes_of(0, 2) <= 232448 && smem_bytes_of(1, 2) <= 232448 && smem_bytes_of(2, 2) <= 232448 &&
                  smem_bytes_of(3, 2) <= 232448 && smem_bytes_of(4, 2) <= 232448,
              "dynamic shared memory above the 227 KB a CTA may use");

constexpr long long kWaitCycles = 4000000000LL;  // bounded waits: ~2 s at 2 GHz

// G_UPDATE_W and G_UPDATE_W1 are G_UPDATE on the last iteration of a step:
// they also apply W <- W - eta * bf16(U) to the fp32 weights (weight ring two
// steps or one step deep).
enum { G_GRAM = 0, G_POLY = 1, G_UPDATE = 2, G_UPDATE_W = 3, G_UPDATE_W1 = 4 };

// CTA group of the Newton-Schulz GEMMs: 2 = CTA pairs (cta_group::2).
constexpr int kCG = 2;

struct alignas(128) NsProb {
  CUtensorMap map_x[3];   // X buffers: 0 = caller's matrix, 1/2 = workspace ping-pong
  CUtensorMap map_a;      // m x m Gram
  CUtensorMap map_b;      // m x m polynomial
  CUtensorMap map_w;      // fp32 weights (stored orientation, 32 x 128 boxes), when w is set
  CUtensorMap map_x32[3]; // the X buffers with 32-row boxes: one epilogue warp's stores
  CUtensorMap map_b32;    // B with 32-row boxes, likewise
  __nv_bfloat16* x[3];
  int64_t x_ld[3];
  __nv_bfloat16* a;
  __nv_bfloat16* b;
  int64_t ab_ld;          // row stride of A and B: m rounded up to 8 (16-byte rows for TMA)
  float* w;               // fp32 weights (stored orientation) or null
  int64_t w_ld;
  const float* inv;       // inverse norm applied on the first iteration, or null
  int32_t rows, cols;     // stored shape
  int32_t m, n;           // m = min(rows, cols), n = max
  int32_t tall;           // rows > cols
  int32_t tiles_n[3];     // output tile columns per product kind
  int32_t tiles[3];       // output tiles per product kind
};

// One entry of a launch's tile schedule: output tile `local` of problem `prob`.
struct TileRef {
  int32_t prob, local;
};

struct GemmArgs {
  const NsProb* probs;
  const int32_t* sched_start;  // [groups + 1]: CTA group g runs sched[sched_start[g] .. sched_start[g + 1])
  const TileRef* sched;
  int32_t src, dst;           // X buffer indices read / written (G_UPDATE); src for G_GRAM
  int32_t first;              // apply inv (first iteration)
  float ca, cb, cc, eta;
  WsHeader* hdr;
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void record_error(WsHeader* h, unsigned code, unsigned where) {
  if (atomicCAS(&h->error, 0u, code) == 0u) h->error_info = where;
}
// Bounded wait: false when the phase did not complete in time (or another
// CTA already gave up), after recording the timeout.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, WsHeader* h, unsigned where) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (unsigned i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0u) {
      if (*reinterpret_cast<volatile unsigned*>(&h->error) != 0u) return false;
      if (clock64() - t0 > kWaitCycles) {
        record_error(h, QMUON_ERR_TIMEOUT, where);
        return false;
      }
    }
  }
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(dst), "l"(map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
// The same with an L2 cache policy (streams read once: evict first).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;"
      ::"r"(dst), "l"(map), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// Make tensor maps written through the generic proxy (host copies into global
// memory) visible to the tensor-map proxy before the first TMA that uses them.
__device__ __forceinline__ void fence_tensormap(const CUtensorMap* map) {
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(map) : "memory");
}
// ---- CTA-pair (cta_group::2) forms: every tcgen05 instruction of a kernel
// uses the same CTA group, so each wrapper is templated on it ----
template <int CG>
__device__ __forceinline__ void tmem_alloc_cg(uint32_t dst_smem, uint32_t ncols) {
  if (CG == 2)
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
template <int CG>
__device__ __forceinline__ void tmem_relinquish_cg() {
  if (CG == 2) asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  else asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
template <int CG>
__device__ __forceinline__ void tmem_dealloc_cg(uint32_t taddr, uint32_t ncols) {
  if (CG == 2) asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
  else asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
template <int CG>
__device__ __forceinline__ void mma_bf16_cg(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  if (CG == 2)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on barrier `bar` (same offset) in every CTA of the group once all
// prior tcgen05 operations of this thread have completed.
template <int CG>
__device__ __forceinline__ void mma_commit_cg(uint32_t bar) {
  if (CG == 2)
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        ::"r"(bar), "h"((unsigned short)0x3)
        : "memory");
  else
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// TMA store of one box from this CTA's shared memory (bulk async group).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
               ::"l"(map), "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, uint32_t src, int x, int y,
                                                  uint64_t policy) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;"
               ::"l"(map), "r"(src), "r"(x), "r"(y), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... all but the most recent group of this thread's bulk stores have read their shared memory
__device__ __forceinline__ void bulk_wait_read_but1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA) before a barrier hands the data to the storing thread.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The address of the same shared-memory offset in cluster CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on the
// barrier of the pair's leader CTA (`bar` is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(dst), "l"(map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// tcgen05.ld without the wait: several loads in flight, then tmem_wait_ld and
// tmem_hold on each destination, so no use of the registers moves above the wait.
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_hold(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

// Shared-memory matrix descriptor (tcgen05): start address, leading- and
// stride-dimension byte offsets (all >> 4), descriptor version 1 at bit 46,
// 128-byte swizzle (layout type 2) at bits 61-63.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// K-major tile (rows of 64 K-elements = 128 B, 8-row swizzle atoms of 1 KB):
// the k-th 16-wide slice starts 32 B further in.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int kk) { return smem_desc(tile + kk * 32, 16, 1024); }
// MN-major tile (one 8 KB box per 64 MN-elements, a K row = 128 B): the k-th
// 16-row slice starts 16 rows (2 KB) further in; MN atoms are 8 KB apart.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int kk) { return smem_desc(tile + kk * 2048, kBox, 1024); }

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A/B
// major-ness, N >> 3 at bit 17, M >> 4 at bit 24.
__device__ __forceinline__ uint32_t make_idesc(bool a_mn, bool b_mn, int M = BM) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}


__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
}

// Load 32 bf16 starting at p (valid elements only when n < 32) as fp32.
__device__ __forceinline__ void load_row32(const __nv_bfloat16* p, int n, float (&v)[32]) {
  if (n >= 32) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 u = q[i];
      v[8 * i + 0] = bf16_lo(u.x); v[8 * i + 1] = bf16_hi(u.x);
      v[8 * i + 2] = bf16_lo(u.y); v[8 * i + 3] = bf16_hi(u.y);
      v[8 * i + 4] = bf16_lo(u.z); v[8 * i + 5] = bf16_hi(u.z);
      v[8 * i + 6] = bf16_lo(u.w); v[8 * i + 7] = bf16_hi(u.w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = (i < n) ? __bfloat162float(p[i]) : 0.0f;
  }
}

// Output tile (I, J) of problem P for product KIND, from its index in the
// problem's tile list.  Tiles are (128 CG) x 256.  The symmetric products list
// only tiles touching the upper triangle, column block J by column block J:
// for CG = 1 the 128 x 256 tiles with 128 I < 256 J + 256, for CG = 2 the
// square tiles with I <= J.
template <int CG>
__device__ __forceinline__ void decode_tile(const NsProb& P, int kind, int local, int& I, int& J) {
  if (kind >= G_UPDATE) {
    // the update product's tiles in the order CTA groups take them up: the
    // tiles that run at the same time share one panel of the X operand, read
    // once from DRAM, while they walk the other operand, B (m x m), which L2
    // holds.  A tall problem's X is the A operand (row panels: row-major
    // order), a wide one's the B operand (column panels: column-major order).
    const int tn = P.tiles_n[G_UPDATE];
    if (P.tall) {
      I = local / tn;
      J = local % tn;
    } else {
      const int tm = P.tiles[G_UPDATE] / tn;
      I = local % tm;
      J = local / tm;
    }
    return;
  }
  const int TM = (P.m + 128 * CG - 1) / (128 * CG);
  int j = 0;
  for (;;) {
    const int want = (CG == 2) ? j + 1 : 2 * j + 2;
    const int cnt = want < TM ? want : TM;
    if (local < cnt) {
      I = local;
      J = j;
      return;
    }
    local -= cnt;
    ++j;
  }
}

struct TileGeom {
  const NsProb* P;
  int row0, col0;    // this CTA's first output row / the tile's first column
  int bcol0;         // first B row (output column) this CTA loads
  int M_, N_, K_;
  bool a_mn, b_mn;
  // The symmetric matrices (the Gram A and the polynomial B) hold only their
  // 256 x 256 tiles on or above the diagonal.  An operand read from one has
  // the index of its 256-row tile here (else -1): its K blocks left of that
  // tile lie below the diagonal and are read as the transposed block above
  // it, by an MN-major box at swapped coordinates.
  int a_sym, b_sym;
  const CUtensorMap* mapA;
  const CUtensorMap* mapB;
};

template <int KIND, int CG>
__device__ __forceinline__ TileGeom tile_geom(const GemmArgs& args, int k, int rank) {
  const int2 e = __ldg(reinterpret_cast<const int2*>(args.sched) + k);
  TileGeom g;
  g.P = args.probs + e.x;
  const NsProb& P = *g.P;
  int I, J;
  decode_tile<CG>(P, KIND, e.y, I, J);
  g.row0 = I * (128 * CG) + 128 * rank;
  g.col0 = J * BN;
  g.bcol0 = g.col0 + (CG == 2 ? 128 * rank : 0);
  g.a_sym = g.b_sym = -1;
  if (KIND == G_GRAM) {
    g.M_ = P.m; g.N_ = P.m; g.K_ = P.n;
    g.mapA = g.mapB = &P.map_x[args.src];
    g.a_mn = g.b_mn = (P.tall != 0);
  } else if (KIND == G_POLY) {
    g.M_ = P.m; g.N_ = P.m; g.K_ = P.m;
    g.mapA = g.mapB = &P.map_a;
    g.a_mn = g.b_mn = false;
    g.a_sym = I;
    g.b_sym = J;
  } else if (!P.tall) {
    g.M_ = P.m; g.N_ = P.n; g.K_ = P.m;
    g.mapA = &P.map_b; g.a_mn = false;
    g.mapB = &P.map_x[args.src]; g.b_mn = true;
    g.a_sym = I;
  } else {
    g.M_ = P.n; g.N_ = P.m; g.K_ = P.m;
    g.mapA = &P.map_x[args.src]; g.a_mn = false;
    g.mapB = &P.map_b; g.b_mn = false;
    g.b_sym = J;
  }
  return g;
}

__device__ __forceinline__ void named_barrier_epilogue() {
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
}
// AND of `v` over the 128 epilogue threads (also a barrier among them), so the
// four epilogue warps always take the same branch around their barriers.
__device__ __forceinline__ bool epilogue_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "n"(kEpiThreads)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Persistent kernel: one CTA (CG = 1) or one CTA pair (CG = 2) per SM (pair)
// runs its own list of tiles, which the host balanced by their cost.  The
// shared-memory ring and the two TMEM accumulators carry over from tile to
// tile, so the loads of the next tile and the epilogue of the last one
// overlap the tensor cores.  In a pair, the leader CTA (rank 0) issues the
// M = 256 MMAs for both; every CTA's loads complete on the leader's "full"
// barriers, and the leader's commits arrive on both CTAs' barriers.
template <int KIND, int CG>
__global__ void __launch_bounds__(kThreads, 1) ns_gemm_kernel(const __grid_constant__ GemmArgs args) {
  constexpr int STAGES = stages_of(KIND, CG);
  constexpr uint32_t SB = stage_bytes_of(CG);          // bytes per stage per CTA
  constexpr uint32_t SA = 2 * kBox;                    // A part: 128 rows (or columns) x 64
  constexpr int NB = (CG == 2) ? 2 : 4;                // B boxes per stage per CTA
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  unsigned char* side = smem + STAGES * SB;                   // staging: half tile (symmetric) or tile (update)
  uint64_t* bars = reinterpret_cast<uint64_t*>(side + side_bytes_of(KIND, CG));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 8);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
  const uint32_t tfull0 = smem_u32(bars + 2 * STAGES), tempty0 = smem_u32(bars + 2 * STAGES + 2);
  const uint32_t wfull0 = smem_u32(bars + 2 * STAGES + 4);   // weight passes: chunk slots 0..3

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (CG == 2) ? (int)cluster_rank() : 0;
  const bool leader = (rank == 0);
  // this CTA group's tiles, in the order the host's schedule lists them
  const int group = blockIdx.x / CG;
  const int k_begin = __ldg(args.sched_start + group), k_end = __ldg(args.sched_start + group + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8 * b, 1);
      mbar_init(tempty0 + 8 * b, kEpiWarps * CG);   // one arrival per epilogue warp of the group
    }
    for (int b = 0; b < 4; ++b) mbar_init(wfull0 + 8 * b, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_cg<CG>(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_cg<CG>();
  }
  tc_fence_before();
  __syncwarp();   // the cluster barrier is warp-aligned: reconverge first
  if (CG == 2) cluster_sync_all();   // the peer's barriers exist before anyone signals them
  else __syncthreads();
  tc_fence_after();
  // The products of a Newton-Schulz call are launched as programmatic
  // dependents of one another: the next one may be scheduled on the SMs this
  // grid leaves free and set up its barriers and tensor memory meanwhile.
  // Until here nothing was read that an earlier kernel writes (the problem
  // and tile tables come from the host before the call); past the wait, every
  // earlier grid of the stream has completed and its writes are visible.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer (every CTA loads its own operand halves) ----
      const uint32_t full_l = (CG == 2) ? cluster_map(full0, 0) : full0;   // the leader's barriers
      int it = 0;
      bool ok = true;
      const CUtensorMap* fenced[2] = {nullptr, nullptr};   // maps fenced for the last tile
      auto fence_once = [&](const CUtensorMap* mp) {
        if (mp != fenced[0] && mp != fenced[1]) fence_tensormap(mp);
      };
      for (int tile = k_begin; tile < k_end && ok; ++tile) {
        const TileGeom g = tile_geom<KIND, CG>(args, tile, rank);
        // a tensor map written by the host is fenced once per run of tiles using it
        fence_once(g.mapA);
        if (g.mapB != g.mapA) fence_once(g.mapB);
        fenced[0] = g.mapA;
        fenced[1] = g.mapB;
        const int num_kb = (g.K_ + BK - 1) / BK;
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % STAGES, round = it / STAGES;
          if (round > 0 && !mbar_wait(empty0 + 8 * s, (round - 1) & 1, args.hdr, 0x100u | KIND)) {
            ok = false;
            break;
          }
          if (leader) mbar_expect_tx(full0 + 8 * s, SB * CG);
          const uint32_t bar = full_l + 8 * s;
          const uint32_t sa = smem_u32(smem + s * SB), sb = sa + SA;
          const int k0 = kb * BK;
          const bool amn = g.a_mn || g.a_sym > k0 / 256, bmn = g.b_mn || g.b_sym > k0 / 256;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int x = amn ? g.row0 + 64 * i : k0, y = amn ? k0 : g.row0 + 64 * i;
            if (CG == 2) tma_load_2d_pair(sa + i * kBox, g.mapA, bar, x, y);
            else tma_load_2d(sa + i * kBox, g.mapA, bar, x, y);
          }
#pragma unroll
          for (int j = 0; j < NB; ++j) {
            const int x = bmn ? g.bcol0 + 64 * j : k0, y = bmn ? k0 : g.bcol0 + 64 * j;
            if (CG == 2) tma_load_2d_pair(sb + j * kBox, g.mapB, bar, x, y);
            else tma_load_2d(sb + j * kBox, g.mapB, bar, x, y);
          }
        }
      }
      // every load issued has landed before the CTA may exit (the leader's
      // full barriers also count the peer's loads)
      if (leader)
        for (int k = (it > STAGES ? it - STAGES : 0); k < it; ++k)
          mbar_wait(full0 + 8 * (k % STAGES), (k / STAGES) & 1, args.hdr, 0x200u | KIND);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---- MMA issuer (the leader CTA of the group) ----
      int it = 0, ti = 0;
      bool ok = true;
      for (int tile = k_begin; tile < k_end && ok; ++tile, ++ti) {
        const TileGeom g = tile_geom<KIND, CG>(args, tile, 0);
        const int acc = ti & 1, use = ti >> 1;
        if (use > 0 && !mbar_wait(tempty0 + 8 * acc, (use - 1) & 1, args.hdr, 0x500u | KIND)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * BN);
        const int num_kb = (g.K_ + BK - 1) / BK;
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % STAGES, round = it / STAGES;
          if (!mbar_wait(full0 + 8 * s, round & 1, args.hdr, 0x300u | KIND)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * SB), sb = sa + SA;
          // each stage's operands are K-major or MN-major as the producer loaded them
          const bool amn = g.a_mn || g.a_sym > (kb * BK) / 256, bmn = g.b_mn || g.b_sym > (kb * BK) / 256;
          const uint32_t idesc = make_idesc(amn, bmn, 128 * CG);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = amn ? desc_mnmajor(sa, kk) : desc_kmajor(sa, kk);
            const uint64_t bd = bmn ? desc_mnmajor(sb, kk) : desc_kmajor(sb, kk);
            mma_bf16_cg<CG>(d, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit_cg<CG>(empty0 + 8 * s);   // frees the stage (in every CTA of the group)
        }
        mma_commit_cg<CG>(tfull0 + 8 * acc);   // accumulator ready (also on the error path)
      }
    }
  } else {
    // ---- epilogue: warps 2..9; TMEM lane quarter = warp % 4 ----
    const int quarter = warp & 3;
    const int ew = warp - 2;          // epilogue warp 0..7
    const int ch = ew >> 2;           // column half of the tile (TMEM lanes are shared per quarter)
    const uint32_t tempty_l = (CG == 2) ? cluster_map(tempty0, 0) : tempty0;
    // Weight passes: the weight ring.  Step w (four per tile) of half h uses
    // slot 2 (w % WD) + h; one thread per half loads and stores that half's
    // chunks, loading each WD steps before it is used.
    constexpr bool WPASS = KIND >= G_UPDATE_W;
    constexpr int WD = w_depth_of(KIND);
    unsigned char* wring = side + 2 * kUSlotBytes;
    const bool wthread = WPASS && (ew & 3) == 1 && lane == 0;
    const int w_steps = 4 * (k_end - k_begin);
    int wstep = 0, w_issued = 0;
    const CUtensorMap* w_fenced = nullptr;
    // weights and the final output are touched once: keep the operands in L2 instead
    const uint64_t stream_policy = WPASS ? policy_evict_first() : 0ull;
    auto issue_w = [&](int w) {
      const TileGeom gw = tile_geom<KIND, CG>(args, k_begin + (w >> 2), rank);
      const CUtensorMap* mw = &gw.P->map_w;
      if (mw != w_fenced) {
        fence_tensormap(mw);
        w_fenced = mw;
      }
      const int slot = 2 * (w % WD) + ch;
      const uint32_t bar = wfull0 + 8 * slot;
      mbar_expect_tx(bar, kWChunkBytes);
      tma_load_2d_hint(smem_u32(wring + slot * kWChunkBytes), mw, bar, gw.col0 + 32 * (2 * (w & 3) + ch), gw.row0,
                       stream_policy);
    };
    if (wthread)
      while (w_issued < WD && w_issued < w_steps) issue_w(w_issued++);
    int ti = 0;
    for (int tile = k_begin; tile < k_end; ++tile, ++ti) {
      const TileGeom g = tile_geom<KIND, CG>(args, tile, rank);
      const NsProb& P = *g.P;
      const int r = g.row0 + quarter * 32 + lane;   // this thread's output row
      const int acc = ti & 1, use = ti >> 1;
      // G_POLY: this thread's A values for the b A term (its row, the four
      // 32-column chunks of its warp's half of the tile) are loaded before the
      // accumulator is ready, so their latency overlaps the tensor cores; a
      // chunk that crosses the matrix edge is read element by element when used
      uint4 apre[4][4];
      if (KIND == G_POLY) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int cb = g.col0 + 128 * ch + 32 * j;
          if (r < g.M_ && cb + 32 <= g.M_) {
            const uint4* q = reinterpret_cast<const uint4*>(P.a + (int64_t)r * P.ab_ld + cb);
#pragma unroll
            for (int i = 0; i < 4; ++i) apre[j][i] = __ldg(q + i);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) apre[j][i] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      bool ok = mbar_wait(tfull0 + 8 * acc, use & 1, args.hdr, 0x400u | KIND);
      tc_fence_after();
      ok = ok && *reinterpret_cast<volatile unsigned*>(&args.hdr->error) == 0u;
      // the staging of the update and polynomial products is per warp: it is
      // free again once this warp's stores of the previous tile have read it.
      // tcgen05.ld is warp-collective, so a warp continues or stops as one;
      // the Gram and the weight passes stage through shared barriers, and all
      // their epilogue warps continue or stop together
      constexpr bool WARP_LOCAL = (KIND == G_UPDATE || KIND == G_POLY);
      if (WARP_LOCAL && lane == 0 && ti > 0) bulk_wait_read_all();
      if (WARP_LOCAL ? !__all_sync(0xffffffffu, ok) : !epilogue_all(ok)) break;
      float s_first = 1.0f;
      if (args.first && P.inv) {
        const float iv = *P.inv;
        s_first = (KIND == G_GRAM) ? iv * iv : iv;
      }
      const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);

      if (KIND == G_UPDATE) {
        // X <- s3 (B X), warp by warp: this warp's 32 rows (its TMEM lane
        // quarter) and 128 columns (its half) leave through its own 4 KB of
        // staging, one 32 x 64 TMA box at a time (128-byte swizzle: 16-byte
        // chunk q of row r at q ^ (r & 7)), by its own TMA stores.  The four
        // TMEM loads are in flight together.
        const CUtensorMap* mo = &P.map_x32[args.dst];
        uint32_t v[4][32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32_async(tbase + (uint32_t)((4 * ch + cc) * 32), v[cc]);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_hold(v[cc]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (CG == 2) mbar_arrive_cluster(tempty_l + 8 * acc);
          else mbar_arrive(tempty0 + 8 * acc);
        }
        unsigned char* wst = side + ew * 4096;
        const int y = g.row0 + 32 * quarter;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          if (b == 1) {   // the first box's store has read the staging
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int cc = 2 * b + h;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int q = 4 * h + t;
              const uint32_t* u = v[cc] + 8 * t;
              *reinterpret_cast<uint4*>(wst + lane * 128 + ((q ^ (lane & 7)) << 4)) =
                  make_uint4(pack_bf16(s_first * __uint_as_float(u[0]), s_first * __uint_as_float(u[1])),
                             pack_bf16(s_first * __uint_as_float(u[2]), s_first * __uint_as_float(u[3])),
                             pack_bf16(s_first * __uint_as_float(u[4]), s_first * __uint_as_float(u[5])),
                             pack_bf16(s_first * __uint_as_float(u[6]), s_first * __uint_as_float(u[7])));
            }
          }
          // a box outside the matrix is skipped, a partial one is clipped by
          // the tensor map
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int x = g.col0 + 128 * ch + 64 * b;
            if (y < g.M_ && x < g.N_) tma_store_2d(mo, smem_u32(wst), x, y);
            bulk_commit();
          }
        }
      } else if (KIND == G_GRAM) {
        // the Gram A = s1^2 (X X^T) on a SYRK tile, in four steps of 64
        // columns: at step st, half h of the epilogue warps takes column chunk
        // c = 2 st + h.  The step's 128 x 64 block is staged in TMA box layout
        // (two 64 x 64 boxes, 128-byte swizzle) in one of two buffers,
        // alternately; one thread TMA-stores it and, before a buffer is
        // written again, waits until the stores of two steps ago have read
        // it.  (Warp-local staging, as in the other products, measured no
        // better for these long-K tiles.)  Only tiles on or above the diagonal
        // are computed and stored: the readers of A and B take the blocks
        // below it transposed from above.
        const CUtensorMap* mo = &P.map_a;
        const int m = g.M_;
        const int rl = quarter * 32 + lane;   // this thread's row of the tile
#pragma unroll
        for (int st = 0; st < 4; ++st) {
          const int c = 2 * st + ch;
          uint32_t v[32];
          tmem_ld32(tbase + (uint32_t)(c * 32), v);
          if (st == 3) {   // every TMEM read of this accumulator is done
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (CG == 2) mbar_arrive_cluster(tempty_l + 8 * acc);
              else mbar_arrive(tempty0 + 8 * acc);
            }
          }
          float out[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) out[i] = s_first * __uint_as_float(v[i]);
          // this step's buffer is free once the stores of two steps ago have read it
          unsigned char* sd = side + (st & 1) * 2 * kBox;   // boxes of rows 0-63 and 64-127
          if (ew == 0 && lane == 0 && (st > 0 || ti > 0)) bulk_wait_read_but1();
          __syncwarp();
          named_barrier_epilogue();
          unsigned char* drow = sd + (rl >> 6) * kBox + (rl & 63) * 128;
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int q = ch * 4 + t;
            *reinterpret_cast<uint4*>(drow + ((q ^ (rl & 7)) << 4)) =
                make_uint4(pack_bf16(out[8 * t], out[8 * t + 1]), pack_bf16(out[8 * t + 2], out[8 * t + 3]),
                           pack_bf16(out[8 * t + 4], out[8 * t + 5]), pack_bf16(out[8 * t + 6], out[8 * t + 7]));
          }
          fence_proxy_async_smem();
          named_barrier_epilogue();
          if (ew == 0 && lane == 0) {
            const int cs = g.col0 + 64 * st;
            if (cs < m) {
#pragma unroll
              for (int b = 0; b < 2; ++b) {
                if (g.row0 + 64 * b < m) tma_store_2d(mo, smem_u32(sd + b * kBox), cs, g.row0 + 64 * b);
              }
            }
            bulk_commit();
          }
        }
      } else if (WPASS) {
        // X <- s3 (B X) and W <- W - eta * bf16(X), in four steps of 64
        // columns: at step s, half h of the epilogue warps takes column chunk
        // c = 2 s + h.  The step's output columns go to an output slot (two
        // 64 x 64 boxes) and leave by TMA; the chunk's weights arrive by TMA
        // in a ring slot, are updated in place and leave by TMA.
        const int rl = quarter * 32 + lane;
        for (int st = 0; st < 4; ++st, ++wstep) {
          const int c = 2 * st + ch;
          const int slot = 2 * (wstep % WD) + ch;
          const bool wok = mbar_wait(wfull0 + 8 * slot, (wstep / WD) & 1, args.hdr, 0x900u | KIND);
          __syncwarp();   // tcgen05.ld is warp-collective: the lane back from its single-thread role rejoins
          uint32_t v[32];
          tmem_ld32(tbase + (uint32_t)(c * 32), v);
          if (st == 3) {   // every TMEM read of this accumulator is done
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (CG == 2) mbar_arrive_cluster(tempty_l + 8 * acc);
              else mbar_arrive(tempty0 + 8 * acc);
            }
          }
          float out[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) out[i] = s_first * __uint_as_float(v[i]);
          unsigned char* ub = side + (wstep & 1) * kUSlotBytes + (rl >> 6) * kBox + (rl & 63) * 128;
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int q = ch * 4 + t;
            *reinterpret_cast<uint4*>(ub + ((q ^ (rl & 7)) << 4)) =
                make_uint4(pack_bf16(out[8 * t], out[8 * t + 1]), pack_bf16(out[8 * t + 2], out[8 * t + 3]),
                           pack_bf16(out[8 * t + 4], out[8 * t + 5]), pack_bf16(out[8 * t + 6], out[8 * t + 7]));
          }
          if (wok) {
            // this thread's 32 weights: one rounded product and one rounded
            // difference per element (128-byte swizzle, like the boxes above)
            unsigned char* wb = wring + slot * kWChunkBytes + rl * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              float4* pw = reinterpret_cast<float4*>(wb + ((j ^ (rl & 7)) << 4));
              float4 w4 = *pw;
              float* e = reinterpret_cast<float*>(&w4);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float u = __bfloat162float(__float2bfloat16_rn(out[4 * j + k]));
                e[k] = __fsub_rn(e[k], __fmul_rn(args.eta, u));
              }
              *pw = w4;
            }
          }
          fence_proxy_async_smem();
          // the output slot written now was last stored two steps ago: its
          // store has read it once the storing thread passes this point
          if (ew == 0 && lane == 0) bulk_wait_read_all();
          __syncwarp();
          named_barrier_epilogue();
          if (ew == 0 && lane == 0) {
            const CUtensorMap* md = &P.map_x[args.dst];
            const uint32_t us = smem_u32(side + (wstep & 1) * kUSlotBytes);
#pragma unroll
            for (int bi = 0; bi < 2; ++bi)
              if (g.row0 + 64 * bi < g.M_ && g.col0 + 64 * st < g.N_)
                tma_store_2d_hint(md, us + bi * kBox, g.col0 + 64 * st, g.row0 + 64 * bi, stream_policy);
            bulk_commit();
          }
          if (wthread) {
            const bool clean = *reinterpret_cast<volatile unsigned*>(&args.hdr->error) == 0u;
            if (wok && clean && g.row0 < g.M_ && g.col0 + 32 * c < g.N_)
              tma_store_2d_hint(&P.map_w, smem_u32(wring + slot * kWChunkBytes), g.col0 + 32 * c, g.row0,
                                stream_policy);
            bulk_commit();
            bulk_wait_read_all();   // the slot is free for the chunk WD steps ahead
            if (clean && w_issued < w_steps) issue_w(w_issued++);
          }
        }
      } else {
        // B = a I + b A + c A^2 on a SYRK tile, warp by warp as above, one
        // 32-column TMEM load at a time (the b A term's values already take
        // 64 registers), two chunks to a 32 x 64 box.  Only tiles on or above
        // the diagonal are computed and stored: the readers of A and B take
        // the blocks below it transposed from above.
        const int m = g.M_;
        unsigned char* wst = side + ew * 4096;
        const int y = g.row0 + 32 * quarter;
        // element (row r, column c) of B, with a on the diagonal (the a X
        // term of the update)
        auto poly = [&](float a, uint32_t acc_bits, int c) {
          return args.cb * a + args.cc * __uint_as_float(acc_bits) + (c == r ? args.ca : 0.0f);
        };
#pragma unroll
        for (int j = 0; j < 4; ++j) {   // 32-column chunk j of the warp's half
          uint32_t v[32];
          tmem_ld32(tbase + (uint32_t)((4 * ch + j) * 32), v);
          if (j == 3) {   // every TMEM read of this accumulator is done
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (CG == 2) mbar_arrive_cluster(tempty_l + 8 * acc);
              else mbar_arrive(tempty0 + 8 * acc);
            }
          }
          if (j == 2) {   // the first box's store has read the staging
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
          }
          const int cb = g.col0 + 128 * ch + 32 * j;
          const int h = j & 1;
          if (r < m && cb < m && cb + 32 > m) {
            // a chunk that crosses the matrix edge, read element by element
            float av[32];
            load_row32(P.a + (int64_t)r * P.ab_ld + cb, m - cb, av);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              uint32_t w[4];
#pragma unroll
              for (int k = 0; k < 4; ++k)
                w[k] = pack_bf16(poly(av[8 * t + 2 * k], v[8 * t + 2 * k], cb + 8 * t + 2 * k),
                                 poly(av[8 * t + 2 * k + 1], v[8 * t + 2 * k + 1], cb + 8 * t + 2 * k + 1));
              *reinterpret_cast<uint4*>(wst + lane * 128 + (((4 * h + t) ^ (lane & 7)) << 4)) =
                  make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const uint4 u = apre[j][t];
              const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
              uint32_t w[4];
#pragma unroll
              for (int k = 0; k < 4; ++k)
                w[k] = pack_bf16(poly(bf16_lo(uw[k]), v[8 * t + 2 * k], cb + 8 * t + 2 * k),
                                 poly(bf16_hi(uw[k]), v[8 * t + 2 * k + 1], cb + 8 * t + 2 * k + 1));
              *reinterpret_cast<uint4*>(wst + lane * 128 + (((4 * h + t) ^ (lane & 7)) << 4)) =
                  make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
          if (h == 1) {   // the box (chunks j - 1 and j) is staged: store it
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int x = g.col0 + 128 * ch + 32 * (j - 1);
              if (y < m && x < m) tma_store_2d(&P.map_b32, smem_u32(wst), x, y);
              bulk_commit();
            }
          }
        }
      }
    }
    // weight chunks loaded but never used (the run stopped early) land before exit
    if (wthread)
      for (int w = wstep; w < w_issued; ++w)
        mbar_wait(wfull0 + 8 * (2 * (w % WD) + ch), (w / WD) & 1, args.hdr, 0xA00u | KIND);
  }

  // ---- teardown: every accumulator read is done, every TMA store has
  // completed and, in a pair, the peer no longer touches this CTA's barriers
  // or shared memory ----
  if (warp >= 2 && lane == 0) bulk_wait_all();
  tc_fence_before();
  __syncwarp();   // lanes that skipped the single-thread roles rejoin before the aligned barrier
  if (CG == 2) cluster_sync_all();
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_cg<CG>(tmem, kTmemCols);
  }
}

// MXFP8 carrier -> bf16 Newton-Schulz input: x[r][c] = E4M3(payload[r][c]) *
// 2^(scale[r][c/32] - 127).  An E4M3 value has at most 4 significant bits, so
// the product with a power of two is exact in bf16 (within bf16's exponent
// range); the carrier is consumed as it is, the inverse norm is applied later
// by the first iteration.  One thread per 16 payload bytes.
// One carrier to expand: rows x cols E4M3 codes and E8M0 row-block scales into
// a bf16 matrix with row stride ld; its 16-element vectors are numbered from
// vec_begin in the launch.
struct DecodeItem {
  const uint8_t* payload;
  const uint8_t* scale;
  __nv_bfloat16* x;
  int64_t rows, cols, ld;
  int64_t vec_begin;
};

// Vector v (16 payload bytes of one row) of one carrier.
__device__ __forceinline__ void decode_vec(const DecodeItem& it, int64_t v) {
  const int64_t per_row = it.cols / 16;
  const int64_t r = v / per_row, c0 = (v % per_row) * 16;
  const uint4 p = *reinterpret_cast<const uint4*>(it.payload + r * it.cols + c0);
  const int e = (int)it.scale[r * (it.cols / 32) + c0 / 32] - 127;
  // 2^e as fp32 (e in [-127, 127]; 2^-127 is the subnormal 0x00400000)
  const float mult = e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
  const uint32_t w[4] = {p.x, p.y, p.z, p.w};
  uint32_t o[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      // two E4M3 codes -> two halves (exact), then fp32, scale, bf16
      const unsigned short pair = (unsigned short)((w[k] >> (16 * h)) & 0xFFFFu);
      uint32_t hh;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hh) : "h"(pair));
      const __half2 hv = *reinterpret_cast<const __half2*>(&hh);
      const float lo = __fmul_rn(__low2float(hv), mult), hi = __fmul_rn(__high2float(hv), mult);
      o[2 * k + h] = pack_bf16(lo, hi);
    }
  }
  uint4* dst = reinterpret_cast<uint4*>(it.x + r * it.ld + c0);
  dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
  dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// Every carrier of a batch in one launch: thread-strided over all vectors;
// a thread finds its first carrier by bisection and then only moves forward.
__global__ void decode_carriers_kernel(const DecodeItem* __restrict__ items, int32_t n, int64_t total) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= total) return;
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (items[mid].vec_begin <= v) lo = mid;
    else hi = mid - 1;
  }
  for (int k = lo; v < total; v += stride) {
    while (k + 1 < n && items[k + 1].vec_begin <= v) ++k;
    decode_vec(items[k], v - items[k].vec_begin);
  }
}

// Copy the workspace result back to the caller's matrix (single-iteration runs).
__global__ void copy_back_kernel(const NsProb* probs, int32_t p, int32_t from) {
  const NsProb& P = probs[p];
  const int64_t total = (int64_t)P.rows * P.cols;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / P.cols, c = i % P.cols;
    P.x[0][r * P.x_ld[0] + c] = P.x[from][r * P.x_ld[from] + c];
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    const cudaError_t e =
        cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (e == cudaSuccess && q == cudaDriverEntryPointSuccess && p) {
      fn = reinterpret_cast<EncodeTiledFn>(p);
    } else {
      char msg[160];
      std::snprintf(msg, sizeof(msg), "driver entry point cuTensorMapEncodeTiled: %s, query result %d",
                    cudaGetErrorString(e), (int)q);
      set_error_msg(msg, QMUON_ERR_CUDA);
    }
  }
  return fn;
}

// 2-D bf16 map (rows x cols, row stride ld elements), boxes of 64 columns x
// box_rows rows, 128-byte swizzle.
bool encode_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, uint32_t box_rows = 64) {
  EncodeTiledFn fn = encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char msg[256];
    std::snprintf(msg, sizeof(msg),
                  "cuTensorMapEncodeTiled returned %d for a %lld x %lld bf16 matrix (row stride %lld) at %p, map at %p",
                  (int)r, (long long)rows, (long long)cols, (long long)ld, base, (void*)m);
    set_error_msg(msg, QMUON_ERR_CUDA);
    return false;
  }
  return true;
}

// 2-D fp32 map of the weights (rows x cols, row stride ld elements), boxes of
// 32 columns x 128 rows (128-byte rows, 128-byte swizzle).
bool encode_w(CUtensorMap* m, const float* base, int64_t rows, int64_t cols, int64_t ld) {
  EncodeTiledFn fn = encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
  cuuint32_t box[2] = {32, 128};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char msg[256];
    std::snprintf(msg, sizeof(msg),
                  "cuTensorMapEncodeTiled returned %d for a %lld x %lld fp32 weight matrix (row stride %lld) at %p",
                  (int)r, (long long)rows, (long long)cols, (long long)ld, (const void*)base);
    set_error_msg(msg, QMUON_ERR_CUDA);
    return false;
  }
  return true;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shape of one problem's scratch: A and B (m x m) and two X buffers (rows x cols, compact).
struct Shape {
  int64_t rows, cols;
};
size_t scratch_bytes(const Shape& s) {
  const int64_t m = std::min(s.rows, s.cols);
  const int64_t ld = (m + 7) / 8 * 8;
  return 2 * align_up((size_t)(m * ld) * 2, 256) + 2 * align_up((size_t)(s.rows * s.cols) * 2, 256);
}

// Output tiles of a rows x cols problem per product kind.  Tiles are
// (128 kCG) x 256; the symmetric products list only tiles touching the upper
// triangle (kCG = 1: 128 I < 256 J + 256; kCG = 2: I <= J).
void count_tiles(int64_t rows, int64_t cols, int32_t tiles_n[3], int32_t tiles[3]) {
  const int64_t m = std::min(rows, cols), n = std::max(rows, cols);
  const int64_t tile_m = 128 * kCG;
  const int64_t tm = (m + tile_m - 1) / tile_m, tnm = (m + BN - 1) / BN;
  int64_t sym = 0;
  for (int64_t j = 0; j < tnm; ++j) sym += std::min<int64_t>(tm, kCG == 2 ? j + 1 : 2 * j + 2);
  tiles_n[G_GRAM] = tiles_n[G_POLY] = (int32_t)tnm;
  tiles[G_GRAM] = tiles[G_POLY] = (int32_t)sym;
  const bool tall = rows > cols;
  const int64_t um = tall ? n : m, un = tall ? m : n;   // G_UPDATE output (stored orientation)
  tiles_n[G_UPDATE] = (int32_t)((un + BN - 1) / BN);
  tiles[G_UPDATE] = (int32_t)(((um + tile_m - 1) / tile_m) * tiles_n[G_UPDATE]);
}

constexpr int kMaxGroups = 512;   // schedule capacity: CTA groups per launch
constexpr int kLightM = 768;      // problems with a short side up to this are DRAM-bound per tile

// Device table of a problem set: the problems, then per product kind the
// group starts [kMaxGroups + 1] and the schedule entries.
size_t table_bytes(int32_t n, const int64_t total_tiles) {
  return align_up((size_t)n * sizeof(NsProb), 256) + 3 * align_up((size_t)(kMaxGroups + 1) * 4, 256) +
         align_up((size_t)total_tiles * 8, 256);
}

// Fill one problem: x0 is the caller's matrix (row stride ld), scratch is carved from `ws`.
bool fill_problem(NsProb& P, void* x0, int64_t rows, int64_t cols, int64_t ld, const float* inv, float* w,
                  int64_t w_ld, unsigned char*& ws) {
  std::memset(&P, 0, sizeof(P));
  P.rows = (int32_t)rows;
  P.cols = (int32_t)cols;
  P.tall = rows > cols;
  P.m = (int32_t)std::min(rows, cols);
  P.n = (int32_t)std::max(rows, cols);
  const int64_t m = P.m;
  P.ab_ld = (m + 7) / 8 * 8;
  P.a = reinterpret_cast<__nv_bfloat16*>(ws);
  ws += align_up((size_t)(m * P.ab_ld) * 2, 256);
  P.b = reinterpret_cast<__nv_bfloat16*>(ws);
  ws += align_up((size_t)(m * P.ab_ld) * 2, 256);
  P.x[0] = static_cast<__nv_bfloat16*>(x0);
  P.x_ld[0] = ld;
  for (int i = 1; i < 3; ++i) {
    P.x[i] = reinterpret_cast<__nv_bfloat16*>(ws);
    P.x_ld[i] = cols;
    ws += align_up((size_t)(rows * cols) * 2, 256);
  }
  P.inv = inv;
  P.w = w;
  P.w_ld = w_ld;
  for (int i = 0; i < 3; ++i)
    if (!encode_bf16(&P.map_x[i], P.x[i], rows, cols, P.x_ld[i]) ||
        !encode_bf16(&P.map_x32[i], P.x[i], rows, cols, P.x_ld[i], 32))
      return false;
  if (!encode_bf16(&P.map_a, P.a, m, m, P.ab_ld) || !encode_bf16(&P.map_b, P.b, m, m, P.ab_ld) ||
      !encode_bf16(&P.map_b32, P.b, m, m, P.ab_ld, 32))
    return false;
  if (w && !encode_w(&P.map_w, w, rows, cols, w_ld)) return false;
  count_tiles(rows, cols, P.tiles_n, P.tiles);
  return true;
}

// Host facts and setup kept per device, for a process that drives several.
constexpr int kDeviceSlots = 64;

int current_device() {
  int dev = 0;
  return cudaGetDevice(&dev) == cudaSuccess ? dev : -1;
}

int num_sms() {
  static std::atomic<int> cached[kDeviceSlots];
  const int dev = current_device();
  const bool slot = dev >= 0 && dev < kDeviceSlots;
  int n = slot ? cached[dev].load(std::memory_order_relaxed) : 0;
  if (n == 0) {
    if (dev < 0 || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    if (slot) cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

struct Launchable {
  NsProb* d_probs = nullptr;
  int32_t* d_sched_start[3] = {nullptr, nullptr, nullptr};   // [groups + 1] per kind
  TileRef* d_sched[3] = {nullptr, nullptr, nullptr};
  int32_t n = 0;
  int32_t total[3] = {0, 0, 0};
  int32_t groups[3] = {0, 0, 0};
  // the update tiles' K loops are long on average (>= 2048): the weight pass
  // then hides behind the tensor cores and runs with more operand stages
  bool long_k = false;
};

// Relative cost of one output tile: its K loop in 64-wide steps plus the
// epilogue, which overlaps the next tile's loop only in part.
int64_t tile_cost(const NsProb& P, int kind) {
  const int64_t K = (kind == G_GRAM) ? P.n : P.m;
  return (K + BK - 1) / BK + 4;
}

// Host-side schedule of each product kind: tiles are dealt, costliest first,
// to the least-loaded CTA group (longest processing time first); each group
// then runs its tiles in that order.  The schedule and the problem table go
// to `table` (device memory) with one copy each.
struct Schedule {
  std::vector<int32_t> start[3];
  std::vector<TileRef> entries[3];
};

void build_schedule(const std::vector<NsProb>& probs, int groups_cap, Launchable& L, Schedule& S) {
  for (int kind = 0; kind < 3; ++kind) {
    std::vector<std::pair<int64_t, TileRef>> tiles;
    for (int32_t p = 0; p < (int32_t)probs.size(); ++p) {
      const int64_t c = tile_cost(probs[p], kind);
      for (int32_t t = 0; t < probs[p].tiles[kind]; ++t) tiles.push_back({c, TileRef{p, t}});
    }
    const int32_t total = (int32_t)tiles.size();
    const int groups = std::max(1, std::min<int>(total, groups_cap));
    std::stable_sort(tiles.begin(), tiles.end(),
                     [](const std::pair<int64_t, TileRef>& a, const std::pair<int64_t, TileRef>& b) {
                       return a.first > b.first;
                     });
    // least-loaded group first, the lower index among equals
    std::vector<std::pair<int64_t, int>> heap;
    for (int g = 0; g < groups; ++g) heap.push_back({0, g});
    auto later = [](const std::pair<int64_t, int>& a, const std::pair<int64_t, int>& b) {
      return a.first != b.first ? a.first > b.first : a.second > b.second;
    };
    std::make_heap(heap.begin(), heap.end(), later);
    std::vector<std::vector<TileRef>> lists(groups);
    for (const auto& t : tiles) {
      std::pop_heap(heap.begin(), heap.end(), later);
      auto& h = heap.back();
      lists[h.second].push_back(t.second);
      h.first += t.first;
      std::push_heap(heap.begin(), heap.end(), later);
    }
    // A group's load does not depend on the order of its tiles.  Tiles of
    // problems with a short side above kLightM are bound by the tensor cores,
    // those at or below it by DRAM (their K loops are short and every tile
    // streams its own X panel); each group runs them interleaved in
    // proportion to their cost, so that at any time the groups together
    // draw on both instead of running one kind after the other.
    for (auto& lst : lists) {
      std::vector<TileRef> heavy, light;
      int64_t ht = 0, lt = 0;
      for (const TileRef& t : lst) {
        const int64_t c = tile_cost(probs[t.prob], kind);
        if (probs[t.prob].m > kLightM) {
          heavy.push_back(t);
          ht += c;
        } else {
          light.push_back(t);
          lt += c;
        }
      }
      if (heavy.empty() || light.empty()) continue;
      lst.clear();
      size_t i = 0, j = 0;
      int64_t h = 0, l = 0;
      while (i < heavy.size() || j < light.size()) {
        // the kind whose done fraction of its cost is behind goes next
        if (j == light.size() || (i < heavy.size() && h * lt <= l * ht)) {
          h += tile_cost(probs[heavy[i].prob], kind);
          lst.push_back(heavy[i++]);
        } else {
          l += tile_cost(probs[light[j].prob], kind);
          lst.push_back(light[j++]);
        }
      }
    }
    S.start[kind].assign(1, 0);
    S.entries[kind].clear();
    for (int g = 0; g < groups; ++g) {
      S.entries[kind].insert(S.entries[kind].end(), lists[g].begin(), lists[g].end());
      S.start[kind].push_back((int32_t)S.entries[kind].size());
    }
    L.total[kind] = total;
    L.groups[kind] = total ? groups : 0;
    if (kind == G_UPDATE) {
      double sum_k = 0.0;
      for (const auto& t : tiles) sum_k += probs[t.second.prob].m;
      L.long_k = total > 0 && sum_k >= 2048.0 * total;
    }
  }
}

// Carve the schedule arrays out of a table laid out as `table_bytes` says.
void carve_table(unsigned char* table, int32_t n, Launchable& L) {
  L.n = n;
  L.d_probs = reinterpret_cast<NsProb*>(table);
  unsigned char* p = table + align_up((size_t)n * sizeof(NsProb), 256);
  for (int k = 0; k < 3; ++k) {
    L.d_sched_start[k] = reinterpret_cast<int32_t*>(p);
    p += align_up((size_t)(kMaxGroups + 1) * 4, 256);
  }
  TileRef* e = reinterpret_cast<TileRef*>(p);
  for (int k = 0; k < 3; ++k) {
    L.d_sched[k] = e;
    e += L.total[k];
  }
}

// The copies of the problem table and the schedule (stream-ordered when `s`
// is given, else synchronous).
cudaError_t upload_table(const Launchable& L, const std::vector<NsProb>& hp, const Schedule& S, cudaStream_t s,
                         bool async) {
  auto copy = [&](void* dst, const void* src, size_t bytes) {
    if (bytes == 0) return cudaSuccess;
    return async ? cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, s)
                 : cudaMemcpy(dst, src, bytes, cudaMemcpyHostToDevice);
  };
  cudaError_t e = copy(L.d_probs, hp.data(), hp.size() * sizeof(NsProb));
  for (int k = 0; k < 3 && e == cudaSuccess; ++k) {
    e = copy(L.d_sched_start[k], S.start[k].data(), S.start[k].size() * 4);
    if (e == cudaSuccess) e = copy(L.d_sched[k], S.entries[k].data(), S.entries[k].size() * sizeof(TileRef));
  }
  return e;
}

int64_t all_tiles(int64_t rows, int64_t cols) {
  int32_t tn[3], t[3];
  count_tiles(rows, cols, tn, t);
  return (int64_t)t[0] + t[1] + t[2];
}

// The dynamic shared memory opt-in of every kernel variant, once per device.
cudaError_t configure_kernels() {
  static std::atomic<bool> done[kDeviceSlots];
  const int dev = current_device();
  const bool slot = dev >= 0 && dev < kDeviceSlots;
  if (slot && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  {
    const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
    cudaError_t e = cudaFuncSetAttribute(ns_gemm_kernel<G_GRAM, kCG>, attr, (int)smem_bytes_of(G_GRAM, kCG));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ns_gemm_kernel<G_POLY, kCG>, attr, (int)smem_bytes_of(G_POLY, kCG));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ns_gemm_kernel<G_UPDATE, kCG>, attr, (int)smem_bytes_of(G_UPDATE, kCG));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(ns_gemm_kernel<G_UPDATE_W, kCG>, attr, (int)smem_bytes_of(G_UPDATE_W, kCG));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(ns_gemm_kernel<G_UPDATE_W1, kCG>, attr, (int)smem_bytes_of(G_UPDATE_W1, kCG));
    if (e != cudaSuccess) return e;
  }
  if (slot) done[dev].store(true, std::memory_order_release);
  return cudaSuccess;
}

cudaError_t launch_gemm(int kind, const Launchable& L, const GemmArgs& a0, cudaStream_t s) {
  const int sk = kind >= G_UPDATE_W ? G_UPDATE : kind;   // the weight passes run the update's tiles
  if (L.total[sk] == 0) return cudaSuccess;
  GemmArgs a = a0;
  a.sched_start = L.d_sched_start[sk];
  a.sched = L.d_sched[sk];
  void* args[] = {&a};
  void* fn = kind == G_GRAM ? (void*)ns_gemm_kernel<G_GRAM, kCG>
           : kind == G_POLY ? (void*)ns_gemm_kernel<G_POLY, kCG>
           : kind == G_UPDATE ? (void*)ns_gemm_kernel<G_UPDATE, kCG>
           : kind == G_UPDATE_W ? (void*)ns_gemm_kernel<G_UPDATE_W, kCG> : (void*)ns_gemm_kernel<G_UPDATE_W1, kCG>;
  // persistent: one CTA group per SM group, never more groups than tiles
  const int groups = L.groups[sk];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(groups * kCG);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes_of(kind, kCG);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch (the kernel waits on griddepcontrol.wait
  // before it touches anything an earlier kernel of the stream wrote)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// The iteration schedule over X buffers: 0 -> 1 -> 2 -> 1 -> ... and the last
// iteration writes back into buffer 0 (its source is never 0 when iters >= 2).
qmuon_status run_iterations(const Launchable& L, int32_t iters, const float coeffs[3], float eta, bool apply_w,
                            WsHeader* hdr, cudaStream_t s, const std::vector<NsProb>& host_probs) {
  const cudaError_t ce = configure_kernels();
  if (ce != cudaSuccess) return set_error("newton-schulz: cudaFuncSetAttribute(max dynamic shared memory)", ce);
  GemmArgs a{};
  a.probs = L.d_probs;
  a.ca = coeffs[0];
  a.cb = coeffs[1];
  a.cc = coeffs[2];
  a.eta = eta;
  a.hdr = hdr;
  int src = 0;
  for (int32_t it = 0; it < iters; ++it) {
    const bool last = (it == iters - 1);
    const int dst = (last && iters >= 2) ? 0 : 1 + (it % 2);
    a.src = src;
    a.dst = dst;
    a.first = (it == 0);
    cudaError_t e = launch_gemm(G_GRAM, L, a, s);
    if (e == cudaSuccess) e = launch_gemm(G_POLY, L, a, s);
    if (e == cudaSuccess) e = launch_gemm((last && apply_w) ? (L.long_k ? G_UPDATE_W1 : G_UPDATE_W) : G_UPDATE, L, a, s);
    if (e != cudaSuccess) return set_error("newton-schulz: cudaLaunchKernel(ns_gemm)", e);
    src = dst;
  }
  if (src != 0) {
    for (int32_t p = 0; p < L.n; ++p) {
      copy_back_kernel<<<256, 256, 0, s>>>(L.d_probs, p, src);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error("newton-schulz: copy-back launch", e);
  }
  (void)host_probs;
  return QMUON_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// qmuon_newton_schulz_batched
// ---------------------------------------------------------------------------
qmuon_status validate_problem(const qmuon_ns_problem& p) {
  if (p.rows <= 0 || p.cols <= 0 || p.rows > (1 << 30) || p.cols > (1 << 30)) return QMUON_ERR_INVALID_ARGUMENT;
  if (p.input != QMUON_NS_BF16 && p.input != QMUON_NS_MXFP8) return QMUON_ERR_INVALID_ARGUMENT;
  if (!p.x || (reinterpret_cast<uintptr_t>(p.x) & 15)) return QMUON_ERR_INVALID_ARGUMENT;
  if (p.ld < p.cols) return QMUON_ERR_INVALID_ARGUMENT;
  if (p.ld % 8 || p.cols % 8) return QMUON_ERR_UNSUPPORTED;
  if (p.inv_norm && (reinterpret_cast<uintptr_t>(p.inv_norm) & 3)) return QMUON_ERR_INVALID_ARGUMENT;
  if (p.input == QMUON_NS_MXFP8) {
    if (!p.payload || !p.scale_inv || (reinterpret_cast<uintptr_t>(p.payload) & 15)) return QMUON_ERR_INVALID_ARGUMENT;
    if (p.cols % 32) return QMUON_ERR_UNSUPPORTED;
  }
  return QMUON_OK;
}

size_t batch_table_bytes(const qmuon_ns_problem* probs, int32_t n) {
  int64_t tiles = 0;
  for (int32_t i = 0; i < n; ++i) tiles += all_tiles(probs[i].rows, probs[i].cols);
  return table_bytes(n, tiles) + align_up((size_t)n * sizeof(DecodeItem), 256);   // + the carriers to expand
}

size_t batch_workspace_bytes(const qmuon_ns_problem* probs, int32_t n) {
  size_t b = batch_table_bytes(probs, n);
  for (int32_t i = 0; i < n; ++i) b += scratch_bytes({probs[i].rows, probs[i].cols});
  return b;
}

qmuon_status run_batch(const qmuon_ns_problem* probs, int32_t n, int32_t iters, const float coeffs[3],
                       WsHeader* hdr, unsigned char* ws, size_t ws_bytes, cudaStream_t s) {
  if (!encoder()) return set_error_msg("cuTensorMapEncodeTiled not available from the driver", QMUON_ERR_CUDA);
  std::vector<NsProb> hp(n);
  unsigned char* table = ws;
  unsigned char* scratch = ws + batch_table_bytes(probs, n);
  for (int32_t i = 0; i < n; ++i) {
    if (!fill_problem(hp[i], probs[i].x, probs[i].rows, probs[i].cols, probs[i].ld, probs[i].inv_norm, nullptr, 0,
                      scratch))
      return QMUON_ERR_CUDA;   // detail recorded by encode_bf16
  }
  if ((size_t)(scratch - ws) > ws_bytes) return QMUON_ERR_WORKSPACE_TOO_SMALL;
  Launchable L;
  Schedule S;
  build_schedule(hp, std::min(num_sms() / kCG, kMaxGroups), L, S);
  carve_table(table, n, L);
  cudaError_t ce = upload_table(L, hp, S, s, true);
  if (ce != cudaSuccess) return set_error("newton-schulz: upload problem table", ce);
  // MXFP8 inputs: every carrier expanded into its problem's bf16 matrix first, in one launch
  std::vector<DecodeItem> items;
  int64_t vecs = 0;
  for (int32_t i = 0; i < n; ++i) {
    if (probs[i].input != QMUON_NS_MXFP8) continue;
    items.push_back(DecodeItem{probs[i].payload, probs[i].scale_inv, static_cast<__nv_bfloat16*>(probs[i].x),
                               probs[i].rows, probs[i].cols, probs[i].ld, vecs});
    vecs += probs[i].rows * (probs[i].cols / 16);
  }
  if (!items.empty()) {
    DecodeItem* d_items = reinterpret_cast<DecodeItem*>(table + batch_table_bytes(probs, n) -
                                                        align_up((size_t)n * sizeof(DecodeItem), 256));
    ce = cudaMemcpyAsync(d_items, items.data(), items.size() * sizeof(DecodeItem), cudaMemcpyHostToDevice, s);
    if (ce != cudaSuccess) return set_error("newton-schulz: upload carrier list", ce);
    const int grid = (int)std::min<int64_t>((vecs + 255) / 256, (int64_t)num_sms() * 8);
    decode_carriers_kernel<<<grid, 256, 0, s>>>(d_items, (int32_t)items.size(), vecs);
    ce = cudaGetLastError();
    if (ce != cudaSuccess) return set_error("newton-schulz: carrier decode launch", ce);
  }
  const qmuon_status st = run_iterations(L, iters, coeffs, 0.0f, false, hdr, s, hp);
  // the pageable host vectors are staged by the copies above before they return
  return st;
}

// ---------------------------------------------------------------------------
// qmuon_step's problem sets
// ---------------------------------------------------------------------------
struct StepTables {
  Launchable L;
  void* d_mem = nullptr;
  size_t d_bytes = 0;
  std::vector<NsProb> host;
  // what the cached tables were built for
  unsigned char* ws = nullptr;
  size_t ws_bytes = 0;
  const float* inv = nullptr;
  std::vector<float*> weights;
  int32_t tile_r = 0, tile_c = 0;
};

size_t step_workspace_bytes(const qmuon_tensor* t, int32_t n, int32_t tile_r, int32_t tile_c) {
  size_t b = 0;
  for (int32_t i = 0; i < n; ++i) {
    if (t[i].rows * t[i].cols == 0) continue;
    const Shape sh{t[i].rows / tile_r, t[i].cols / tile_c};
    b += (size_t)tile_r * tile_c * scratch_bytes(sh);
  }
  return b;
}

qmuon_status ensure_step_tables(StepTables** tabs, const qmuon_tensor* t, int32_t n, int32_t tile_r, int32_t tile_c,
                                float* const* weights, const float* inv, unsigned char* ws, size_t ws_bytes,
                                bool ordered, cudaStream_t s) {
  StepTables* T = *tabs;
  if (T && T->ws == ws && T->ws_bytes == ws_bytes && T->inv == inv && T->tile_r == tile_r && T->tile_c == tile_c &&
      std::equal(T->weights.begin(), T->weights.end(), weights))
    return QMUON_OK;
  if (!encoder()) return set_error_msg("cuTensorMapEncodeTiled not available from the driver", QMUON_ERR_CUDA);
  std::vector<NsProb> hp;
  unsigned char* scratch = ws;
  int32_t g = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int64_t R = t[i].rows, C = t[i].cols;
    if (R * C == 0) continue;
    const int64_t th = R / tile_r, tw = C / tile_c;
    for (int32_t bi = 0; bi < tile_r; ++bi)
      for (int32_t bj = 0; bj < tile_c; ++bj, ++g) {
        NsProb P;
        const int64_t off = bi * th * C + bj * tw;
        void* x0 = static_cast<__nv_bfloat16*>(t[i].grad) + off;
        if (!fill_problem(P, x0, th, tw, C, inv + g, weights[i] + off, C, scratch))
          return QMUON_ERR_CUDA;   // detail recorded by encode_bf16
        hp.push_back(P);
      }
  }
  if ((size_t)(scratch - ws) > ws_bytes) return QMUON_ERR_WORKSPACE_TOO_SMALL;
  if (!T) {
    T = new StepTables;
    *tabs = T;
  } else if (!ordered) {
    // earlier steps, on any stream, may still read the tables rewritten below
    const cudaError_t se = cudaDeviceSynchronize();
    if (se != cudaSuccess) return set_error("qmuon_step_prepare: synchronize before rebuilding tables", se);
  }
  // From here until the rebuild completes the tables match no request, so a
  // rebuild that fails part-way is redone by the next call instead of reused.
  T->ws = nullptr;
  T->weights.clear();
  const int32_t np = (int32_t)hp.size();
  int64_t tiles = 0;
  for (const NsProb& P : hp) tiles += (int64_t)P.tiles[0] + P.tiles[1] + P.tiles[2];
  const size_t need = table_bytes(np, tiles);
  if (T->d_bytes < need) {
    if (T->d_mem) cudaFree(T->d_mem);
    T->d_mem = nullptr;
    T->d_bytes = 0;
    const cudaError_t me = cudaMalloc(&T->d_mem, need);
    if (me != cudaSuccess) return set_error("qmuon_step: cudaMalloc problem table", me);
    T->d_bytes = need;
  }
  Schedule S;
  build_schedule(hp, std::min(num_sms() / kCG, kMaxGroups), T->L, S);
  carve_table(static_cast<unsigned char*>(T->d_mem), np, T->L);
  const cudaError_t ue = upload_table(T->L, hp, S, s, ordered);
  if (ue != cudaSuccess) return set_error("qmuon_step: upload problem table", ue);
  T->host = std::move(hp);
  T->ws = ws;
  T->ws_bytes = ws_bytes;
  T->inv = inv;
  T->weights.assign(weights, weights + n);
  T->tile_r = tile_r;
  T->tile_c = tile_c;
  return QMUON_OK;
}

qmuon_status run_step(StepTables* tabs, int32_t iters, const float coeffs[3], float eta, WsHeader* hdr,
                      cudaStream_t s) {
  if (!tabs) return QMUON_ERR_INVALID_ARGUMENT;
  return run_iterations(tabs->L, iters, coeffs, eta, true, hdr, s, tabs->host);
}

void destroy_step_tables(StepTables* t) {
  if (!t) return;
  if (t->d_mem) cudaFree(t->d_mem);
  delete t;
}

}  // namespace ns
}  // namespace qm

// Blockwise 8-bit Muon momentum update for sm_103a.
//
// Implements "Quantized Muon Momentum", section "Algorithm", steps 1-9, over
// many tensors in one launch (section "What Exists": the multi-tensor in-place
// update, the fused sum of squares, the grouped normalisation of section
// "Grouped QKV And Sharding"), and the MXFP8 carrier of section "Wave18B
// MXFP8 Carrier Probe".
//
// Layout on the GPU: a CTA owns a contiguous chunk of quantization blocks
// (the grid is a whole number of waves of resident CTAs).  Its producer warp
// streams the chunk through a ring of four shared-memory stages of 16 blocks:
// one bulk asynchronous copy per tensor segment for the codes and one for the
// gradient, and a 4-byte asynchronous copy per block for the old absmax, all
// counted on the stage's mbarrier.  Its eight compute warps take one block
// per half-warp and stage: a lane reads its 16 consecutive elements (16 bytes
// of codes, 32 or 64 bytes of gradient) from shared memory, hands the stage
// back, and computes; results leave by coalesced 16-byte stores.  absmax and
// the block sum of squares are shuffle reductions inside the half-warp.  The
// codec arithmetic uses the round-to-nearest intrinsics (__fmul_rn, __fadd_rn,
// __fdiv_rn), which the compiler never contracts into FMAs, in exactly the
// order of the page's steps.  Every wait on a stage is bounded: on expiry it
// records QMUON_ERR_TIMEOUT in the workspace header and the CTA winds down.
//
// Group sums without a second pass over HBM: every CTA writes its block sums
// into shared memory, folds them per norm group into one partial per
// (CTA, group) slot, and takes a ticket; the CTA that takes the last ticket
// adds the slots of every group in a fixed order (fp64) and writes the sums
// and inverse norms.  No CTA waits on another, and the result does not depend
// on scheduling.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstddef>
#include <cstdio>
#include <mutex>
#include <set>
#include <utility>

#include "qm_internal.h"

namespace qm {
namespace {

// ---------------------------------------------------------------------------
// gradient element I/O: 16 consecutive elements per lane
// ---------------------------------------------------------------------------
template <int DT> struct Grad;

template <> struct Grad<QMUON_BF16> {
  static constexpr int kVecs = 2;   // 16 x 2 B = 2 x 16 B
  __device__ __forceinline__ static float get(const uint4* v, int i) {
    const uint32_t w = reinterpret_cast<const uint32_t*>(v)[i >> 1];
    return __uint_as_float((i & 1) ? (w & 0xFFFF0000u) : (w << 16));
  }
  __device__ __forceinline__ static uint32_t pack2(float a, float b) {
    // one cvt.rn.bf16x2.f32: both halves rounded to nearest even
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  __device__ __forceinline__ static float load1(const void* p, int64_t i) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  }
  __device__ __forceinline__ static void store1(void* p, int64_t i, float v) {
    reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  }
};

template <> struct Grad<QMUON_FP16> {
  static constexpr int kVecs = 2;
  __device__ __forceinline__ static float get(const uint4* v, int i) {
    const uint32_t w = reinterpret_cast<const uint32_t*>(v)[i >> 1];
    return __half2float(__ushort_as_half((unsigned short)((i & 1) ? (w >> 16) : (w & 0xFFFFu))));
  }
  __device__ __forceinline__ static uint32_t pack2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  __device__ __forceinline__ static float load1(const void* p, int64_t i) {
    return __half2float(reinterpret_cast<const __half*>(p)[i]);
  }
  __device__ __forceinline__ static void store1(void* p, int64_t i, float v) {
    reinterpret_cast<__half*>(p)[i] = __float2half_rn(v);
  }
};

template <> struct Grad<QMUON_FP32> {
  static constexpr int kVecs = 4;
  __device__ __forceinline__ static float get(const uint4* v, int i) {
    return __uint_as_float(reinterpret_cast<const uint32_t*>(v)[i]);
  }
  __device__ __forceinline__ static float load1(const void* p, int64_t i) {
    return reinterpret_cast<const float*>(p)[i];
  }
  __device__ __forceinline__ static void store1(void* p, int64_t i, float v) {
    reinterpret_cast<float*>(p)[i] = v;
  }
};

// Stored codes as offset binary (u = q + 128): uint8 storage already is,
// int8 storage differs in the top bit of every byte.
template <int QK>
__device__ __forceinline__ uint32_t to_offset_binary(uint32_t w) {
  return (QK == QMUON_Q8_INT8) ? (w ^ 0x80808080u) : w;
}

// For byte b of an offset-binary word, prmt builds the fp32 pattern
// 0x4B0000uu = 2^23 + u; subtracting 2^23 + 128 (both exact) leaves
// u - 128 = q, so float(q) takes one prmt and one exact subtraction.
__device__ __forceinline__ float code_bits(uint32_t u, int b) {
  return __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650u | (uint32_t)b));
}

// Packed fp32 pairs (one instruction for two lanes of arithmetic), each
// component rounded to nearest exactly as the scalar __fmul_rn / __fsub_rn.
// ptxas fuses a packed multiply whose only use is a packed add into a packed
// FMA (one rounding instead of two), so a product that feeds an addition is
// always added with the scalar __fadd_rn: those chains were checked bit for
// bit against the scalar ones on the GPU (sub -> mul, mul -> scalar add,
// mul -> max -> add, mul -> E4M3 conversion).
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

// Four codes (their int32 low bytes, two's complement) into one stored word.
template <int QK>
__device__ __forceinline__ uint32_t pack_codes(int q0, int q1, int q2, int q3) {
  const uint32_t lo = __byte_perm((uint32_t)q0, (uint32_t)q1, 0x0040u);
  const uint32_t hi = __byte_perm((uint32_t)q2, (uint32_t)q3, 0x0040u);
  const uint32_t w = __byte_perm(lo, hi, 0x5410u);
  return (QK == QMUON_Q8_INT8) ? w : (w ^ 0x80808080u);
}

// E8M0 exponent byte of a 32-element block: 127 + e with e the smallest
// integer such that amax <= 448 * 2^e (448 = 1.75 * 2^8 is the largest E4M3
// value), clamped to [0, 254]; 127 for amax == 0, 254 for amax == inf.
// With amax = f * 2^E (f in [1, 2), biased exponent field ef = E + 127),
// e = E - 8 + [f > 1.75], so the byte is ef - 8 + [mantissa > 0.75].  A
// subnormal amax (ef = 0, below 2^-126) and any amax below 2^-119 give a
// negative byte and clamp to 0, so no subnormal case is needed: the byte is
// a few integer operations and selects, without branches.
__device__ __forceinline__ int e8m0_of_amax(float amax) {
  const uint32_t b = __float_as_uint(amax);   // amax >= 0: the sign bit is clear
  const int ef = (int)(b >> 23);
  const int byte = ef - 8 + (((b & 0x7FFFFFu) > 0x600000u) ? 1 : 0);
  const int clamped = byte < 0 ? 0 : (byte > 254 ? 254 : byte);
  return b == 0u ? 127 : (ef == 0xFF ? 254 : clamped);
}

// 2^(127 - byte) as an fp32 (byte in [0, 254]: exponent in [-127, 127]); the
// one subnormal power, 2^-127 (byte 254), is the pattern 0x00400000.
__device__ __forceinline__ float pow2_from_e8m0(int byte) {
  return __uint_as_float(byte < 254 ? (uint32_t)(254 - byte) << 23 : 0x00400000u);
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC'11): ten rounds of the 4 x 32-bit bijection; a round
// multiplies c0 and c2 by M0 = 0xD2511F53 and M1 = 0xCD9E8D57 and mixes the
// halves of the products with c1, c3 and the key, which is bumped by the Weyl
// constants 0x9E3779B9, 0xBB67AE85 between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Input of one block held by a lane between its loads and its compute.
template <int DT>
struct LaneIn {
  uint4 q;
  uint4 g[Grad<DT>::kVecs];
  float amax_old;
  int valid;   // elements of this lane inside the tensor (16 for a full block)
};

template <int QK, int DT>
__device__ __forceinline__ void load_lane(LaneIn<DT>& in, const UpdTensor& T, int64_t lb, int hl, bool full) {
  const int64_t e0 = lb * kBlock + hl * 16;
  in.amax_old = __ldcs(T.absmax + lb);
  const int64_t rem = T.numel - e0;
  in.valid = rem >= 16 ? 16 : (rem > 0 ? (int)rem : 0);
  if (full) {
    in.q = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(T.q8) + e0));
    constexpr int esz = (DT == QMUON_FP32) ? 4 : 2;
    const uint4* gp = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(T.grad) + e0 * esz);
#pragma unroll
    for (int v = 0; v < Grad<DT>::kVecs; ++v) in.g[v] = __ldcs(gp + v);
  } else {
    // tail of a tensor whose size is not a multiple of 256: element loads
    uint32_t qw[4] = {0u, 0u, 0u, 0u};
    uint32_t gw[4 * Grad<DT>::kVecs];
#pragma unroll
    for (int i = 0; i < 4 * Grad<DT>::kVecs; ++i) gw[i] = 0u;
    const uint8_t* qp = static_cast<const uint8_t*>(T.q8) + e0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i >= in.valid) continue;
      qw[i >> 2] |= (uint32_t)qp[i] << (8 * (i & 3));
      const float gv = Grad<DT>::load1(T.grad, e0 + i);
      if (DT == QMUON_FP32) {
        gw[i] = __float_as_uint(gv);
      } else {
        const uint32_t bits = (DT == QMUON_BF16)
            ? (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(gv))
            : (uint32_t)__half_as_ushort(__float2half_rn(gv));
        gw[i >> 1] |= bits << (16 * (i & 1));
      }
    }
    in.q = make_uint4(qw[0], qw[1], qw[2], qw[3]);
#pragma unroll
    for (int v = 0; v < Grad<DT>::kVecs; ++v)
      in.g[v] = make_uint4(gw[4 * v], gw[4 * v + 1], gw[4 * v + 2], gw[4 * v + 3]);
  }
}

// Steps 1-9 for one lane's 16 elements; returns the block's sum of m*m
// (identical in all 16 lanes of the half-warp).  The two half-warps of a warp
// may be on different blocks or one may have none, so every shuffle names
// only the 16 lanes of its own half.  FULL: the whole block lies inside the
// tensor (every lane has 16 elements); the tail block of a tensor takes the
// masked path, chosen by the whole half-warp together.
template <int QK, int DT, bool CARRIER, bool FULL, bool SR>
__device__ __forceinline__ float compute_lane(const LaneIn<DT>& in, const UpdTensor& T, int64_t lb,
                                              int hl, float beta, float omb, const UpdLaunch& L) {
  const unsigned hmask = 0xFFFFu << (threadIdx.x & 16u);
  const int64_t e0 = lb * kBlock + hl * 16;
  const uint32_t* qw = reinterpret_cast<const uint32_t*>(&in.q);
  uint32_t u[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) u[w] = to_offset_binary<QK>(qw[w]);
  // (1)-(2) dequantise: one division per block, one multiply per element
  const float s_old = __fdiv_rn(in.amax_old, 127.0f);
  float m[16];
  float amax = 0.0f, ss = 0.0f;
  const float2 s_old2 = make_float2(s_old, s_old), beta2 = make_float2(beta, beta), omb2 = make_float2(omb, omb);
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    // elements i and i + 1 as packed pairs: old = (2^23 + u - (2^23 + 128)) * s_old, the subtraction exact
    const float2 old = mul2_rn(sub2_rn(make_float2(code_bits(u[i >> 2], i & 3), code_bits(u[i >> 2], (i + 1) & 3)),
                                       make_float2(8388736.0f, 8388736.0f)),
                               s_old2);
    // (4) m = beta * old + (1 - beta) * g: two rounded products, one rounded sum
    const float2 pb = mul2_rn(beta2, old);
    const float2 pg = mul2_rn(omb2, make_float2(Grad<DT>::get(in.g, i), Grad<DT>::get(in.g, i + 1)));
    float mi[2] = {__fadd_rn(pb.x, pg.x), __fadd_rn(pb.y, pg.y)};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (!FULL && i + j >= in.valid) mi[j] = 0.0f;
      m[i + j] = mi[j];
      amax = fmaxf(amax, fabsf(mi[j]));
      ss = fmaf(mi[j], mi[j], ss);
    }
  }
  // (6) block absmax and (9) block sum of squares across the half-warp
  float amax_l = amax;
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {
    amax = fmaxf(amax, __shfl_xor_sync(hmask, amax, o));
    ss += __shfl_xor_sync(hmask, ss, o);
  }
  // (7) requantise: sc = 127 / amax, q = rint(m * sc).  No clamp is needed:
  // |m| <= amax, so |m * sc| <= 127 (1 + 2^-24) and rounds to at most 127;
  // amax == 0 gives sc = 0 and q = 0.  The rounding to an integer (ties to
  // even) is one fp32 addition of 1.5 * 2^23: the sum lies in [2^23, 2^24),
  // where the spacing is 1, and its low byte is q in two's complement.
  // A NaN product (a NaN in m, or an infinity times sc = 0) must give q = 0,
  // but the GPU's NaN has a nonzero low byte; max(product, -inf) turns it
  // into -inf, whose low byte is 0, and leaves every other product as it is.
  // (Taking that step only in blocks whose sum of squares is not finite
  // duplicated the loop and made the kernel spill.)
  const float sc = (amax == 0.0f) ? 0.0f : __fdiv_rn(127.0f, amax);
  uint32_t qo[4];
  if constexpr (!SR) {
    const float2 sc2 = make_float2(sc, sc);
    auto code = [](float x) { return (int)__float_as_uint(__fadd_rn(fmaxf(x, -INFINITY), 12582912.0f)); };
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float2 lo = mul2_rn(make_float2(m[4 * w], m[4 * w + 1]), sc2);
      const float2 hi = mul2_rn(make_float2(m[4 * w + 2], m[4 * w + 3]), sc2);
      qo[w] = pack_codes<QK>(code(lo.x), code(lo.y), code(hi.x), code(hi.y));
    }
  } else {
    // stochastic: q = clamp(floor(x + u), -127, 127) with x = m * sc and u the
    // top 24 bits of the element's Philox word over 2^24.  x + u rounded
    // toward -inf has the floor of the exact sum (integers are representable
    // there), and cvt.rmi maps NaN to 0.  Element e of the tensor takes word
    // e & 3 of the generator at counter (e / 4, high word, tensor, step).
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint64_t j = (uint64_t)(e0 >> 2) + (uint64_t)w;
      const uint4 r = philox4x32_10(make_uint4((uint32_t)j, (uint32_t)(j >> 32), (uint32_t)T.index, L.sr_step),
                                    L.sr_key0, L.sr_key1);
      const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
      int qi[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float u = __fmul_rn(__uint2float_rn(rw[b] >> 8), 5.9604644775390625e-8f);   // exact: k * 2^-24
        int qv = __float2int_rd(__fadd_rd(__fmul_rn(m[4 * w + b], sc), u));
        qi[b] = qv < -127 ? -127 : (qv > 127 ? 127 : qv);
      }
      qo[w] = pack_codes<QK>(qi[0], qi[1], qi[2], qi[3]);
    }
  }
  uint8_t* q8p = static_cast<uint8_t*>(T.q8) + e0;
  if (FULL) {
    __stcs(reinterpret_cast<uint4*>(q8p), make_uint4(qo[0], qo[1], qo[2], qo[3]));
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (i < in.valid) q8p[i] = (uint8_t)((qo[i >> 2] >> (8 * (i & 3))) & 0xFFu);
  }
  if (hl == 0) __stcs(T.absmax + lb, amax);  // (8)

  if constexpr (!CARRIER) {
    // (5) the momentum overwrites the gradient
    if (FULL) {
      constexpr int esz = (DT == QMUON_FP32) ? 4 : 2;
      uint4* gp = reinterpret_cast<uint4*>(static_cast<uint8_t*>(T.grad) + e0 * esz);
      if constexpr (DT == QMUON_FP32) {
#pragma unroll
        for (int v = 0; v < 4; ++v)
          __stcs(gp + v, make_uint4(__float_as_uint(m[4 * v]), __float_as_uint(m[4 * v + 1]),
                                    __float_as_uint(m[4 * v + 2]), __float_as_uint(m[4 * v + 3])));
      } else {
#pragma unroll
        for (int v = 0; v < 2; ++v)
          __stcs(gp + v, make_uint4(Grad<DT>::pack2(m[8 * v], m[8 * v + 1]),
                                    Grad<DT>::pack2(m[8 * v + 2], m[8 * v + 3]),
                                    Grad<DT>::pack2(m[8 * v + 4], m[8 * v + 5]),
                                    Grad<DT>::pack2(m[8 * v + 6], m[8 * v + 7])));
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (i < in.valid) Grad<DT>::store1(T.grad, e0 + i, m[i]);
    }
  } else {
    // MXFP8 carrier: a 32-element row block is two neighbouring lanes (the
    // tensor's columns are a multiple of 32, so flat 32-groups are row blocks)
    const float amax32 = fmaxf(amax_l, __shfl_xor_sync(hmask, amax_l, 1));
    const int byte = e8m0_of_amax(amax32);
    const float mult = pow2_from_e8m0(byte);
    const float2 mult2 = make_float2(mult, mult);
    uint32_t pw[4];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const float2 a = mul2_rn(make_float2(m[4 * v], m[4 * v + 1]), mult2);
      const float2 b = mul2_rn(make_float2(m[4 * v + 2], m[4 * v + 3]), mult2);
      pw[v] = __byte_perm(cvt_e4m3x2(a.x, a.y), cvt_e4m3x2(b.x, b.y), 0x5410u);
    }
    if (FULL || in.valid == 16) {
      __stcs(reinterpret_cast<uint4*>(T.payload + e0), make_uint4(pw[0], pw[1], pw[2], pw[3]));
      if ((hl & 1) == 0) T.scale[e0 >> 5] = (uint8_t)byte;
    }
    // valid is 0 or 16 here: the element count is a multiple of 32
  }
  return ss;
}

// ---------------------------------------------------------------------------
// The input stream: a producer warp copies each CTA's blocks into a ring of
// shared-memory stages (16 blocks per stage, one per half-warp) with bulk
// asynchronous copies, four stages ahead of the compute warps.
// ---------------------------------------------------------------------------
constexpr int kStageBlocks = 16;                 // one block per half-warp of the compute warps
constexpr int kUpdStages = 4;
constexpr int kUpdWarps = kUpdThreads / 32;      // compute warps
constexpr int kUpdThreadsAll = kUpdThreads + 32; // plus the producer warp
constexpr long long kUpdWaitCycles = 4000000000LL;   // bounded waits: ~2 s at 2 GHz

template <int DT>
struct UpdStage {
  static constexpr int kEsz = (DT == QMUON_FP32) ? 4 : 2;
  static constexpr uint32_t kQBytes = kStageBlocks * kBlock;          // codes
  static constexpr uint32_t kGBytes = kStageBlocks * kBlock * kEsz;   // gradient
  static constexpr uint32_t kABytes = kStageBlocks * 4;               // old absmax
  static constexpr uint32_t kBytes = kQBytes + kGBytes + kABytes;
};

template <int DT>
constexpr size_t upd_smem_bytes() {
  return (size_t)kUpdStages * UpdStage<DT>::kBytes + (size_t)kMaxChunk * (sizeof(float) + sizeof(int32_t)) +
         2 * kUpdStages * sizeof(uint64_t);
}

__device__ __forceinline__ uint32_t upd_smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ bool upd_try_wait(uint32_t bar, uint32_t parity) {
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
// Bounded wait: false once the phase has not completed in ~2 s (or another
// CTA already gave up), after recording QMUON_ERR_TIMEOUT in the header.
__device__ __noinline__ bool upd_wait(uint32_t bar, uint32_t parity, WsHeader* h, unsigned where) {
  if (upd_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (upd_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile unsigned*>(&h->error) != 0u) return false;
    if (clock64() - t0 > kUpdWaitCycles) {
      if (atomicCAS(&h->error, 0u, (unsigned)QMUON_ERR_TIMEOUT) == 0u) h->error_info = where;
      return false;
    }
  }
}
__device__ __forceinline__ void upd_bar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void upd_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void upd_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// global -> shared bulk copy (16-byte aligned ends, size a multiple of 16)
// counted on `bar` as transaction bytes
__device__ __forceinline__ void upd_bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// 4-byte asynchronous copy, and an arrival on `bar` once this thread's
// earlier asynchronous copies have landed (the barrier's count includes it)
__device__ __forceinline__ void upd_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void upd_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

template <int QK, int DT, bool CARRIER, bool SR>
__global__ void __launch_bounds__(kUpdThreadsAll, 3) update_kernel(UpdLaunch L) {
  using ST = UpdStage<DT>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* stage0 = smem_raw;   // kUpdStages x (codes | gradient | old absmax)
  float* s_bsum = reinterpret_cast<float*>(smem_raw + kUpdStages * ST::kBytes);
  int32_t* s_bgrp = reinterpret_cast<int32_t*>(s_bsum + kMaxChunk);
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_bgrp + kMaxChunk);
  const uint32_t full0 = upd_smem_u32(bars), empty0 = upd_smem_u32(bars + kUpdStages);
  __shared__ int s_last;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int64_t kb = (int64_t)blockIdx.x * L.chunk;
  const int64_t ke = (kb + L.chunk < L.nb_total) ? kb + L.chunk : L.nb_total;
  const int n_stages = (int)((ke - kb + kStageBlocks - 1) / kStageBlocks);
  const bool reduce = L.layout.n_groups > 0;
  const bool keep = reduce || L.nonfinite != nullptr;   // the block sums are needed after the loop
  const bool single = (L.tensors == nullptr);

  if (tid == 0) {
    for (int s = 0; s < kUpdStages; ++s) {
      upd_bar_init(full0 + 8 * s, 1 + kStageBlocks);   // the copying lane + one async-copy arrival per block lane
      upd_bar_init(empty0 + 8 * s, kUpdWarps);          // every compute warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == kUpdWarps) {
    // ---- producer: stage i holds blocks kb + 16 i .. kb + 16 i + 15.  The
    // tensor of the stage's first block is cached with its fields (block
    // indices only grow) ----
    int t = 0;
    if (!single) {
      int lo = 0, hi = L.n_tensors - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(L.tensor_begin + mid) <= kb) lo = mid; else hi = mid - 1;
      }
      t = lo;
    }
    UpdTensor T = single ? L.single : L.tensors[t];
    int64_t tend = single ? L.nb_total : __ldg(L.tensor_begin + t + 1);
    bool ok = true;
    int i = 0;
    for (; i < n_stages; ++i) {
      const int slot = i % kUpdStages;
      // lane 0 waits for the slot, the warp follows its decision
      if (lane == 0 && i >= kUpdStages) ok = upd_wait(empty0 + 8 * slot, ((i / kUpdStages) - 1) & 1, L.header, 0x1100u);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      unsigned char* st = stage0 + slot * ST::kBytes;
      const uint32_t fb = full0 + 8 * slot;
      const int64_t k0 = kb + (int64_t)i * kStageBlocks;
      const int64_t k1 = (k0 + kStageBlocks < ke) ? k0 + kStageBlocks : ke;
      while (k0 >= tend) {   // never for a single tensor
        ++t;
        T = L.tensors[t];
        tend = __ldg(L.tensor_begin + t + 1);
      }
      // lane j < 16: the old absmax of block k0 + j (4-byte asynchronous copy)
      if (lane < kStageBlocks) {
        const int64_t k = k0 + lane;
        if (k < k1) {
          const float* src;
          if (k < tend) {
            src = T.absmax + (k - T.block_begin);
          } else {   // the stage crosses into a later tensor
            int tt = t + 1;
            while (k >= __ldg(L.tensor_begin + tt + 1)) ++tt;
            src = L.tensors[tt].absmax + (k - __ldg(L.tensor_begin + tt));
          }
          upd_async4(upd_smem_u32(st + ST::kQBytes + ST::kGBytes + 4 * lane), src);
        }
        upd_async_arrive(fb);
      }
      // lane 0: codes and gradient of the whole blocks, one bulk copy each per
      // tensor segment (a tensor's partial last block is read by its compute
      // lanes directly); the byte count is armed before the copies start
      if (lane == 0) {
        uint32_t bytes = 0;
        for (int pass = 0; pass < 2; ++pass) {
          if (pass == 1) upd_arrive_expect_tx(fb, bytes);
          int tt = t;
          UpdTensor TT = T;
          int64_t te = tend;
          for (int64_t a = k0; a < k1;) {
            if (a >= te) {
              ++tt;
              TT = L.tensors[tt];
              te = __ldg(L.tensor_begin + tt + 1);
              continue;
            }
            const int64_t b = (te < k1) ? te : k1;
            const int64_t lb = a - TT.block_begin;
            int64_t nfull = b - a;
            if ((lb + nfull) * kBlock > TT.numel) nfull = TT.numel / kBlock - lb;   // drop a partial last block
            if (nfull > 0) {
              if (pass == 0) {
                bytes += (uint32_t)(nfull * kBlock * (1 + ST::kEsz));
              } else {
                const int j = (int)(a - k0);
                upd_bulk_load(upd_smem_u32(st + j * kBlock), static_cast<const uint8_t*>(TT.q8) + lb * kBlock,
                              (uint32_t)(nfull * kBlock), fb);
                upd_bulk_load(upd_smem_u32(st + ST::kQBytes + j * kBlock * ST::kEsz),
                              static_cast<const uint8_t*>(TT.grad) + lb * kBlock * ST::kEsz,
                              (uint32_t)(nfull * kBlock * ST::kEsz), fb);
              }
            }
            a = b;
          }
        }
      }
      __syncwarp();
    }
    // every copy issued lands before the CTA moves on
    if (lane == 0)
      for (int k = (i > kUpdStages ? i - kUpdStages : 0); k < i; ++k)
        upd_wait(full0 + 8 * (k % kUpdStages), (k / kUpdStages) & 1, L.header, 0x1200u);
    __syncwarp();
  } else {
    // ---- compute warps: half-warp hw takes block kb + 16 i + hw of stage i ----
    const int hw = tid >> 4, hl = tid & 15;
    const float beta = L.beta;
    const float omb = __fsub_rn(1.0f, beta);
    int t = 0;
    if (!single) {
      const int64_t k0 = kb + hw;
      int lo = 0, hi = L.n_tensors - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(L.tensor_begin + mid) <= k0) lo = mid; else hi = mid - 1;
      }
      t = lo;
    }
    // this half-warp's current tensor, cached with its fields
    UpdTensor T = single ? L.single : L.tensors[t];
    int64_t tend = single ? L.nb_total : __ldg(L.tensor_begin + t + 1);
    for (int i = 0; i < n_stages; ++i) {
      const int slot = i % kUpdStages;
      const int64_t k = kb + (int64_t)i * kStageBlocks + hw;
      const bool has = k < ke;
      // the whole warp goes on or stops together (half-warp shuffles follow)
      const bool ok = __all_sync(0xffffffffu, upd_wait(full0 + 8 * slot, (i / kUpdStages) & 1, L.header, 0x1300u));
      const unsigned char* st = stage0 + slot * ST::kBytes;
      LaneIn<DT> in;
      int64_t lb = 0;
      bool full = true;
      if (has && ok) {
        while (k >= tend) {
          ++t;
          T = L.tensors[t];
          tend = __ldg(L.tensor_begin + t + 1);
        }
        lb = k - T.block_begin;
        full = (lb + 1) * kBlock <= T.numel;   // uniform across the half-warp
        if (full) {
          in.q = *reinterpret_cast<const uint4*>(st + hw * kBlock + hl * 16);
          const uint4* gs = reinterpret_cast<const uint4*>(st + ST::kQBytes + hw * kBlock * ST::kEsz + hl * 16 * ST::kEsz);
#pragma unroll
          for (int v = 0; v < Grad<DT>::kVecs; ++v) in.g[v] = gs[v];
          in.amax_old = *reinterpret_cast<const float*>(st + ST::kQBytes + ST::kGBytes + 4 * hw);
          in.valid = 16;
        } else {
          load_lane<QK, DT>(in, T, lb, hl, false);
        }
      }
      __syncwarp();
      if (lane == 0) upd_arrive(empty0 + 8 * slot);   // this warp is done reading the stage
      if (!ok) break;
      if (has) {
        int32_t g = 0;
        if (reduce && hl == 0 && L.layout.block_group) g = __ldg(L.layout.block_group + k);
        const float ss = full ? compute_lane<QK, DT, CARRIER, true, SR>(in, T, lb, hl, beta, omb, L)
                              : compute_lane<QK, DT, CARRIER, false, SR>(in, T, lb, hl, beta, omb, L);
        if (keep && hl == 0) {
          s_bsum[k - kb] = ss;
          if (reduce) s_bgrp[k - kb] = g;
        }
      }
    }
  }
  if (!keep) return;
  __syncthreads();
  const int nloc = (int)(ke - kb);
  // blocks whose momentum holds a NaN or an infinity (or whose squares overflow)
  if (L.nonfinite && warp == 0) {
    unsigned bad = 0;
    for (int i = lane; i < nloc; i += 32) bad += isfinite(s_bsum[i]) ? 0u : 1u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if (lane == 0 && bad) atomicAdd(L.nonfinite, bad);
  }
  if (!reduce) return;

  // ---- per-(CTA, group) partial sums, fixed order ----
  const bool one_group = (L.layout.block_group == nullptr);
  const int s0 = one_group ? (int)blockIdx.x : __ldg(L.layout.cta_slot_begin + blockIdx.x);
  const int s1 = one_group ? (int)blockIdx.x + 1 : __ldg(L.layout.cta_slot_begin + blockIdx.x + 1);
  for (int s = s0 + warp; s < s1 && warp < kUpdWarps; s += kUpdWarps) {
    const int g = one_group ? 0 : __ldg(L.layout.slot_group + s);
    float sum = 0.0f, comp = 0.0f;   // compensated fp32 sum per lane
    for (int i = lane; i < nloc; i += 32) {
      if (s_bgrp[i] == g) {
        const float y = s_bsum[i] - comp;
        const float tt = sum + y;
        comp = (tt - sum) - y;
        sum = tt;
      }
    }
    const double v = warp_sum((double)sum - (double)comp);
    if (lane == 0) L.partials[s] = v;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&L.header->ticket, 1u) == gridDim.x - 1) ? 1 : 0;
  __syncthreads();
  if (!s_last) return;

  // ---- the last CTA: per-group totals in slot order ----
  __threadfence();
  for (int g = warp; g < L.layout.n_groups && warp < kUpdWarps; g += kUpdWarps) {
    const int j0 = one_group ? 0 : __ldg(L.layout.grp_ptr + g);
    const int j1 = one_group ? (int)gridDim.x : __ldg(L.layout.grp_ptr + g + 1);
    double acc = 0.0;
    for (int j = j0 + lane; j < j1; j += 32)
      acc += __ldcg(L.partials + (one_group ? j : __ldg(L.layout.grp_slots + j)));
    acc = warp_sum(acc);
    if (lane == 0) {
      if (L.group_sumsq) L.group_sumsq[g] = (float)acc;
      if (L.group_inv) L.group_inv[g] = (float)(1.0 / (sqrt(acc) + kEps));
    }
  }
  if (tid == 0) L.header->ticket = 0u;
}

// In-place normalisation (second pass): grad <- store(float(grad) * inv[group]).
template <int DT>
__global__ void __launch_bounds__(kUpdThreads) scale_groups_kernel(UpdLaunch L, const float* inv) {
  const int hw = threadIdx.x >> 4, hl = threadIdx.x & 15;
  const bool single = (L.tensors == nullptr);
  int t = 0;   // k only grows, so the tensor index only grows
  for (int64_t k = (int64_t)blockIdx.x * 16 + hw; k < L.nb_total; k += (int64_t)gridDim.x * 16) {
    if (!single) while (k >= __ldg(L.tensor_begin + t + 1)) ++t;
    const int32_t g = L.layout.block_group ? __ldg(L.layout.block_group + k) : 0;
    if (g < 0) continue;
    const float s = __ldg(inv + g);
    const UpdTensor T = single ? L.single : L.tensors[t];
    const int64_t e0 = (k - T.block_begin) * kBlock + hl * 16;
    const int64_t rem = T.numel - e0;
    const int valid = rem >= 16 ? 16 : (rem > 0 ? (int)rem : 0);
    for (int i = 0; i < valid; ++i)
      Grad<DT>::store1(T.grad, e0 + i, __fmul_rn(Grad<DT>::load1(T.grad, e0 + i), s));
  }
}

template <int QK, int DT, bool C, bool SR>
void* kernel_ptr() { return reinterpret_cast<void*>(&update_kernel<QK, DT, C, SR>); }

template <int QK, int DT>
void* pick_variant(bool carrier, bool sr) {
  if (carrier) return sr ? nullptr : kernel_ptr<QK, DT, true, false>();   // the carrier rounds to nearest only
  return sr ? kernel_ptr<QK, DT, false, true>() : kernel_ptr<QK, DT, false, false>();
}

void* pick_kernel(qmuon_q8_kind q8, qmuon_dtype dt, bool carrier, bool sr = false) {
  const bool i8 = (q8 == QMUON_Q8_INT8);
  if (q8 != QMUON_Q8_INT8 && q8 != QMUON_Q8_UINT8) return nullptr;
  switch (dt) {
    case QMUON_BF16: return i8 ? pick_variant<QMUON_Q8_INT8, QMUON_BF16>(carrier, sr)
                               : pick_variant<QMUON_Q8_UINT8, QMUON_BF16>(carrier, sr);
    case QMUON_FP16: return i8 ? pick_variant<QMUON_Q8_INT8, QMUON_FP16>(carrier, sr)
                               : pick_variant<QMUON_Q8_UINT8, QMUON_FP16>(carrier, sr);
    case QMUON_FP32: return i8 ? pick_variant<QMUON_Q8_INT8, QMUON_FP32>(carrier, sr)
                               : pick_variant<QMUON_Q8_UINT8, QMUON_FP32>(carrier, sr);
  }
  return nullptr;
}

size_t upd_smem(qmuon_dtype dt) { return dt == QMUON_FP32 ? upd_smem_bytes<QMUON_FP32>() : upd_smem_bytes<QMUON_BF16>(); }

// Dynamic shared memory above the 48 KB default needs an opt-in per kernel.
// The shared-memory opt-in belongs to a (kernel, device) pair: it is set once
// per pair, so that a step's launches make no other CUDA call (a step can be
// captured into a CUDA graph).
cudaError_t prepare_kernel(void* k, qmuon_dtype dt) {
  static std::mutex mu;
  static std::set<std::pair<void*, int>> done;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({k, dev})) return cudaSuccess;
  }
  const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)upd_smem(dt));
  if (e == cudaSuccess) {
    std::lock_guard<std::mutex> lock(mu);
    done.insert({k, dev});
  }
  return e;
}

}  // namespace

int update_blocks_per_sm(qmuon_q8_kind q8, qmuon_dtype dt, bool carrier) {
  void* k = pick_kernel(q8, dt, carrier);
  if (!k || prepare_kernel(k, dt) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kUpdThreadsAll, upd_smem(dt)) != cudaSuccess) return 0;
  return n;
}

cudaError_t launch_update(const UpdLaunch& L, qmuon_q8_kind q8, qmuon_dtype dt, bool carrier,
                          cudaStream_t stream) {
  void* k = pick_kernel(q8, dt, carrier, L.sr != 0);
  if (!k) return cudaErrorInvalidValue;
  const cudaError_t e = prepare_kernel(k, dt);
  if (e != cudaSuccess) return e;
  UpdLaunch arg = L;
  void* args[] = {&arg};
  return cudaLaunchKernel(k, dim3(L.grid), dim3(kUpdThreadsAll), args, upd_smem(dt), stream);
}

cudaError_t launch_scale_groups(const UpdLaunch& L, qmuon_dtype dt, const float* inv,
                                cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t want = (L.nb_total + 15) / 16;
  int grid = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
  if (grid < 1) grid = 1;
  switch (dt) {
    case QMUON_BF16: scale_groups_kernel<QMUON_BF16><<<grid, kUpdThreads, 0, stream>>>(L, inv); break;
    case QMUON_FP16: scale_groups_kernel<QMUON_FP16><<<grid, kUpdThreads, 0, stream>>>(L, inv); break;
    case QMUON_FP32: scale_groups_kernel<QMUON_FP32><<<grid, kUpdThreads, 0, stream>>>(L, inv); break;
  }
  return cudaGetLastError();
}

}  // namespace qm

// ---------------------------------------------------------------------------
// Allocation-free single-tensor update (qmuon_update_normalize_noalloc).
//
// The same update kernel as above, launched for one tensor and one norm
// group, with its scratch -- the workspace header holding the last-CTA ticket
// and one fp64 partial sum per CTA -- in a file-scope device array instead of
// a caller-provided workspace.  Host code cannot use the array's name as a
// device address, so the address is looked up once per device with
// cudaGetSymbolAddress (that device current) and passed to the kernel.
//
// A kernel records a failure (a bounded wait that expired) in the header's
// error word, and its waits give up at once while that word is set.  So
// before each launch a one-thread kernel moves a recorded status into a
// pending pair of words (the first failure is kept) and clears the error word
// and the ticket; qmuon_noalloc_sync_status reports the pending status, else
// the error word, and clears both.
// ---------------------------------------------------------------------------
namespace {

constexpr int kStaticSlots = 8192;  // partial-sum slots: one per CTA of the launch
static __device__ __align__(256) unsigned char g_static_scratch[qm::kWsHeader + kStaticSlots * sizeof(double)];
// the pending status and its site live in the header's spare words
constexpr int kPendingStatus = 0, kPendingSite = 1;

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on the
// first call per device).
cudaError_t static_scratch(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_static_addr[dev] = p;
  }
  *out = g_static_addr[dev];
  return cudaSuccess;
}

// Carries a status recorded by the previous call into the pending words and
// clears what the update kernel needs at zero: the error word and the ticket.
__global__ void noalloc_carry_status_kernel(qm::WsHeader* h) {
  if (h->error != 0u && h->pad[kPendingStatus] == 0u) {
    h->pad[kPendingStatus] = h->error;
    h->pad[kPendingSite] = h->error_info;
  }
  h->error = 0u;
  h->error_info = 0u;
  h->ticket = 0u;
}

qmuon_status current_device(const char* where, int* dev) {
  const cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return qm::set_error(where, e);
  if (*dev < 0 || *dev >= kMaxDevices)
    return qm::set_error_what(where, "device ordinal beyond the static table", QMUON_ERR_UNSUPPORTED);
  return QMUON_OK;
}

}  // namespace

extern "C" qmuon_status qmuon_update_normalize_noalloc(const qmuon_tensor* tensor, qmuon_q8_kind q8_kind,
                                                       qmuon_dtype grad_dtype, float beta, float* sumsq,
                                                       float* inv_norm, void* stream) {
  qm::NvtxRange nvtx_range("qmuon_update_normalize_noalloc");
  using namespace qm;
  // ---- host validation, before any CUDA call ----
  if (!tensor) return set_error_msg("qmuon_update_normalize_noalloc: null tensor", QMUON_ERR_INVALID_ARGUMENT);
  if (q8_kind != QMUON_Q8_INT8 && q8_kind != QMUON_Q8_UINT8) return QMUON_ERR_INVALID_ARGUMENT;
  if (grad_dtype != QMUON_BF16 && grad_dtype != QMUON_FP16 && grad_dtype != QMUON_FP32) return QMUON_ERR_INVALID_ARGUMENT;
  if (tensor->rows <= 0 || tensor->cols <= 0) return QMUON_ERR_INVALID_ARGUMENT;
  if (tensor->cols > QMUON_NOALLOC_MAX_ELEMS / tensor->rows)
    return set_error_msg("qmuon_update_normalize_noalloc: tensor larger than QMUON_NOALLOC_MAX_ELEMS, the capacity "
                         "of the static scratch array", QMUON_ERR_INVALID_ARGUMENT);
  const int64_t n = tensor->rows * tensor->cols;
  if (!tensor->q8 || !tensor->absmax || !tensor->grad) return QMUON_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(tensor->q8) & 15) || (reinterpret_cast<uintptr_t>(tensor->grad) & 15) ||
      (reinterpret_cast<uintptr_t>(tensor->absmax) & 3))
    return QMUON_ERR_INVALID_ARGUMENT;
  if ((sumsq && (reinterpret_cast<uintptr_t>(sumsq) & 3)) || (inv_norm && (reinterpret_cast<uintptr_t>(inv_norm) & 3)))
    return QMUON_ERR_INVALID_ARGUMENT;

  int dev = 0, sms = 0;
  qmuon_status st = current_device("qmuon_update_normalize_noalloc (device)", &dev);
  if (st != QMUON_OK) return st;
  void* scratch = nullptr;
  cudaError_t e = static_scratch(dev, &scratch);
  if (e != cudaSuccess) return set_error("qmuon_update_normalize_noalloc (cudaGetSymbolAddress)", e);
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return set_error("qmuon_update_normalize_noalloc (SM count)", e);
  const int per_sm = update_blocks_per_sm(q8_kind, grad_dtype, false);
  if (per_sm <= 0) return set_error_msg("qmuon_update_normalize_noalloc: occupancy query failed", QMUON_ERR_CUDA);

  // the launch geometry of the planned entry point, so the sums are formed alike
  const int64_t nb = (n + kBlock - 1) / kBlock;
  int32_t grid = 0;
  int64_t chunk = 0;
  update_geometry(nb, sms, per_sm, &grid, &chunk);
  if (grid > kStaticSlots)
    return set_error_msg("qmuon_update_normalize_noalloc: launch needs more partial-sum slots than the static "
                         "scratch array holds", QMUON_ERR_INVALID_ARGUMENT);

  UpdLaunch L{};
  L.tensors = nullptr;
  L.single.q8 = tensor->q8;
  L.single.absmax = tensor->absmax;
  L.single.grad = tensor->grad;
  L.single.numel = n;
  L.single.block_begin = 0;
  L.n_tensors = 1;
  L.nb_total = nb;
  L.chunk = chunk;
  L.grid = grid;
  L.beta = beta;
  L.layout.n_groups = (sumsq || inv_norm) ? 1 : 0;  // block_group null: one group, one slot per CTA
  L.header = static_cast<WsHeader*>(scratch);
  L.partials = reinterpret_cast<double*>(static_cast<unsigned char*>(scratch) + kWsHeader);
  L.group_sumsq = sumsq;
  L.group_inv = inv_norm;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: keep its status for
  // qmuon_noalloc_sync_status, and start the error word and ticket at zero
  noalloc_carry_status_kernel<<<1, 1, 0, s>>>(L.header);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = launch_update(L, q8_kind, grad_dtype, false, s);
  if (e != cudaSuccess) return set_error("qmuon_update_normalize_noalloc (launch)", e);
  tally(T_UPDATE_CALLS);
  tally_grad_state(grad_dtype, q8_kind, 1);
  return QMUON_OK;
}

extern "C" qmuon_status qmuon_noalloc_sync_status(void* stream) {
  using namespace qm;
  int dev = 0;
  qmuon_status st = current_device("qmuon_noalloc_sync_status (device)", &dev);
  if (st != QMUON_OK) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return set_error("qmuon_noalloc_sync_status (stream synchronize)", e);
  // the symbol copies read and write the array on the current device and
  // allocate nothing
  WsHeader h{};
  e = cudaMemcpyFromSymbol(&h, g_static_scratch, sizeof(h), 0, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return set_error("qmuon_noalloc_sync_status (read header)", e);
  const unsigned status = h.pad[kPendingStatus] ? h.pad[kPendingStatus] : h.error;
  const unsigned site = h.pad[kPendingStatus] ? h.pad[kPendingSite] : h.error_info;
  if (status == 0u) return QMUON_OK;
  const unsigned zero[2] = {0u, 0u};
  e = cudaMemcpyToSymbol(g_static_scratch, zero, sizeof(zero), offsetof(WsHeader, error), cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpyToSymbol(g_static_scratch, zero, sizeof(zero), offsetof(WsHeader, pad) + kPendingStatus * 4,
                           cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return set_error("qmuon_noalloc_sync_status (clear header)", e);
  char msg[128];
  std::snprintf(msg, sizeof(msg), "qmuon_update_normalize_noalloc: kernel reported status %u at site 0x%x", status,
                site);
  return set_error_msg(msg, (qmuon_status)status);
}

extern "C" qmuon_status qmuon_noalloc_inject_status(qmuon_status status, uint32_t site) {
  using namespace qm;
  if ((int)status <= (int)QMUON_OK || (int)status > (int)QMUON_ERR_OUT_OF_MEMORY)
    return set_error_msg("qmuon_noalloc_inject_status: not a failure status", QMUON_ERR_INVALID_ARGUMENT);
  int dev = 0;
  qmuon_status st = current_device("qmuon_noalloc_inject_status (device)", &dev);
  if (st != QMUON_OK) return st;
  const unsigned words[2] = {(unsigned)status, site};
  const cudaError_t e = cudaMemcpyToSymbol(g_static_scratch, words, sizeof(words),
                                           offsetof(WsHeader, pad) + kPendingStatus * 4, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return set_error("qmuon_noalloc_inject_status (write header)", e);
  return QMUON_OK;
}

// kvp_decode.cuh -- paged-KV decode attention kernels for sm_103a.
//
// What is computed ("ATB PagedAttention", "PagedAttention 的 Attention 计算修改";
// "KV Cache 优化与显存管理", 二): for request b with n = context_lens[b] and
// query head h, out[b,h] = sum_i softmax_i(scale * q.K_i) V_i over the n cached
// tokens, K_i/V_i gathered through the block table (16 tokens per block) from
// K/V head h / G.  The pages walk one page at a time with an online softmax;
// here that walk is reorganised for GB300:
//
//   * One CTA per (request, kv head, split-context partition) serves the whole
//     query group of that kv head, so each K/V byte is read from HBM once.
//   * The CTA's slice of the block table is staged in shared memory first
//     ("踩坑一": the page table is copied on chip once, not looked up in HBM per
//     page) and every id is range-checked before any copy is issued.
//   * Each of the CTA's 4 warps owns a ring of 2 shared-memory stages.  Lane 0
//     issues TMA tensor copies (cp.async.bulk.tensor, 128-byte swizzle) of the
//     block's K and V tiles ([16 tokens][D] contiguous per (block, head)) into
//     a stage, completing on an mbarrier; the warp consumes blocks
//     w, w+4, w+8, ... with its own online-softmax state, refilling each stage
//     as soon as it is consumed.  Across 3 resident CTAs this keeps ~100 KB of
//     K/V in flight per SM.
//   * Consumers: CUDA cores (fp32 FMA, shuffle reductions) when a kv head serves
//     1-2 query heads; warp tensor cores (mma.m16n8k16, fp32 accumulate) when it
//     serves 3-8 query heads, where S^T = K Q^T (16 tokens x 8 heads) and
//     O^T += V^T P^T (D x 8 heads) per block are genuine dense tiles.
//   * The warps' partial states are merged in shared memory; a request that
//     fits one partition writes its output directly, otherwise the partition
//     writes (m, l, o) to the workspace for the reduce kernel (flash-decoding).
#pragma once

#include "kvp_device.cuh"
#include "kvp_internal.h"

namespace kvp {

// ---------------------------------------------------------------------------
// Shuffle reduction of N partial sums held by every lane across groups of L
// lanes (N <= L, both powers of two): each step halves the number of values a
// lane holds while summing over one lane bit, so N values need N-1 shuffles
// instead of N*log2(L).  Afterwards lane l holds the full sum of value index
// (l % L) >> log2(L / N).
template <int N, int BIT>
struct Butterfly {
  __device__ __forceinline__ static void run(float* v, int lane) {
    if constexpr (BIT >= 1) {
      if constexpr (N > 1) {
        const bool upper = (lane & BIT) != 0;
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
          const float send = upper ? v[i] : v[i + N / 2];
          const float keep = upper ? v[i + N / 2] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, BIT);
        }
        Butterfly<N / 2, BIT / 2>::run(v, lane);
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], BIT);
        Butterfly<1, BIT / 2>::run(v, lane);
      }
    }
  }
};

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// Offset of 16-byte chunk c of token row t in a 16-bit tile whose rows are
// split into 128-byte TMA boxes ([box][16 rows][128 B], 128-byte swizzle).
__device__ __forceinline__ uint32_t tile16_off(int t, int c) {
  return static_cast<uint32_t>((c >> 3) * (16 * 128)) +
         dev::swz128(static_cast<uint32_t>(t * 128 + ((c & 7) << 4)));
}

// ===========================================================================
// CUDA-core consumer: a kv head serving G = 1 or 2 query heads.
// Lane (c, r): c = lane % (D/8) owns elements [8c, 8c+8) of every row,
// r = lane / (D/8) owns tokens r, r + R, ... (R = 32 / (D/8) rows per pass).
template <bool kBf16, int D, int G>
struct SimtPath {
  static constexpr int kD = D;
  static constexpr int kHeads = G;
  static constexpr int kElemBytes = 2;
  static constexpr int kTileBytes = 16 * D * 2;
  static constexpr int kScaleStageBytes = 0;
  static constexpr int kLpr = D / 8;        // lanes per row
  static constexpr int kRpp = 32 / kLpr;    // rows per pass
  static constexpr int kKpl = 16 / kRpp;    // tokens per lane
  static constexpr int kNv = G * kKpl;      // partial scores per lane
  static_assert(kNv <= kLpr, "score reduction assumes at most one value per lane");
  static constexpr int kSh = ilog2(kLpr / kNv);

  struct State {
    float q[G][8];
    float o[G][8];
    float m[G];
    float l[G];
  };

  __device__ __forceinline__ static void init(State& st, const DecodeParams& p, int b, int head0,
                                              int /*nheads*/, int lane) {
    const int c = lane % kLpr;
    const uint16_t* q = static_cast<const uint16_t*>(p.q);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const uint4 raw = *reinterpret_cast<const uint4*>(
          q + (static_cast<size_t>(b) * p.num_q_heads + head0 + g) * D + c * 8);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = dev::unpack2<kBf16>(w[i]);
        st.q[g][2 * i] = f.x;
        st.q[g][2 * i + 1] = f.y;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) st.o[g][e] = 0.f;
      st.m[g] = -INFINITY;
      st.l[g] = 0.f;
    }
  }

  __device__ __forceinline__ static void consume(State& st, const uint8_t* kt, const uint8_t* vt,
                                                 const float*, int valid, int lane,
                                                 float scale_log2) {
    const int c = lane % kLpr;
    const int r = lane / kLpr;
    float ps[kNv];
#pragma unroll
    for (int k = 0; k < kKpl; ++k) {
      const uint4 raw = *reinterpret_cast<const uint4*>(kt + tile16_off(r + kRpp * k, c));
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
      float kf[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = dev::unpack2<kBf16>(w[i]);
        kf[2 * i] = f.x;
        kf[2 * i + 1] = f.y;
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(st.q[g][e], kf[e], acc);
        ps[g * kKpl + k] = acc;
      }
    }
    Butterfly<kNv, kLpr / 2>::run(ps, lane);
    const int v = (lane % kLpr) >> kSh;
    const int gl = v / kKpl;
    const int tl = r + kRpp * (v % kKpl);
    float s = ps[0] * scale_log2;
    if (tl >= valid) s = -INFINITY;

    float mine_m = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mb = dev::warp_max((G == 1 || gl == g) ? s : -INFINITY);
      const float mn = fmaxf(st.m[g], mb);
      if (mn > st.m[g]) {  // warp-uniform
        const float a = exp2f(st.m[g] - mn);
#pragma unroll
        for (int e = 0; e < 8; ++e) st.o[g][e] *= a;
        st.l[g] *= a;
        st.m[g] = mn;
      }
      if (G == 1 || gl == g) mine_m = st.m[g];
    }
    const float pe = exp2f(s - mine_m);
    const bool owner = ((lane % kLpr) & ((1 << kSh) - 1)) == 0;
#pragma unroll
    for (int g = 0; g < G; ++g) st.l[g] += (owner && (G == 1 || gl == g)) ? pe : 0.f;

#pragma unroll
    for (int k = 0; k < kKpl; ++k) {
      const int t = r + kRpp * k;
      const uint4 raw = *reinterpret_cast<const uint4*>(vt + tile16_off(t, c));
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
      float vf[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = dev::unpack2<kBf16>(w[i]);
        vf[2 * i] = f.x;
        vf[2 * i + 1] = f.y;
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float pk = __shfl_sync(0xffffffffu, pe, r * kLpr + ((g * kKpl + k) << kSh));
        if (t < valid) {  // slots past the context may hold anything, even NaN
#pragma unroll
          for (int e = 0; e < 8; ++e) st.o[g][e] = fmaf(pk, vf[e], st.o[g][e]);
        }
      }
    }
  }

  // Write this warp's (m, l, o[head][D]) to the merge area.
  __device__ __forceinline__ static void finalize(State& st, float* mo, float* mm, float* ml,
                                                  int lane) {
    const int c = lane % kLpr;
    const int r = lane / kLpr;
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float x = st.o[g][e];
#pragma unroll
        for (int o = kLpr; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        st.o[g][e] = x;
      }
      const float lsum = dev::warp_sum(st.l[g]);
      if (r == 0) {
        float4* dst = reinterpret_cast<float4*>(mo + g * D + c * 8);
        dst[0] = make_float4(st.o[g][0], st.o[g][1], st.o[g][2], st.o[g][3]);
        dst[1] = make_float4(st.o[g][4], st.o[g][5], st.o[g][6], st.o[g][7]);
      }
      if (lane == 0) {
        mm[g] = st.m[g];
        ml[g] = lsum;
      }
    }
  }
};

// ===========================================================================
// Tensor-core consumer for 16-bit pools: up to 8 query heads per kv head.
// Per block: S^T[16 tok x 8 heads] = K[16 x D] . Q^T[D x 8] (D/16 mma) and
// O^T[D x 8] += V^T[D x 16] . P^T[16 x 8] (D/16 mma; bf16 P is split into a
// bf16 high part and a bf16 residual so P keeps ~16 significant bits).
// Fragments: g8 = lane / 4, t4 = lane % 4 (the mma "group" and "thread in group").
template <bool kBf16, int D>
struct MmaPath {
  static constexpr int kD = D;
  static constexpr int kHeads = 8;
  static constexpr int kElemBytes = 2;
  static constexpr int kTileBytes = 16 * D * 2;
  static constexpr int kScaleStageBytes = 0;
  static constexpr int kMt = D / 16;

  struct State {
    uint32_t qb[kMt][2];
    float o[kMt][4];
    float m[2];
    float l[2];
  };

  __device__ __forceinline__ static void init(State& st, const DecodeParams& p, int b, int head0,
                                              int nheads, int lane) {
    const int g8 = lane >> 2, t4 = lane & 3;
    const uint16_t* q = static_cast<const uint16_t*>(p.q) +
                        (static_cast<size_t>(b) * p.num_q_heads + head0 + g8) * D;
#pragma unroll
    for (int s = 0; s < kMt; ++s) {
      if (g8 < nheads) {
        st.qb[s][0] = *reinterpret_cast<const uint32_t*>(q + 16 * s + 2 * t4);
        st.qb[s][1] = *reinterpret_cast<const uint32_t*>(q + 16 * s + 2 * t4 + 8);
      } else {
        st.qb[s][0] = 0u;
        st.qb[s][1] = 0u;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) st.o[s][i] = 0.f;
    }
    st.m[0] = st.m[1] = -INFINITY;
    st.l[0] = st.l[1] = 0.f;
  }

  __device__ __forceinline__ static void consume(State& st, const uint8_t* kt, const uint8_t* vt,
                                                 const float*, int valid, int lane,
                                                 float scale_log2) {
    const int g8 = lane >> 2, t4 = lane & 3;
    const uint32_t kbase = dev::smem_addr(kt);
    const uint32_t vbase = dev::smem_addr(vt);
    // ---- scores: S^T = K Q^T
    float sacc[4] = {0.f, 0.f, 0.f, 0.f};
    const int tok_a = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int ch_a = lane >> 4;
#pragma unroll
    for (int s = 0; s < kMt; ++s) {
      uint32_t a0, a1, a2, a3;
      dev::ldsm_x4(kbase + tile16_off(tok_a, 2 * s + ch_a), a0, a1, a2, a3);
      dev::mma16816<kBf16>(sacc, a0, a1, a2, a3, st.qb[s][0], st.qb[s][1]);
    }
    float s0 = sacc[0] * scale_log2, s1 = sacc[1] * scale_log2;
    float s2 = sacc[2] * scale_log2, s3 = sacc[3] * scale_log2;
    if (valid < 16) {
      if (g8 >= valid) s0 = s1 = -INFINITY;
      if (g8 + 8 >= valid) s2 = s3 = -INFINITY;
    }
    // ---- online softmax (per head: heads 2*t4 and 2*t4+1 live in this lane)
    float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const float mn0 = fmaxf(st.m[0], mx0), mn1 = fmaxf(st.m[1], mx1);
    if (__any_sync(0xffffffffu, (mn0 > st.m[0]) || (mn1 > st.m[1]))) {
      const float al0 = exp2f(st.m[0] - mn0), al1 = exp2f(st.m[1] - mn1);
#pragma unroll
      for (int mt = 0; mt < kMt; ++mt) {
        st.o[mt][0] *= al0;
        st.o[mt][1] *= al1;
        st.o[mt][2] *= al0;
        st.o[mt][3] *= al1;
      }
      st.l[0] *= al0;
      st.l[1] *= al1;
      st.m[0] = mn0;
      st.m[1] = mn1;
    }
    const float p0 = exp2f(s0 - st.m[0]), p1 = exp2f(s1 - st.m[1]);
    const float p2 = exp2f(s2 - st.m[0]), p3 = exp2f(s3 - st.m[1]);
    st.l[0] += p0 + p2;
    st.l[1] += p1 + p3;
    // ---- P^T as the B operand: transpose the (token x head) fragments
    const uint32_t x01 = dev::pack2<kBf16>(p0, p1);
    const uint32_t x23 = dev::pack2<kBf16>(p2, p3);
    const uint32_t b0 = dev::movm_t(x01);
    const uint32_t b1 = dev::movm_t(x23);
    uint32_t b0r = 0, b1r = 0;
    if constexpr (kBf16) {
      const float2 h01 = dev::unpack2<true>(x01);
      const float2 h23 = dev::unpack2<true>(x23);
      b0r = dev::movm_t(dev::pack2<true>(p0 - h01.x, p1 - h01.y));
      b1r = dev::movm_t(dev::pack2<true>(p2 - h23.x, p3 - h23.y));
    }
    // ---- O^T += V^T P^T
    uint32_t m01 = 0xffffffffu, m23 = 0xffffffffu;
    if (valid < 16) {
      m01 = (2 * t4 < valid ? 0x0000ffffu : 0u) | (2 * t4 + 1 < valid ? 0xffff0000u : 0u);
      m23 = (2 * t4 + 8 < valid ? 0x0000ffffu : 0u) | (2 * t4 + 9 < valid ? 0xffff0000u : 0u);
    }
    const int tok_b = (lane & 7) + ((lane >> 4) & 1) * 8;
    const int ch_b = (lane >> 3) & 1;
#pragma unroll
    for (int mt = 0; mt < kMt; ++mt) {
      uint32_t a0, a1, a2, a3;
      dev::ldsm_x4_t(vbase + tile16_off(tok_b, 2 * mt + ch_b), a0, a1, a2, a3);
      a0 &= m01;
      a1 &= m01;
      a2 &= m23;
      a3 &= m23;
      dev::mma16816<kBf16>(st.o[mt], a0, a1, a2, a3, b0, b1);
      if constexpr (kBf16) dev::mma16816<true>(st.o[mt], a0, a1, a2, a3, b0r, b1r);
    }
  }

  __device__ __forceinline__ static void finalize(State& st, float* mo, float* mm, float* ml,
                                                  int lane) {
    const int g8 = lane >> 2, t4 = lane & 3;
    float l0 = st.l[0], l1 = st.l[1];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
#pragma unroll
    for (int mt = 0; mt < kMt; ++mt) {
      const int d = 16 * mt + g8;
      mo[(2 * t4) * D + d] = st.o[mt][0];
      mo[(2 * t4 + 1) * D + d] = st.o[mt][1];
      mo[(2 * t4) * D + d + 8] = st.o[mt][2];
      mo[(2 * t4 + 1) * D + d + 8] = st.o[mt][3];
    }
    if (g8 == 0) {
      mm[2 * t4] = st.m[0];
      mm[2 * t4 + 1] = st.m[1];
      ml[2 * t4] = l0;
      ml[2 * t4 + 1] = l1;
    }
  }
};

// ===========================================================================
// Tensor-core consumer for 8-bit code pools (INT8, or FP8 E4M3 when kFp8) with
// per-token-per-head fp32 scales, up to 8 query heads per kv head.  Codes
// convert exactly to fp16 (or bf16 when q is bf16).  The contraction index d
// is permuted so each lane reads a contiguous run of codes: for K, lane t4
// feeds d in [t4*D/4, (t4+1)*D/4); for V, lane g8 produces d in
// [g8*D/8, (g8+1)*D/8).  The K scale multiplies the 16 scores after the mma;
// the V scale is folded into P (normalised by the block's largest V scale to
// stay in fp16 range) and restored in fp32.
template <bool kQBf16, int D, bool kFp8 = false>
struct MmaInt8Path {
  static constexpr int kD = D;
  static constexpr int kHeads = 8;
  static constexpr int kElemBytes = 1;
  static constexpr int kTileBytes = 16 * D;
  static constexpr int kScaleStageBytes = 2 * 16 * 4;
  static constexpr int kMt = D / 16;      // k-steps of QK and m-tiles of PV
  static constexpr int kVw = D / 32;      // 32-bit words of V per token per lane

  struct State {
    uint32_t qb[kMt][2];
    float o[kMt][4];
    float m[2];
    float l[2];
  };

  __device__ __forceinline__ static void init(State& st, const DecodeParams& p, int b, int head0,
                                              int nheads, int lane) {
    const int g8 = lane >> 2, t4 = lane & 3;
    const uint16_t* q = static_cast<const uint16_t*>(p.q) +
                        (static_cast<size_t>(b) * p.num_q_heads + head0 + g8) * D + (D / 4) * t4;
#pragma unroll
    for (int s = 0; s < kMt; ++s) {
      if (g8 < nheads) {
        const uint2 w = *reinterpret_cast<const uint2*>(q + 4 * s);
        st.qb[s][0] = w.x;
        st.qb[s][1] = w.y;
      } else {
        st.qb[s][0] = 0u;
        st.qb[s][1] = 0u;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) st.o[s][i] = 0.f;
    }
    st.m[0] = st.m[1] = -INFINITY;
    st.l[0] = st.l[1] = 0.f;
  }

  // Tiles with 128-byte rows arrive 128B-swizzled; 64-byte rows (D = 64)
  // arrive unswizzled (a 64-byte box does not take the 128-byte pattern).
  __device__ __forceinline__ static uint32_t off(uint32_t o) {
    if constexpr (D >= 128) {
      return dev::swz128(o);
    } else {
      return o;
    }
  }

  // FP8 codes are widened by the hardware E4M3 -> fp16 convert.  (Measured
  // alternatives: an exact bit move into fp16 at value * 2^-8 for K and V, or
  // for V only, both ran slower because the move is all integer-pipe work.)
  static constexpr float kCodeUnscale = 1.0f;
  static constexpr float kVUnscale = 1.0f;

  // Codes (bytes 0,1 or 2,3 of w) as the QK operand type.
  template <bool kHigh>
  __device__ __forceinline__ static uint32_t k_pair(uint32_t w) {
    if constexpr (kFp8) {
      const uint32_t h = dev::e4m3x2_to_f16x2(static_cast<uint16_t>(kHigh ? (w >> 16) : w));
      if constexpr (kQBf16) {
        const float2 f = dev::unpack2<false>(h);
        return dev::pack2<true>(f.x, f.y);
      } else {
        return h;
      }
    } else if constexpr (kQBf16) {
      return dev::i8x2_to_bf16x2<kHigh>(w);
    } else {
      return dev::i8x2_to_f16x2<kHigh>(w ^ 0x80808080u);
    }
  }

  // V codes of tokens A and B (byte j of each word, j = 0..3) as the fp16
  // pair (A_j, B_j) for the PV mma (FP8: times 2^-8).
  template <int J>
  __device__ __forceinline__ static uint32_t v_pair(uint32_t a, uint32_t b) {
    if constexpr (kFp8) {
      // interleave (A_j, B_j) as the two bytes of a 16-bit pair, then convert
      const uint32_t x = dev::prmt(a, b, (J < 2) ? 0x5140u : 0x7362u);
      return dev::e4m3x2_to_f16x2(static_cast<uint16_t>((J & 1) ? (x >> 16) : x));
    } else {
      // interleave (A_j, B_j) as bytes, then the biased-byte conversion
      const uint32_t x = dev::prmt(a ^ 0x80808080u, b ^ 0x80808080u,
                                   (J < 2) ? 0x5140u : 0x7362u);
      return dev::i8x2_to_f16x2<(J & 1) != 0>(x);
    }
  }

  __device__ __forceinline__ static void consume(State& st, const uint8_t* kt, const uint8_t* vt,
                                                 const float* sc, int valid, int lane,
                                                 float scale_log2) {
    const int g8 = lane >> 2, t4 = lane & 3;
    // ---- K codes of rows g8 and g8+8, bytes [t4*D/4, (t4+1)*D/4)
    uint32_t k0[kMt], k1[kMt];
#pragma unroll
    for (int i = 0; i < kMt / 4; ++i) {
      const uint32_t o = (D / 4) * t4 + 16 * i;
      const uint4 r0 = *reinterpret_cast<const uint4*>(kt + off(g8 * D + o));
      const uint4 r1 = *reinterpret_cast<const uint4*>(kt + off((g8 + 8) * D + o));
      k0[4 * i] = r0.x; k0[4 * i + 1] = r0.y; k0[4 * i + 2] = r0.z; k0[4 * i + 3] = r0.w;
      k1[4 * i] = r1.x; k1[4 * i + 1] = r1.y; k1[4 * i + 2] = r1.z; k1[4 * i + 3] = r1.w;
    }
    float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s = 0; s < kMt; ++s) {
      dev::mma16816<kQBf16>(sacc, k_pair<false>(k0[s]), k_pair<false>(k1[s]), k_pair<true>(k0[s]),
                            k_pair<true>(k1[s]), st.qb[s][0], st.qb[s][1]);
    }
    const float* ks = sc;
    const float* vs = sc + 16;
    const float kg = ks[g8] * (scale_log2 * kCodeUnscale);
    const float kg8 = ks[g8 + 8] * (scale_log2 * kCodeUnscale);
    float s0 = sacc[0] * kg, s1 = sacc[1] * kg, s2 = sacc[2] * kg8, s3 = sacc[3] * kg8;
    const bool ok_lo = g8 < valid, ok_hi = g8 + 8 < valid;
    if (!ok_lo) s0 = s1 = -INFINITY;
    if (!ok_hi) s2 = s3 = -INFINITY;
    // ---- online softmax
    float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const float mn0 = fmaxf(st.m[0], mx0), mn1 = fmaxf(st.m[1], mx1);
    if (__any_sync(0xffffffffu, (mn0 > st.m[0]) || (mn1 > st.m[1]))) {
      const float al0 = exp2f(st.m[0] - mn0), al1 = exp2f(st.m[1] - mn1);
#pragma unroll
      for (int mt = 0; mt < kMt; ++mt) {
        st.o[mt][0] *= al0;
        st.o[mt][1] *= al1;
        st.o[mt][2] *= al0;
        st.o[mt][3] *= al1;
      }
      st.l[0] *= al0;
      st.l[1] *= al1;
      st.m[0] = mn0;
      st.m[1] = mn1;
    }
    const float p0 = exp2f(s0 - st.m[0]), p1 = exp2f(s1 - st.m[1]);
    const float p2 = exp2f(s2 - st.m[0]), p3 = exp2f(s3 - st.m[1]);
    st.l[0] += p0 + p2;
    st.l[1] += p1 + p3;
    // ---- fold the V scales into P (select, so NaN scales of unused slots vanish)
    const float vg = ok_lo ? vs[g8] : 0.f, vg8 = ok_hi ? vs[g8 + 8] : 0.f;
    float vmax = fmaxf(vg, vg8);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
    const float inv = vmax > 0.f ? 1.f / vmax : 0.f;
    const float r0 = vg * inv, r8 = vg8 * inv;
    const uint32_t b0 = dev::movm_t(dev::pack2<false>(p0 * r0, p1 * r0));
    const uint32_t b1 = dev::movm_t(dev::pack2<false>(p2 * r8, p3 * r8));
    // ---- V codes of tokens 2t4, 2t4+1, 2t4+8, 2t4+9, bytes [g8*D/8, (g8+1)*D/8)
    uint32_t va[kVw], vb[kVw], vc[kVw], vd[kVw];
    {
      const int ta = 2 * t4, tb = 2 * t4 + 1, tc = 2 * t4 + 8, td = 2 * t4 + 9;
      const uint32_t o = (D / 8) * g8;
      if constexpr (kVw == 4) {
        const uint4 ra = *reinterpret_cast<const uint4*>(vt + off(ta * D + o));
        const uint4 rb = *reinterpret_cast<const uint4*>(vt + off(tb * D + o));
        const uint4 rc = *reinterpret_cast<const uint4*>(vt + off(tc * D + o));
        const uint4 rd = *reinterpret_cast<const uint4*>(vt + off(td * D + o));
        va[0] = ra.x; va[1] = ra.y; va[2] = ra.z; va[3] = ra.w;
        vb[0] = rb.x; vb[1] = rb.y; vb[2] = rb.z; vb[3] = rb.w;
        vc[0] = rc.x; vc[1] = rc.y; vc[2] = rc.z; vc[3] = rc.w;
        vd[0] = rd.x; vd[1] = rd.y; vd[2] = rd.z; vd[3] = rd.w;
      } else {
        const uint2 ra = *reinterpret_cast<const uint2*>(vt + off(ta * D + o));
        const uint2 rb = *reinterpret_cast<const uint2*>(vt + off(tb * D + o));
        const uint2 rc = *reinterpret_cast<const uint2*>(vt + off(tc * D + o));
        const uint2 rd = *reinterpret_cast<const uint2*>(vt + off(td * D + o));
        va[0] = ra.x; va[1] = ra.y;
        vb[0] = rb.x; vb[1] = rb.y;
        vc[0] = rc.x; vc[1] = rc.y;
        vd[0] = rd.x; vd[1] = rd.y;
      }
      if constexpr (kFp8) {
        // E4M3 has NaN codes: V of tokens past the context (unused slots may
        // hold any bytes) must not reach the product, where 0 * NaN = NaN
        if (valid < 16) {
#pragma unroll
          for (int w = 0; w < kVw; ++w) {
            va[w] = ta < valid ? va[w] : 0u;
            vb[w] = tb < valid ? vb[w] : 0u;
            vc[w] = tc < valid ? vc[w] : 0u;
            vd[w] = td < valid ? vd[w] : 0u;
          }
        }
      }
    }
    float ct[kMt][4];
#pragma unroll
    for (int mt = 0; mt < kMt; ++mt) ct[mt][0] = ct[mt][1] = ct[mt][2] = ct[mt][3] = 0.f;
#pragma unroll
    for (int w = 0; w < kVw; ++w) {
      // m-tile 2w takes bytes 0 (rows g8) and 1 (rows g8+8) of word w; m-tile
      // 2w+1 takes bytes 2 and 3
      dev::mma16816<false>(ct[2 * w], v_pair<0>(va[w], vb[w]), v_pair<1>(va[w], vb[w]),
                           v_pair<0>(vc[w], vd[w]), v_pair<1>(vc[w], vd[w]), b0, b1);
      dev::mma16816<false>(ct[2 * w + 1], v_pair<2>(va[w], vb[w]), v_pair<3>(va[w], vb[w]),
                           v_pair<2>(vc[w], vd[w]), v_pair<3>(vc[w], vd[w]), b0, b1);
    }
    const float vrestore = vmax * kVUnscale;
#pragma unroll
    for (int mt = 0; mt < kMt; ++mt) {
#pragma unroll
      for (int i = 0; i < 4; ++i) st.o[mt][i] = fmaf(ct[mt][i], vrestore, st.o[mt][i]);
    }
  }

  __device__ __forceinline__ static void finalize(State& st, float* mo, float* mm, float* ml,
                                                  int lane) {
    const int g8 = lane >> 2, t4 = lane & 3;
    float l0 = st.l[0], l1 = st.l[1];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
#pragma unroll
    for (int mt = 0; mt < kMt; ++mt) {
      const int d = (D / 8) * g8 + 2 * mt;
      mo[(2 * t4) * D + d] = st.o[mt][0];
      mo[(2 * t4 + 1) * D + d] = st.o[mt][1];
      mo[(2 * t4) * D + d + 1] = st.o[mt][2];
      mo[(2 * t4 + 1) * D + d + 1] = st.o[mt][3];
    }
    if (g8 == 0) {
      mm[2 * t4] = st.m[0];
      mm[2 * t4 + 1] = st.m[1];
      ml[2 * t4] = l0;
      ml[2 * t4 + 1] = l1;
    }
  }
};

// ===========================================================================
template <class Path>
constexpr size_t decode_smem_for(int part_blocks) {
  constexpr int S = kWarps * kStagesPerWarp;
  return 1024 + static_cast<size_t>(S) * 2 * Path::kTileBytes +
         static_cast<size_t>(S) * Path::kScaleStageBytes + S * 8 +
         static_cast<size_t>(part_blocks) * 4 + 16;
}

// Zero the output rows [b, head0 .. head0+nheads) (requests with no tokens or
// with an invalid length).
template <int D>
__device__ __forceinline__ void zero_rows(const DecodeParams& p, int b, int head0, int nheads) {
  uint16_t* out = static_cast<uint16_t*>(p.out) +
                  (static_cast<size_t>(b) * p.num_q_heads + head0) * D;
  for (int i = threadIdx.x; i < nheads * D; i += blockDim.x) out[i] = 0;
}

// What one decode CTA works on: request b, kv head kvh, query heads head0 ..
// head0 + nheads - 1, and blocks blk0 .. blk0 + nb - 1 of the request's table
// (partition `part` of nparts); tail_valid tokens in the sequence's last block.
struct DecodeCta {
  int part, kvh, b, head0, nheads, n, nparts, nb, tail_valid;
  bool last_part;
};

// Shared memory of a decode CTA (1024-byte aligned stage area first).
struct DecodeSmem {
  uint8_t* stages;   // kWarps * kStagesPerWarp tiles of K then V
  float* scales;     // per tile: 16 K scales, 16 V scales (8-bit pools)
  uint64_t* bars;    // kWarps * kStagesPerWarp mbarriers
  int32_t* tbl;      // the partition's block ids
};

template <class Path>
__device__ __forceinline__ DecodeSmem decode_smem(uint8_t* smem_raw) {
  constexpr int S = kWarps * kStagesPerWarp;
  uint8_t* smem = dev::align1024(smem_raw);
  DecodeSmem m;
  m.stages = smem;
  m.scales = reinterpret_cast<float*>(smem + S * 2 * Path::kTileBytes);
  m.bars = reinterpret_cast<uint64_t*>(smem + S * 2 * Path::kTileBytes +
                                       S * Path::kScaleStageBytes);
  m.tbl = reinterpret_cast<int32_t*>(m.bars + S);
  return m;
}

// Behind a shared prefix's pass: the grid's first CTA waits for that pass
// before it exits (see decode_prologue).
__device__ __forceinline__ void shared_prefix_exit_wait(const DecodeParams& p) {
  if (p.skip_blocks > 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
    dev::grid_dependency_wait();
}

// Prologue shared by both pipelines: which work this CTA has, the partition's
// block ids staged in shared memory and range-checked ("踩坑一": the page table
// is copied on chip once, not looked up in HBM per page), and the fused
// append.  Returns false when the CTA has nothing to stream (its rows are
// already written or belong to another partition).  *any_bad: an id is out of
// range.  `init_bars` runs on thread 0 before the barrier that publishes the
// table.
template <class Path, class InitBars>
__device__ __forceinline__ bool decode_prologue(const DecodeParams& p, const DecodeSmem& sm,
                                                DecodeCta& c, bool* any_bad,
                                                InitBars init_bars) {
  using namespace dev;
  constexpr int D = Path::kD;
  c.part = blockIdx.x;
  c.kvh = blockIdx.y / p.qgroups;
  const int qg = blockIdx.y % p.qgroups;
  c.b = blockIdx.z;
  c.head0 = c.kvh * p.group + qg * p.heads_per_cta;
  c.nheads = min(p.heads_per_cta, p.group - qg * p.heads_per_cta);

  // the previous kernel (e.g. the append) has landed.  Behind a shared
  // prefix's pass (skip_blocks > 0) the two run side by side instead: that
  // pass -- a plain launch, so the append had landed before it began --
  // writes only partition 0, which this kernel never reads; the grid's first
  // CTA waits for it before it exits (shared_prefix_exit_wait), so this grid
  // completes after it and the reduce behind finds both written, while every
  // other CTA leaves its SM as soon as it is done
  if (p.skip_blocks == 0) grid_dependency_wait();
  c.n = p.context_lens[c.b];
  if (c.n <= 0 || c.n > p.max_blocks * kBlockSize) {
    if (c.part == 0) {
      zero_rows<D>(p, c.b, c.head0, c.nheads);
      if (c.n != 0 && threadIdx.x == 0) set_status(p.status, kErrBadBlock);
    }
    return false;
  }
  const int nblk_seq = (c.n + kBlockSize - 1) / kBlockSize;
  c.nparts = (nblk_seq - p.skip_blocks + p.part_blocks - 1) / p.part_blocks;
  const int blk0 = p.skip_blocks + c.part * p.part_blocks;
  if (blk0 >= nblk_seq) return false;
  c.nb = min(p.part_blocks, nblk_seq - blk0);
  c.last_part = blk0 + c.nb == nblk_seq;
  c.tail_valid = c.n - (nblk_seq - 1) * kBlockSize;

  // ---- stage this partition's slice of the block table and check every id
  bool bad = false;
  const int32_t* row = p.block_tables + static_cast<size_t>(c.b) * p.max_blocks + blk0;
  for (int i = threadIdx.x; i < c.nb; i += blockDim.x) {
    const int id = row[i];
    bad |= (id < 0) || (id >= p.num_blocks);
    sm.tbl[i] = id;
  }
  if (threadIdx.x == 0) {
    init_bars();
    fence_barrier_init();
  }
  *any_bad = __syncthreads_or(bad);

  // ---- fused append: the new token of this request (position n-1) lies in
  // the sequence's last block, which only last-partition CTAs read; they write
  // its K/V row for this kv head into the slot, then make the write visible to
  // the TMA (async proxy) before any copy is issued.  CTAs of other query
  // groups of the same kv head write the same bytes.
  if constexpr (Path::kElemBytes == 2) {
    if (p.new_k != nullptr && c.last_part && !*any_bad) {
      constexpr int kChunks = D * 2 / 16;  // 16-byte chunks per row
      const size_t srow =
          (static_cast<size_t>(sm.tbl[c.nb - 1]) * p.num_kv_heads + c.kvh) * kBlockSize +
          (c.n - 1) % kBlockSize;
      const size_t nrow = static_cast<size_t>(c.b) * p.num_kv_heads + c.kvh;
      if (threadIdx.x < 2 * kChunks) {
        const int ch = threadIdx.x % kChunks;
        const bool is_v = threadIdx.x >= kChunks;
        const uint4* src = static_cast<const uint4*>(is_v ? p.new_v : p.new_k) + nrow * kChunks;
        uint4* dst = reinterpret_cast<uint4*>(const_cast<void*>(is_v ? p.v_pool : p.k_pool)) +
                     srow * kChunks;
        dst[ch] = src[ch];
        fence_proxy_async_global();
      }
      __syncthreads();
    }
  }
  return true;
}

// Epilogue shared by both pipelines: merge the warps' partial states (the
// stage memory is free by now) and write the output rows (single partition)
// or this partition's (m, l, o) to the workspace.  cta_bad: a block id was out
// of range or a transfer timed out; the rows are then zero (or L < 0 marks the
// partition failed for the reduce).
template <class Path>
__device__ __forceinline__ void decode_epilogue(const DecodeParams& p, const DecodeSmem& sm,
                                                const DecodeCta& c, typename Path::State& st,
                                                bool cta_bad) {
  using namespace dev;
  constexpr int H = Path::kHeads;
  constexpr int D = Path::kD;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  float* mo = reinterpret_cast<float*>(sm.stages);
  float* mm = mo + kWarps * H * D;
  float* ml = mm + kWarps * H;
  if (!cta_bad) Path::finalize(st, mo + warp * H * D, mm + warp * H, ml + warp * H, lane);
  __syncthreads();

  const size_t rowbase = static_cast<size_t>(c.b) * p.num_q_heads + c.head0;
  if (c.nparts == 1 && p.skip_blocks == 0) {
    uint16_t* out = static_cast<uint16_t*>(p.out) + rowbase * D;
    for (int idx = threadIdx.x; idx < c.nheads * D; idx += blockDim.x) {
      const int hh = idx / D, d = idx % D;
      float res = 0.f;
      if (!cta_bad) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mm[w * H + hh]);
        float L = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float f = exp2f(mm[w * H + hh] - M);
          L = fmaf(f, ml[w * H + hh], L);
          acc = fmaf(f, mo[(w * H + hh) * D + d], acc);
        }
        res = L > 0.f ? acc / L : 0.f;
      }
      out[idx] = p.q_bf16 ? from_float<true>(res) : from_float<false>(res);
    }
  } else {
    for (int idx = threadIdx.x; idx < c.nheads * D; idx += blockDim.x) {
      const int hh = idx / D, d = idx % D;
      float M = -INFINITY, L = -1.f, acc = 0.f;  // L < 0 marks a failed partition
      if (!cta_bad) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mm[w * H + hh]);
        L = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float f = exp2f(mm[w * H + hh] - M);
          L = fmaf(f, ml[w * H + hh], L);
          acc = fmaf(f, mo[(w * H + hh) * D + d], acc);
        }
      }
      const size_t prow = (rowbase + hh) * p.max_parts + c.part + (p.skip_blocks > 0 ? 1 : 0);
      p.ws_o[prow * D + d] = acc;
      if (d == 0) {
        p.ws_ml[2 * prow] = M;
        p.ws_ml[2 * prow + 1] = L;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Per-block fetch: each of the CTA's 4 warps owns a ring of 2 stages and
// streams its own blocks w, w+4, ... (lane 0 issues the block's TMA boxes and
// waits with the warp), independently of the other warps.
template <class Path>
__global__ void __launch_bounds__(kWarps * 32)
    decode_partial_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tmv) {
  using namespace dev;
  constexpr int S = kWarps * kStagesPerWarp;
  constexpr int TB = Path::kTileBytes;
  constexpr int SB = Path::kScaleStageBytes;
  constexpr int H = Path::kHeads;
  constexpr int D = Path::kD;
  constexpr int kRowBytes = D * Path::kElemBytes;
  constexpr int kBoxBytes = kRowBytes < 128 ? kRowBytes : 128;  // inner extent of a TMA box
  constexpr int kBoxes = kRowBytes / kBoxBytes;                 // TMA boxes per tile
  static_assert(kWarps * H * (D + 2) * 4 <= S * 2 * TB, "merge area must fit in the stages");

  extern __shared__ uint8_t smem_raw[];
  const DecodeSmem sm = decode_smem<Path>(smem_raw);
  __shared__ int cta_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  DecodeCta c;
  bool any_bad = false;
  if (!decode_prologue<Path>(p, sm, c, &any_bad, [&] {
        cta_flag = 0;
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
#pragma unroll
        for (int s = 0; s < S; ++s) mbar_init(smem_addr(sm.bars + s), 1);
      })) {
    shared_prefix_exit_wait(p);
    return;
  }

  const float* ksrc = p.k_scale;
  const float* vsrc = p.v_scale;
  auto issue = [&](int j) {  // lane 0 of this warp: fetch the warp's j-th block
    const int i = warp + j * kWarps;
    const int stage = warp * kStagesPerWarp + (j % kStagesPerWarp);
    const uint32_t bar = smem_addr(sm.bars + stage);
    uint8_t* kdst = sm.stages + stage * 2 * TB;
    uint8_t* vdst = kdst + TB;
    const int y = (sm.tbl[i] * p.num_kv_heads + c.kvh) * kBlockSize;
    mbar_arrive_expect_tx(bar, 2 * TB + SB);
#pragma unroll
    for (int x = 0; x < kBoxes; ++x) {
      const int xe = x * (kBoxBytes / Path::kElemBytes);
      tma_load_2d(smem_addr(kdst + x * 16 * kBoxBytes), &tmk, xe, y, bar);
      tma_load_2d(smem_addr(vdst + x * 16 * kBoxBytes), &tmv, xe, y, bar);
    }
    if constexpr (SB > 0) {
      float* sdst = sm.scales + stage * (SB / 4);
      bulk_load(smem_addr(sdst), ksrc + y, 64, bar);
      bulk_load(smem_addr(sdst + 16), vsrc + y, 64, bar);
    }
  };

  typename Path::State st;
  bool ok = !any_bad;
  if (ok) {
    Path::init(st, p, c.b, c.head0, c.nheads, lane);
    const int my_blocks = c.nb > warp ? (c.nb - warp + kWarps - 1) / kWarps : 0;
    const int prologue = my_blocks < kStagesPerWarp ? my_blocks : kStagesPerWarp;
    if (lane == 0) {
      for (int j = 0; j < prologue; ++j) issue(j);
    }
    int issued = prologue;
    int j = 0;
    for (; j < my_blocks; ++j) {
      const int stage = warp * kStagesPerWarp + (j % kStagesPerWarp);
      const bool landed =
          mbar_wait_bounded(smem_addr(sm.bars + stage), (j / kStagesPerWarp) & 1);
      if (!__all_sync(0xffffffffu, landed)) {
        ok = false;
        break;
      }
      const int i = warp + j * kWarps;
      const int valid = (c.last_part && i == c.nb - 1) ? c.tail_valid : kBlockSize;
      const uint8_t* kt = sm.stages + stage * 2 * TB;
      Path::consume(st, kt, kt + TB, sm.scales + stage * (SB / 4), valid, lane, p.scale_log2);
      __syncwarp();
      if (j + kStagesPerWarp < my_blocks) {
        if (lane == 0) {
          fence_proxy_async_smem();
          issue(j + kStagesPerWarp);
        }
        ++issued;
      }
    }
    if (!ok) {
      // A transfer did not land in time: wait (bounded) for this warp's copies
      // still in flight so no TMA write outlives the CTA, then report.
      if (lane == 0) {
        for (int jj = j; jj < issued; ++jj) {
          const int stage = warp * kStagesPerWarp + (jj % kStagesPerWarp);
          mbar_wait_bounded(smem_addr(sm.bars + stage), (jj / kStagesPerWarp) & 1);
        }
        set_status(p.status, kErrTimeout);
        atomicExch(&cta_flag, 1);
      }
    }
  } else if (threadIdx.x == 0) {
    set_status(p.status, kErrBadBlock);
  }

  shared_prefix_exit_wait(p);
  launch_dependents();
  __syncthreads();
  decode_epilogue<Path>(p, sm, c, st, any_bad || cta_flag != 0);
}

// ---------------------------------------------------------------------------
// Run-merged fetch ("ATB KV Cache management", "显存碎片问题": blocks are
// allocated contiguously first, so most of a request's table is runs of
// consecutive physical blocks).  The CTA streams its blocks in groups of
// kWarps consecutive table entries (warp w still consumes blocks w, w+4, ...,
// so the softmax and the merge are those of the per-block pipeline); a group
// stage holds the group's K tiles back to back, then its V tiles.  Thread 0
// issues each group as maximal runs of 4, 2 or 1 physically consecutive
// blocks, one TMA box per run and tensor (5-D maps {row piece, 16 rows,
// pieces per row, Hkv, NB} whose box holds r whole tiles in the per-block
// layout), so a contiguous group costs 2 copies instead of 2 per block and
// row piece.  Barriers per group stage: full (the copies landed) and empty
// (all 4 warps consumed their tiles: kWarps arrivals).
template <class Path>
__global__ void __launch_bounds__(kWarps * 32)
    decode_merged_kernel(const DecodeParams p, const __grid_constant__ RunMaps maps) {
  using namespace dev;
  constexpr int kGS = kStagesPerWarp;  // group stages
  constexpr int TB = Path::kTileBytes;
  constexpr int SB = Path::kScaleStageBytes;
  constexpr int H = Path::kHeads;
  constexpr int D = Path::kD;
  constexpr int kGroupBytes = 2 * kWarps * TB;
  static_assert(kWarps == 4, "runs are cut into boxes of 4, 2 and 1 blocks");
  static_assert(kWarps * H * (D + 2) * 4 <= kGS * kGroupBytes, "merge area must fit");

  extern __shared__ uint8_t smem_raw[];
  const DecodeSmem sm = decode_smem<Path>(smem_raw);
  uint64_t* full = sm.bars;          // [kGS]
  uint64_t* empty = sm.bars + kGS;   // [kGS]
  __shared__ int cta_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  DecodeCta c;
  bool any_bad = false;
  if (!decode_prologue<Path>(p, sm, c, &any_bad, [&] {
        cta_flag = 0;
#pragma unroll
        for (int r = 0; r < 3; ++r) {
          prefetch_tensormap(&maps.k[r]);
          prefetch_tensormap(&maps.v[r]);
        }
#pragma unroll
        for (int s = 0; s < kGS; ++s) {
          mbar_init(smem_addr(full + s), 1);
          mbar_init(smem_addr(empty + s), kWarps);
        }
      })) {
    shared_prefix_exit_wait(p);
    return;
  }

  const int ngroups = (c.nb + kWarps - 1) / kWarps;
  // thread 0: fetch group g into group stage g % kGS
  auto issue_group = [&](int g) {
    const int st = g % kGS;
    const int i0 = g * kWarps;
    const int nt = min(kWarps, c.nb - i0);
    const uint32_t bar = smem_addr(full + st);
    uint8_t* kbase = sm.stages + st * kGroupBytes;
    uint8_t* vbase = kbase + kWarps * TB;
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nt * (2 * TB + SB)));
    for (int w = 0; w < nt;) {
      const int id = sm.tbl[i0 + w];
      int run = 1;
      while (w + run < nt && run < kWarps && sm.tbl[i0 + w + run] == id + run) ++run;
      const int box = run >= 4 ? 2 : (run >= 2 ? 1 : 0);  // map index: 4, 2 or 1 blocks
      tma_load_5d(smem_addr(kbase + w * TB), &maps.k[box], 0, 0, 0, c.kvh, id, bar);
      tma_load_5d(smem_addr(vbase + w * TB), &maps.v[box], 0, 0, 0, c.kvh, id, bar);
      w += 1 << box;
    }
    if constexpr (SB > 0) {
      for (int w = 0; w < nt; ++w) {
        const int y = (sm.tbl[i0 + w] * p.num_kv_heads + c.kvh) * kBlockSize;
        float* sdst = sm.scales + (st * kWarps + w) * (SB / 4);
        bulk_load(smem_addr(sdst), p.k_scale + y, 64, bar);
        bulk_load(smem_addr(sdst + 16), p.v_scale + y, 64, bar);
      }
    }
  };

  typename Path::State st;
  bool ok = !any_bad;
  if (ok) {
    Path::init(st, p, c.b, c.head0, c.nheads, lane);
    const int prologue = min(ngroups, kGS);
    if (threadIdx.x == 0) {
      for (int g = 0; g < prologue; ++g) issue_group(g);
    }
    int issued = prologue;
    int g = 0;
    for (; g < ngroups; ++g) {
      const int gs = g % kGS;
      const int i = g * kWarps + warp;
      if (i < c.nb) {
        const bool landed = mbar_wait_bounded(smem_addr(full + gs), (g / kGS) & 1);
        if (!__all_sync(0xffffffffu, landed)) {
          ok = false;
          break;
        }
        const int valid = (c.last_part && i == c.nb - 1) ? c.tail_valid : kBlockSize;
        const uint8_t* kt = sm.stages + gs * kGroupBytes + warp * TB;
        Path::consume(st, kt, kt + kWarps * TB, sm.scales + (gs * kWarps + warp) * (SB / 4),
                      valid, lane, p.scale_log2);
      }
      __syncwarp();
      if (lane == 0) {
        fence_proxy_async_smem();
        mbar_arrive(smem_addr(empty + gs));
      }
      if (g + kGS < ngroups) {
        if (threadIdx.x == 0) {
          // every warp has read its tile of group g: refill the stage
          if (mbar_wait_bounded(smem_addr(empty + gs), (g / kGS) & 1)) {
            issue_group(g + kGS);
          } else {
            ok = false;
          }
        }
        ++issued;
        if (!__all_sync(0xffffffffu, ok)) break;
      }
    }
    if (!ok) {
      // A wait timed out: thread 0 waits (bounded) for the copies it issued
      // that may still be in flight, so no TMA write outlives the CTA.
      if (threadIdx.x == 0) {
        for (int gg = max(0, issued - kGS); gg < issued; ++gg)
          mbar_wait_bounded(smem_addr(full + gg % kGS), (gg / kGS) & 1);
      }
      if (lane == 0) {
        set_status(p.status, kErrTimeout);
        atomicExch(&cta_flag, 1);
      }
    }
  } else if (threadIdx.x == 0) {
    set_status(p.status, kErrBadBlock);
  }

  shared_prefix_exit_wait(p);
  launch_dependents();
  __syncthreads();
  decode_epilogue<Path>(p, sm, c, st, any_bad || cta_flag != 0);
}

template <class Path>
cudaError_t launch_partial(const DecodeParams& p, const DecodeMaps& m, int grid_x,
                           cudaStream_t s) {
  const size_t smem = decode_smem_for<Path>(p.part_blocks);
  const dim3 grid(grid_x, p.num_kv_heads * p.qgroups, p.batch);
  if (m.merged) {
    const cudaError_t e = ensure_smem_attr(
        reinterpret_cast<const void*>(&decode_merged_kernel<Path>),
        decode_smem_for<Path>(kMaxPartBlocks));
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_merged_kernel<Path>, grid, dim3(kWarps * 32), smem, s, p, m.runs);
  }
  const cudaError_t e = ensure_smem_attr(
      reinterpret_cast<const void*>(&decode_partial_kernel<Path>),
      decode_smem_for<Path>(kMaxPartBlocks));
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_partial_kernel<Path>, grid, dim3(kWarps * 32), smem, s, p, m.k, m.v);
}

}  // namespace kvp

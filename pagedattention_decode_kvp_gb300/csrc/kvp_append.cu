// kvp_append.cu -- the write side of the paged cache:
//   * append: scatter new tokens' K/V rows to their slots ("KV Cache 优化与显存管理",
//     三, write_page; "ATB PagedAttention", "踩坑三", WriteKV), slot = block * 16 +
//     offset ("ATB 的 PagedAttention 实现": page = pos / size, offset = pos % size);
//   * append_int8: per token and head abs-max / 127 quantisation, then scatter
//     ("KV Cache 优化与显存管理", 三, KVCacheQuantizer per-channel branch); the
//     fixed-scale variant (per-tensor branch) and the FP8 (E4M3) variant
//     ("KV Cache 优化与显存管理", 二: INT8 or FP8) share the kernel;
//   * copy_blocks: whole-block copies for copy-on-write ("踩坑三", ExtendKVPage).
// All three are pure HBM streams: 16-byte vector loads and stores, one thread
// per 16-byte chunk, rows of a block contiguous so every warp access coalesces.
#include "kvp_device.cuh"
#include "kvp_internal.h"

namespace kvp {
namespace {

// grid = (ceil(T / tokens per CTA), Hkv); CPR 16-byte chunks per row, one per
// thread, so a row's chunks are adjacent lanes (coalesced source and slot).
template <int CPR>
__global__ void __launch_bounds__(256)
    append_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                  uint4* __restrict__ kc, uint4* __restrict__ vc, const int32_t* __restrict__ slots,
                  int num_tokens, int num_kv_heads, int num_slots, int32_t* status) {
  constexpr int kTokens = 256 / CPR;
  dev::grid_dependency_wait();
  dev::launch_dependents();
  const int t = blockIdx.x * kTokens + static_cast<int>(threadIdx.x) / CPR;
  const int ch = threadIdx.x % CPR;
  const int h = blockIdx.y;
  if (t >= num_tokens) return;
  const int slot = slots[t];
  if (slot < 0) return;  // padding token
  if (slot >= num_slots) {
    if (h == 0 && ch == 0) dev::set_status(status, kErrBadBlock);
    return;
  }
  const size_t src = (static_cast<size_t>(t) * num_kv_heads + h) * CPR + ch;
  const size_t dst =
      ((static_cast<size_t>(slot / kBlockSize) * num_kv_heads + h) * kBlockSize +
       slot % kBlockSize) * CPR + ch;
  kc[dst] = key[src];
  vc[dst] = value[src];
}

// Codes rint(x_e / s) of 8 elements, x / s being the IEEE float32 quotient,
// packed 4 per word (low byte first).
//
// Fast path: with r = x * (1/s), fma(x, 1/s, 1.5 * 2^23) rounds r once to an
// integer k, half to even, held in the low mantissa bits (|r| < 2^22), so the
// low byte of its bit pattern is k as an int8; d = fma(x, 1/s, -k) is r - k.
// r is within 2e-5 of x / s for |x / s| <= 127.0001 (1/s is a correctly
// rounded reciprocal; the product is exact inside the FMA), and RN(x / s)
// within 8e-6 of x / s, so whenever |d| < 0.5 - 1e-4 both round to the same
// integer.  Elements inside that band around a half-integer take the exact
// quotient instead.  Pairs of elements go through the packed two-lane FMA.
// kClip (a caller's fixed scale, where x / s may be anything) clamps r to
// [-1024, 1024] first, so the rounding trick stays in range, and clips the
// codes to [-128, 127]; clamped elements fail the band test and take the
// exact path.  Without kClip the clip never binds: s = RN(amax / 127) keeps
// |x / s| <= 127 * (1 + 2^-23), which rounds to at most 127.
template <bool kClip>
__device__ __forceinline__ void quantise8(const float (&x)[8], float s, float inv,
                                          uint32_t (&packed)[2]) {
  constexpr float kMagic = 12582912.0f;   // 1.5 * 2^23
  constexpr float kBand = 0.5f - 1.0e-4f;
  uint32_t bits[8];
  float d[8];
  const uint64_t inv2 = dev::f2pack(inv, inv);
  const uint64_t magic2 = dev::f2pack(kMagic, kMagic);
  const uint64_t nmagic2 = dev::f2pack(-kMagic, -kMagic);
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const uint64_t x2 = dev::f2pack(x[e], x[e + 1]);
    uint64_t m2;
    if constexpr (kClip) {
      const float2 r = dev::f2unpack(dev::fmul2(x2, inv2));
      m2 = dev::fadd2(dev::f2pack(fminf(fmaxf(r.x, -1024.f), 1024.f),
                                  fminf(fmaxf(r.y, -1024.f), 1024.f)), magic2);
    } else {
      m2 = dev::ffma2(x2, inv2, magic2);
    }
    const uint64_t k2 = dev::fadd2(m2, nmagic2);                 // exact
    const uint64_t nk2 = dev::f2pack(-dev::f2unpack(k2).x, -dev::f2unpack(k2).y);
    const float2 dd = dev::f2unpack(dev::ffma2(x2, inv2, nk2));  // r - k
    d[e] = dd.x;
    d[e + 1] = dd.y;
    float2 k = dev::f2unpack(k2);
    if constexpr (kClip) {
      k.x = fminf(fmaxf(k.x, -128.f), 127.f);
      k.y = fminf(fmaxf(k.y, -128.f), 127.f);
      bits[e] = static_cast<uint32_t>(static_cast<int>(k.x));
      bits[e + 1] = static_cast<uint32_t>(static_cast<int>(k.y));
    } else {
      const float2 m = dev::f2unpack(m2);
      bits[e] = __float_as_uint(m.x);
      bits[e + 1] = __float_as_uint(m.y);
    }
  }
  const float dmax = fmaxf(dev::max3f(fabsf(d[0]), fabsf(d[1]), fabsf(d[2])),
                           fmaxf(dev::max3f(fabsf(d[3]), fabsf(d[4]), fabsf(d[5])),
                                 fmaxf(fabsf(d[6]), fabsf(d[7]))));
  if (dmax > kBand) {  // rare: some element sits near a half-integer
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (fabsf(d[e]) > kBand) {
        int q = __float2int_rn(__fdiv_rn(x[e], s));
        if constexpr (kClip) q = min(127, max(-128, q));
        bits[e] = static_cast<uint32_t>(q);
      }
    }
  }
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    const uint32_t lo = __byte_perm(bits[4 * w], bits[4 * w + 1], 0x0040);
    const uint32_t hi = __byte_perm(bits[4 * w + 2], bits[4 * w + 3], 0x0040);
    packed[w] = __byte_perm(lo, hi, 0x5410);
  }
}

// E4M3 codes of x_e / s (IEEE float32 quotient), round-to-nearest-even,
// saturating at 448, packed 4 per word (low byte first).
__device__ __forceinline__ void quantise8_fp8(const float (&x)[8], float s, uint32_t (&packed)[2]) {
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    const uint32_t lo = dev::f32x2_to_e4m3x2(__fdiv_rn(x[4 * w], s), __fdiv_rn(x[4 * w + 1], s));
    const uint32_t hi =
        dev::f32x2_to_e4m3x2(__fdiv_rn(x[4 * w + 2], s), __fdiv_rn(x[4 * w + 3], s));
    packed[w] = lo | (hi << 16);
  }
}

enum class QuantMode { kInt8, kInt8Fixed, kFp8 };

// Quantise-and-scatter.  Eight lanes per (token, head) row, four rows per
// warp; lane j of a row owns the 16-byte chunks j, j + 8, ... of its K and of
// its V row (8 elements each, D / 64 chunks), so every load and store
// instruction covers whole rows' contiguous bytes.  grid = (ceil(T / 32),
// Hkv).
//   kInt8:      scale = amax / 127 (1 if not > 0), code = rint(x / scale)
//   kInt8Fixed: the given scale, code = clip(rint(x / scale), -128, 127)
//   kFp8:       scale = amax / 448 (1 if not > 0), code = E4M3(x / scale)
// and the scale is stored beside the codes.  The abs-max runs on the packed
// 16-bit source pairs (exact) and K's and V's travel in one shuffle word.
constexpr int kQuantLanes = 8;
constexpr int kQuantRowsPerCta = 256 / kQuantLanes;

template <bool kBf16, int D, QuantMode kMode>
__global__ void __launch_bounds__(256)
    append_quant_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                        uint8_t* __restrict__ kc, uint8_t* __restrict__ vc,
                        float* __restrict__ ks, float* __restrict__ vs, float fixed_ks,
                        float fixed_vs, const int32_t* __restrict__ slots, int num_tokens,
                        int num_kv_heads, int num_slots, int32_t* status) {
  constexpr int kChunks = D / 64;     // 16-byte chunks per lane, of K and of V
  constexpr int kRowChunks = D / 8;   // 16-byte chunks per row
  dev::grid_dependency_wait();
  dev::launch_dependents();
  const int t = blockIdx.x * kQuantRowsPerCta + static_cast<int>(threadIdx.x) / kQuantLanes;
  const int sub = threadIdx.x % kQuantLanes;
  const int h = blockIdx.y;
  const bool in = t < num_tokens;
  int slot = -1;
  uint4 rk[kChunks], rv[kChunks];
#pragma unroll
  for (int c = 0; c < kChunks; ++c) rk[c] = rv[c] = make_uint4(0u, 0u, 0u, 0u);
  if (in) {
    slot = slots[t];
    const size_t src = (static_cast<size_t>(t) * num_kv_heads + h) * kRowChunks + sub;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      rk[c] = key[src + c * kQuantLanes];
      rv[c] = value[src + c * kQuantLanes];
    }
  }
  float sk = fixed_ks, sv = fixed_vs;
  if constexpr (kMode != QuantMode::kInt8Fixed) {
    uint32_t mk = 0u, mv = 0u;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      mk = dev::absmax2<kBf16>(mk, dev::absmax2<kBf16>(dev::absmax2<kBf16>(rk[c].x, rk[c].y),
                                                       dev::absmax2<kBf16>(rk[c].z, rk[c].w)));
      mv = dev::absmax2<kBf16>(mv, dev::absmax2<kBf16>(dev::absmax2<kBf16>(rv[c].x, rv[c].y),
                                                       dev::absmax2<kBf16>(rv[c].z, rv[c].w)));
    }
    // K's two halves in the low half-word, V's in the high one
    uint32_t kv = dev::absmax2<kBf16>(__byte_perm(mk, mv, 0x5410), __byte_perm(mk, mv, 0x7632));
#pragma unroll
    for (int o = kQuantLanes / 2; o >= 1; o >>= 1)
      kv = dev::absmax2<kBf16>(kv, __shfl_xor_sync(0xffffffffu, kv, o));
    const float2 a = dev::unpack2<kBf16>(kv);
    // float32 IEEE division for the scale, as the quantiser is defined
    const float qmax = kMode == QuantMode::kFp8 ? 448.0f : 127.0f;
    sk = __fdiv_rn(a.x, qmax);
    sv = __fdiv_rn(a.y, qmax);
    sk = sk > 0.f ? sk : 1.0f;
    sv = sv > 0.f ? sv : 1.0f;
  }
  if (!in || slot < 0) return;
  if (slot >= num_slots) {
    if (sub == 0 && h == 0) dev::set_status(status, kErrBadBlock);
    return;
  }
  const size_t srow = (static_cast<size_t>(slot / kBlockSize) * num_kv_heads + h) * kBlockSize +
                      slot % kBlockSize;
  const float ik = kMode == QuantMode::kFp8 ? 0.f : __frcp_rn(sk);
  const float iv = kMode == QuantMode::kFp8 ? 0.f : __frcp_rn(sv);
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    float xk[8], xv[8];
    const uint32_t wk[4] = {rk[c].x, rk[c].y, rk[c].z, rk[c].w};
    const uint32_t wv[4] = {rv[c].x, rv[c].y, rv[c].z, rv[c].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 fk = dev::unpack2<kBf16>(wk[i]);
      const float2 fv = dev::unpack2<kBf16>(wv[i]);
      xk[2 * i] = fk.x;
      xk[2 * i + 1] = fk.y;
      xv[2 * i] = fv.x;
      xv[2 * i + 1] = fv.y;
    }
    uint32_t pk[2], pv[2];
    if constexpr (kMode == QuantMode::kFp8) {
      quantise8_fp8(xk, sk, pk);
      quantise8_fp8(xv, sv, pv);
    } else {
      quantise8<kMode == QuantMode::kInt8Fixed>(xk, sk, ik, pk);
      quantise8<kMode == QuantMode::kInt8Fixed>(xv, sv, iv, pv);
    }
    const size_t off = srow * D + (sub + c * kQuantLanes) * 8;
    *reinterpret_cast<uint2*>(kc + off) = make_uint2(pk[0], pk[1]);
    *reinterpret_cast<uint2*>(vc + off) = make_uint2(pv[0], pv[1]);
  }
  if (sub == 0) {
    ks[srow] = sk;
    vs[srow] = sv;
  }
}

// grid.y = pair index; grid.x strides over the 16-byte chunks of one block.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint4* kc, uint4* vc, uint4* ks, uint4* vs, const int32_t* __restrict__ pairs,
                       int num_pairs, long long chunks_kv, long long chunks_scale, int num_blocks,
                       int32_t* status) {
  dev::grid_dependency_wait();
  dev::launch_dependents();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long first = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int pr = blockIdx.y; pr < num_pairs; pr += gridDim.y) {
  const int src = pairs[2 * pr], dst = pairs[2 * pr + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) dev::set_status(status, kErrBadBlock);
    continue;
  }
  if (src == dst) continue;
  const uint4* ksrc = kc + src * chunks_kv;
  const uint4* vsrc = vc + src * chunks_kv;
  uint4* kdst = kc + dst * chunks_kv;
  uint4* vdst = vc + dst * chunks_kv;
  for (long long i = first; i < chunks_kv; i += stride) {
    const uint4 a = ksrc[i];
    const uint4 b = vsrc[i];
    kdst[i] = a;
    vdst[i] = b;
  }
  if (ks != nullptr) {
    for (long long i = first; i < chunks_scale; i += stride) {
      ks[dst * chunks_scale + i] = ks[src * chunks_scale + i];
      vs[dst * chunks_scale + i] = vs[src * chunks_scale + i];
    }
  }
  }
}

}  // namespace

cudaError_t launch_append(const void* key, const void* value, void* k_cache, void* v_cache,
                          const int32_t* slots, int num_tokens, const kvp_cache_desc& c,
                          int elem_bytes, int32_t* status, cudaStream_t s) {
  if (num_tokens == 0) return cudaSuccess;
  const int cpr = c.head_dim * elem_bytes / 16;
  const int nslots = c.num_blocks * kBlockSize;
  const auto* k = static_cast<const uint4*>(key);
  const auto* v = static_cast<const uint4*>(value);
  auto* kd = static_cast<uint4*>(k_cache);
  auto* vd = static_cast<uint4*>(v_cache);
  if (cpr == 16) {
    const dim3 grid((num_tokens + 15) / 16, c.num_kv_heads);
    return launch_pdl(append_kernel<16>, grid, dim3(256), 0, s, k, v, kd, vd, slots, num_tokens,
                      c.num_kv_heads, nslots, status);
  }
  if (cpr == 8) {
    const dim3 grid((num_tokens + 31) / 32, c.num_kv_heads);
    return launch_pdl(append_kernel<8>, grid, dim3(256), 0, s, k, v, kd, vd, slots, num_tokens,
                      c.num_kv_heads, nslots, status);
  }
  return cudaErrorInvalidValue;
}

template <QuantMode kMode>
cudaError_t launch_quant(const void* key, const void* value, bool src_bf16, void* k_cache,
                         void* v_cache, float* k_scale, float* v_scale, float fixed_ks,
                         float fixed_vs, const int32_t* slots, int num_tokens,
                         const kvp_cache_desc& c, int32_t* status, cudaStream_t s) {
  if (num_tokens == 0) return cudaSuccess;
  const int nslots = c.num_blocks * kBlockSize;
  const auto* k = static_cast<const uint4*>(key);
  const auto* v = static_cast<const uint4*>(value);
  auto* kd = static_cast<uint8_t*>(k_cache);
  auto* vd = static_cast<uint8_t*>(v_cache);
  const dim3 grid((num_tokens + kQuantRowsPerCta - 1) / kQuantRowsPerCta, c.num_kv_heads);
#define KVP_Q_CASE(BF, DD)                                                                     \
  if (src_bf16 == BF && c.head_dim == DD)                                                      \
    return launch_pdl(append_quant_kernel<BF, DD, kMode>, grid, dim3(256), 0, s, k, v, kd, vd, \
                      k_scale, v_scale, fixed_ks, fixed_vs, slots, num_tokens, c.num_kv_heads, \
                      nslots, status);
  KVP_Q_CASE(false, 64)
  KVP_Q_CASE(false, 128)
  KVP_Q_CASE(true, 64)
  KVP_Q_CASE(true, 128)
#undef KVP_Q_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_append_int8(const void* key, const void* value, bool src_bf16,
                               int8_t* k_cache, int8_t* v_cache, float* k_scale,
                               float* v_scale, const int32_t* slots, int num_tokens,
                               const kvp_cache_desc& c, int32_t* status, cudaStream_t s) {
  return launch_quant<QuantMode::kInt8>(key, value, src_bf16, k_cache, v_cache, k_scale, v_scale,
                                        0.f, 0.f, slots, num_tokens, c, status, s);
}

cudaError_t launch_append_int8_fixed(const void* key, const void* value, bool src_bf16,
                                     int8_t* k_cache, int8_t* v_cache, float* k_scale_pool,
                                     float* v_scale_pool, float k_scale, float v_scale,
                                     const int32_t* slots, int num_tokens,
                                     const kvp_cache_desc& c, int32_t* status, cudaStream_t s) {
  return launch_quant<QuantMode::kInt8Fixed>(key, value, src_bf16, k_cache, v_cache,
                                             k_scale_pool, v_scale_pool, k_scale, v_scale, slots,
                                             num_tokens, c, status, s);
}

cudaError_t launch_append_fp8(const void* key, const void* value, bool src_bf16,
                              uint8_t* k_cache, uint8_t* v_cache, float* k_scale, float* v_scale,
                              const int32_t* slots, int num_tokens, const kvp_cache_desc& c,
                              int32_t* status, cudaStream_t s) {
  return launch_quant<QuantMode::kFp8>(key, value, src_bf16, k_cache, v_cache, k_scale, v_scale,
                                       0.f, 0.f, slots, num_tokens, c, status, s);
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                               int elem_bytes, const int32_t* pairs, int num_pairs,
                               const kvp_cache_desc& c, int32_t* status, cudaStream_t s) {
  if (num_pairs == 0) return cudaSuccess;
  const long long block_bytes =
      static_cast<long long>(c.num_kv_heads) * kBlockSize * c.head_dim * elem_bytes;
  const long long chunks_kv = block_bytes / 16;
  const long long chunks_scale = static_cast<long long>(c.num_kv_heads) * kBlockSize * 4 / 16;
  long long gx = (chunks_kv + 1023) / 1024;  // ~4 chunks per thread
  if (gx < 1) gx = 1;
  if (gx > 1024) gx = 1024;
  const dim3 grid(static_cast<unsigned>(gx),
                  static_cast<unsigned>(num_pairs < 65535 ? num_pairs : 65535));
  return launch_pdl(copy_blocks_kernel, grid, dim3(256), 0, s, static_cast<uint4*>(k_cache),
                    static_cast<uint4*>(v_cache), reinterpret_cast<uint4*>(k_scale),
                    reinterpret_cast<uint4*>(v_scale), pairs, num_pairs, chunks_kv,
                    chunks_scale, c.num_blocks, status);
}

}  // namespace kvp

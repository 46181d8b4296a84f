// kvp_append.cu -- the write side of the paged cache:
//   * append: scatter new tokens' K/V rows to their slots ("KV Cache 优化与显存管理",
//     三, write_page; "ATB PagedAttention", "踩坑三", WriteKV), slot = block * 16 +
//     offset ("ATB 的 PagedAttention 实现": page = pos / size, offset = pos % size);
//   * append_int8: per token and head abs-max / 127 quantisation, then scatter
//     ("KV Cache 优化与显存管理", 三, KVCacheQuantizer per-channel branch);
//   * copy_blocks: whole-block copies for copy-on-write ("踩坑三", ExtendKVPage).
// All three are pure HBM streams: 16-byte vector loads and stores, one thread
// per 16-byte chunk, rows of a block contiguous so every warp access coalesces.
#include "kvp_device.cuh"
#include "kvp_internal.h"

namespace kvp {
namespace {

__global__ void __launch_bounds__(256)
    append_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                  uint4* __restrict__ kc, uint4* __restrict__ vc, const int32_t* __restrict__ slots,
                  long long total_chunks, int num_kv_heads, int chunks_per_row,
                  long long num_slots, int32_t* status) {
  dev::grid_dependency_wait();
  dev::launch_dependents();
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= total_chunks) return;
  const int ch = static_cast<int>(idx % chunks_per_row);
  const long long row = idx / chunks_per_row;  // t * Hkv + h
  const long long t = row / num_kv_heads;
  const int h = static_cast<int>(row % num_kv_heads);
  const int slot = slots[t];
  if (slot < 0) return;  // padding token
  if (slot >= num_slots) {
    if (h == 0 && ch == 0) dev::set_status(status, kErrBadBlock);
    return;
  }
  const long long blk = slot / kBlockSize, off = slot % kBlockSize;
  const long long dst = ((blk * num_kv_heads + h) * kBlockSize + off) * chunks_per_row + ch;
  kc[dst] = key[row * chunks_per_row + ch];
  vc[dst] = value[row * chunks_per_row + ch];
}

// rint(x / s) clipped to [-128, 127], with x / s the IEEE float32 quotient.
// r = x * (1/s) is within 2e-5 of x / s for |x / s| <= 127.0001 (two roundings
// of relative size 2^-24 each), and RN(x / s) within 8e-6 of it, so whenever r
// lies more than 1e-4 from a half-integer both round to the same integer; only
// inside that band is the exact quotient computed.
__device__ __forceinline__ int quantise_code(float x, float s, float inv) {
  const float r = x * inv;
  const float fl = floorf(r);
  const float frac = r - fl;
  int q;
  if (fabsf(frac - 0.5f) > 1.0e-4f) {
    q = static_cast<int>(frac > 0.5f ? fl + 1.0f : fl);
  } else {
    q = __float2int_rn(__fdiv_rn(x, s));
  }
  return min(127, max(-128, q));
}

// One group of D/4 lanes per (token, head) row; each lane owns 4 elements.
template <bool kBf16, int D>
__global__ void __launch_bounds__(256)
    append_int8_kernel(const uint16_t* __restrict__ key, const uint16_t* __restrict__ value,
                       int8_t* __restrict__ kc, int8_t* __restrict__ vc, float* __restrict__ ks,
                       float* __restrict__ vs, const int32_t* __restrict__ slots, long long rows,
                       int num_kv_heads, long long num_slots, int32_t* status) {
  constexpr int L = D / 4;
  dev::grid_dependency_wait();
  dev::launch_dependents();
  const long long gt = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = gt / L;
  const int sub = static_cast<int>(gt % L);
  const bool in = row < rows;
  int slot = -1;
  float xk[4] = {0.f, 0.f, 0.f, 0.f}, xv[4] = {0.f, 0.f, 0.f, 0.f};
  if (in) {
    slot = slots[row / num_kv_heads];
    const uint2 rk = *reinterpret_cast<const uint2*>(key + row * D + sub * 4);
    const uint2 rv = *reinterpret_cast<const uint2*>(value + row * D + sub * 4);
    const float2 k0 = dev::unpack2<kBf16>(rk.x), k1 = dev::unpack2<kBf16>(rk.y);
    const float2 v0 = dev::unpack2<kBf16>(rv.x), v1 = dev::unpack2<kBf16>(rv.y);
    xk[0] = k0.x; xk[1] = k0.y; xk[2] = k1.x; xk[3] = k1.y;
    xv[0] = v0.x; xv[1] = v0.y; xv[2] = v1.x; xv[3] = v1.y;
  }
  float ak = 0.f, av = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    ak = fmaxf(ak, fabsf(xk[e]));
    av = fmaxf(av, fabsf(xv[e]));
  }
#pragma unroll
  for (int o = L / 2; o >= 1; o >>= 1) {
    ak = fmaxf(ak, __shfl_xor_sync(0xffffffffu, ak, o));
    av = fmaxf(av, __shfl_xor_sync(0xffffffffu, av, o));
  }
  if (!in || slot < 0) return;
  const int h = static_cast<int>(row % num_kv_heads);
  if (slot >= num_slots) {
    if (sub == 0 && h == 0) dev::set_status(status, kErrBadBlock);
    return;
  }
  // float32 IEEE division and round-half-even, as the quantiser is defined
  float sk = __fdiv_rn(ak, 127.0f);
  float sv = __fdiv_rn(av, 127.0f);
  sk = sk > 0.f ? sk : 1.0f;
  sv = sv > 0.f ? sv : 1.0f;
  const float ik = __frcp_rn(sk), iv = __frcp_rn(sv);
  uint32_t pk = 0u, pv = 0u;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int qk = quantise_code(xk[e], sk, ik);
    const int qv = quantise_code(xv[e], sv, iv);
    pk |= (static_cast<uint32_t>(qk) & 0xffu) << (8 * e);
    pv |= (static_cast<uint32_t>(qv) & 0xffu) << (8 * e);
  }
  const long long blk = slot / kBlockSize, off = slot % kBlockSize;
  const long long srow = (blk * num_kv_heads + h) * kBlockSize + off;
  *reinterpret_cast<uint32_t*>(kc + srow * D + sub * 4) = pk;
  *reinterpret_cast<uint32_t*>(vc + srow * D + sub * 4) = pv;
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
  const int cpr = c.head_dim * elem_bytes / 16;
  const long long total = static_cast<long long>(num_tokens) * c.num_kv_heads * cpr;
  if (total == 0) return cudaSuccess;
  const long long grid = (total + 255) / 256;
  return launch_pdl(append_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s,
                    static_cast<const uint4*>(key), static_cast<const uint4*>(value),
                    static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slots, total,
                    c.num_kv_heads, cpr, static_cast<long long>(c.num_blocks) * kBlockSize,
                    status);
}

cudaError_t launch_append_int8(const void* key, const void* value, bool src_bf16,
                               int8_t* k_cache, int8_t* v_cache, float* k_scale,
                               float* v_scale, const int32_t* slots, int num_tokens,
                               const kvp_cache_desc& c, int32_t* status, cudaStream_t s) {
  const long long rows = static_cast<long long>(num_tokens) * c.num_kv_heads;
  if (rows == 0) return cudaSuccess;
  const long long threads = rows * (c.head_dim / 4);
  const unsigned grid = static_cast<unsigned>((threads + 255) / 256);
  const long long nslots = static_cast<long long>(c.num_blocks) * kBlockSize;
  const uint16_t* k = static_cast<const uint16_t*>(key);
  const uint16_t* v = static_cast<const uint16_t*>(value);
#define KVP_I8_CASE(BF, DD)                                                                   \
  if (src_bf16 == BF && c.head_dim == DD) {                                                   \
    return launch_pdl(append_int8_kernel<BF, DD>, dim3(grid), dim3(256), 0, s, k, v,         \
                      k_cache, v_cache, k_scale, v_scale, slots, rows, c.num_kv_heads,        \
                      nslots, status);                                                        \
  }
  KVP_I8_CASE(false, 64)
  KVP_I8_CASE(false, 128)
  KVP_I8_CASE(true, 64)
  KVP_I8_CASE(true, 128)
#undef KVP_I8_CASE
  return cudaErrorInvalidValue;
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

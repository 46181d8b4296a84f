// kvp_prefill.cu -- multi-query (prefill / chunked-prefill) paged attention on
// the 5th-generation tensor cores.
//
// What is computed ("ATB KV Cache management", "Prefix Caching": requests that
// share a system prompt reuse its cached K/V and only their own part is new):
// request b holds n = context_lens[b] cached tokens whose last L are this
// chunk's queries (their K/V already appended); query i of the chunk sits at
// position n - L + i and attends causally to positions 0 .. n - L + i through
// the block table.  Unlike the decode, this is a dense contraction: a 128-row
// query tile against 64-key tiles.
//
// Design (one CTA of 4 warps per (request, kv head, 128-row query tile)):
//   * Tile rows are (query token, query head of the kv head's group) pairs, so
//     every K/V byte a tile reads serves the whole GQA group.
//   * Per 64-key chunk (4 blocks): TMA copies the K and V tiles of the chunk's
//     4 blocks into one of two shared-memory stages (128-byte swizzle, the
//     layout the tensor core reads directly); one thread issues
//     S = Q K^T as tcgen05.mma (M=128, N=64, K=D) into tensor memory.
//   * Thread r owns TMEM lane r, i.e. query row r: it loads its 64 scores,
//     applies the causal mask and the scale, and keeps the row's running max
//     and sum in registers -- no shuffles.  The running max is updated lazily:
//     only when a row's max grows by more than 2^8 are its O columns rescaled
//     in TMEM (exact, since numerator and denominator share the stale max).
//   * P goes to shared memory (fp16; bf16 as a high part plus a bf16 residual
//     so P keeps ~16 bits) and one thread issues O += P V (M=128, N=D, K=64).
//   * At the end each thread divides its O row by its sum and writes it out.
#include "kvp_device.cuh"
#include "kvp_internal.h"
#include "kvp_umma.cuh"

namespace kvp {
namespace {

constexpr int kRows = 128;             // M: query rows per CTA
constexpr int kKeys = 64;              // key tokens per chunk
constexpr int kThreads = 128;

template <bool kBf16, int D>
struct PrefillLayout {
  static constexpr int kHalves = D / 64;                  // 64-element K-major halves
  static constexpr uint32_t kQ = kRows * D * 2;           // Q tile
  static constexpr uint32_t kKV = kKeys * D * 2;          // one K or V stage
  static constexpr uint32_t kP = kRows * kKeys * 2;       // P tile (one part)
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKOff = kQ;                   // K stages 0, 1
  static constexpr uint32_t kVOff = kQ + 2 * kKV;         // V stages 0, 1
  static constexpr uint32_t kPOff = kQ + 4 * kKV;
  static constexpr uint32_t kPloOff = kPOff + kP;
  static constexpr uint32_t kBarOff = kPloOff + (kBf16 ? kP : 0);
  static constexpr size_t kSmem = 1024 + kBarOff + 64;    // + alignment slack, barriers, slot
  // TMEM: S in columns [0, 64), O in [kOCol, kOCol + D); a power of two >= 32
  // columns, small enough for every CTA the shared memory lets reside on an SM
  static constexpr uint32_t kOCol = D == 64 ? 64 : 128;
  static constexpr uint32_t kTmemCols = D == 64 ? 128 : 256;
};

// Swizzled offset of 16-byte chunk c of row r in a 128-byte-row tile.
__device__ __forceinline__ uint32_t sw_chunk(int r, int c) {
  return static_cast<uint32_t>(r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

template <int D>
__device__ __forceinline__ void zero_tile_rows(const PrefillParams& p, int kvh, int q0, int t0,
                                               int ntok) {
  const int G = p.group;
  uint16_t* out = static_cast<uint16_t*>(p.out);
  for (int idx = threadIdx.x; idx < ntok * G * D; idx += blockDim.x) {
    const int t = idx / (G * D), g = (idx / D) % G, d = idx % D;
    out[(static_cast<size_t>(q0 + t0 + t) * p.num_q_heads + kvh * G + g) * D + d] = 0;
  }
}

template <bool kBf16, int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv) {
  using namespace dev;
  using L = PrefillLayout<kBf16, D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sQ = sm + L::kQOff;
  uint8_t* sP = sm + L::kPOff;
  uint8_t* sPlo = sm + L::kPloOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBarOff);  // kv[0], kv[1], s, pv
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int b = blockIdx.z, kvh = blockIdx.y, tile = blockIdx.x;
  const int G = p.group;
  const int tok_per_tile = kRows / G;

  grid_dependency_wait();
  const int q0 = p.query_start[b];
  const int qlen = p.query_start[b + 1] - q0;
  const int n = p.context_lens[b];
  const int t0 = tile * tok_per_tile;
  // rows past the grid's coverage (a chunk longer than the launch's maximum)
  if (tile == gridDim.x - 1 && tid == 0 && qlen > static_cast<int>(gridDim.x) * tok_per_tile)
    set_status(p.status, kErrBadBlock);
  if (qlen <= 0 || t0 >= qlen) return;
  const int ntok = min(tok_per_tile, qlen - t0);
  if (qlen > n || n > p.max_blocks * kBlockSize) {
    zero_tile_rows<D>(p, kvh, q0, t0, ntok);
    if (tid == 0) set_status(p.status, kErrBadBlock);
    return;
  }
  const int pos0 = n - qlen + t0;  // position of this tile's first query token
  const int nkeys = pos0 + ntok;   // keys needed: 0 .. nkeys - 1
  const int nblk = (nkeys + kBlockSize - 1) / kBlockSize;
  const int nchunks = (nkeys + kKeys - 1) / kKeys;
  const int32_t* tbl = p.block_tables + static_cast<size_t>(b) * p.max_blocks;
  bool bad = false;
  for (int i = tid; i < nblk; i += kThreads) {
    const int id = tbl[i];
    bad |= (id < 0) || (id >= p.num_blocks);
  }
  if (__syncthreads_or(bad)) {
    zero_tile_rows<D>(p, kvh, q0, t0, ntok);
    if (tid == 0) set_status(p.status, kErrBadBlock);
    return;
  }

  // ---- Q tile: row r = (query token r / G, query head r % G), K-major swizzled
  const int my_t = tid / G;
  const int my_g = tid % G;
  const bool row_valid = my_t < ntok;
  {
    const uint4* src =
        reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                       (static_cast<size_t>(q0 + t0 + (row_valid ? my_t : 0)) *
                                            p.num_q_heads +
                                        kvh * G + my_g) *
                                           D);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const uint4 v = row_valid ? src[c] : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(sQ + (c >> 3) * (kRows * 128) + sw_chunk(tid, c)) = v;
    }
  }
  fence_proxy_async_smem();  // Q is read by the tensor core (async proxy)
  if (tid == 0) {
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
#pragma unroll
    for (int i = 0; i < 4; ++i) mbar_init(smem_addr(bars + i), 1);
    fence_barrier_init();
  }
  if (warp == 0) umma::alloc(smem_addr(tmem_slot), L::kTmemCols);
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;
  const uint32_t tO = tmem + L::kOCol;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

  auto issue = [&](int j) {  // thread 0: K and V tiles of chunk j into stage j & 1
    const int st = j & 1;
    const int blk0 = j * (kKeys / kBlockSize);
    const int nb = min(kKeys / kBlockSize, nblk - blk0);
    const uint32_t bar = smem_addr(bars + st);
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nb * 2 * L::kHalves * 2048));
    for (int i = 0; i < nb; ++i) {
      const int y = (tbl[blk0 + i] * p.num_kv_heads + kvh) * kBlockSize;
#pragma unroll
      for (int hf = 0; hf < L::kHalves; ++hf) {
        const uint32_t off = hf * (kKeys * 128) + i * 2048;
        tma_load_2d(smem_addr(sm + L::kKOff + st * L::kKV + off), &tmk, hf * 64, y, bar);
        tma_load_2d(smem_addr(sm + L::kVOff + st * L::kKV + off), &tmv, hf * 64, y, bar);
      }
    }
  };
  if (tid == 0) {
    issue(0);
    if (nchunks > 1) issue(1);
  }

  const int qpos = pos0 + my_t;
  const float sl2 = p.scale_log2;
  constexpr uint32_t kIdS = umma::instr_desc_f16(kRows, kKeys, kBf16, false, false);
  constexpr uint32_t kIdO = umma::instr_desc_f16(kRows, D, kBf16, false, true);
  float m = -INFINITY, l = 0.f;
  bool ok = true;

  for (int j = 0; j < nchunks; ++j) {
    const int st = j & 1;
    uint8_t* sK = sm + L::kKOff + st * L::kKV;
    uint8_t* sV = sm + L::kVOff + st * L::kKV;
    ok &= mbar_wait_bounded(smem_addr(bars + st), (j >> 1) & 1);
    // rows past the context or past the loaded blocks: clear K and V so no
    // stale or NaN bytes reach the tensor core (masked scores get P = 0)
    const int zero_from = min(n, nblk * kBlockSize) - j * kKeys;
    if (zero_from < kKeys) {
      const int first = zero_from > 0 ? zero_from : 0;
      for (int idx = tid; idx < (kKeys - first) * L::kHalves * 8; idx += kThreads) {
        const int row = first + idx / (L::kHalves * 8);
        const int rem = idx % (L::kHalves * 8);
        const uint32_t off = (rem >> 3) * (kKeys * 128) + row * 128 + ((rem & 7) << 4);
        *reinterpret_cast<uint4*>(sK + off) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(sV + off) = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
    }
    umma::fence_before_sync();
    __syncthreads();
    // ---- S = Q K^T
    if (tid == 0) {
      umma::fence_after_sync();
#pragma unroll
      for (int s = 0; s < D / 16; ++s) {
        const uint32_t qoff = (s >> 2) * (kRows * 128) + (s & 3) * 32;
        const uint32_t koff = (s >> 2) * (kKeys * 128) + (s & 3) * 32;
        umma::mma_f16(tS, umma::smem_desc_sw128(smem_addr(sQ) + qoff, 16, 1024),
                      umma::smem_desc_sw128(smem_addr(sK) + koff, 16, 1024), kIdS,
                      s > 0 ? 1u : 0u);
      }
      umma::commit(smem_addr(bars + 2));
    }
    ok &= mbar_wait_bounded(smem_addr(bars + 2), j & 1);
    umma::fence_after_sync();
    float sa[32], sb[32];
    umma::ld32(tS + lane_base, sa);
    umma::ld32(tS + lane_base + 32, sb);
    umma::wait_ld();
    float rowmax = -INFINITY;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const int ka = j * kKeys + k, kb = ka + 32;
      sa[k] = (row_valid && ka <= qpos) ? sa[k] * sl2 : -INFINITY;
      sb[k] = (row_valid && kb <= qpos) ? sb[k] * sl2 : -INFINITY;
      rowmax = fmaxf(rowmax, fmaxf(sa[k], sb[k]));
    }
    // ---- O and P are free once the previous chunk's P V has completed
    if (j > 0) {
      ok &= mbar_wait_bounded(smem_addr(bars + 3), (j - 1) & 1);
      umma::fence_after_sync();
    }
    if (tid == 0 && j >= 1 && j + 1 < nchunks) issue(j + 1);  // its stage was chunk j-1's
    const float mnew = fmaxf(m, rowmax);
    const bool grow = mnew > m + 8.0f;  // lazy: rescale only when the max grows by > 2^8
    if (__any_sync(0xffffffffu, grow && j > 0)) {
      const float alpha = grow ? exp2f(m - mnew) : 1.0f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        umma::ld32(tO + lane_base + c * 32, o);
        umma::wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] *= alpha;
        umma::st32(tO + lane_base + c * 32, o);
      }
      umma::wait_st();
    }
    if (grow) {
      l *= exp2f(m - mnew);
      m = mnew;
    }
    // ---- P row (64 keys) into the K-major swizzled P tile
    float psum = 0.f;
    uint32_t hi[32], lo[32];
#pragma unroll
    for (int k = 0; k < 32; k += 2) {
      const float p0 = sa[k] == -INFINITY ? 0.f : exp2f(sa[k] - m);
      const float p1 = sa[k + 1] == -INFINITY ? 0.f : exp2f(sa[k + 1] - m);
      const float p2 = sb[k] == -INFINITY ? 0.f : exp2f(sb[k] - m);
      const float p3 = sb[k + 1] == -INFINITY ? 0.f : exp2f(sb[k + 1] - m);
      psum += (p0 + p1) + (p2 + p3);
      hi[k / 2] = pack2<kBf16>(p0, p1);
      hi[16 + k / 2] = pack2<kBf16>(p2, p3);
      if constexpr (kBf16) {
        const float2 h01 = unpack2<true>(hi[k / 2]);
        const float2 h23 = unpack2<true>(hi[16 + k / 2]);
        lo[k / 2] = pack2<true>(p0 - h01.x, p1 - h01.y);
        lo[16 + k / 2] = pack2<true>(p2 - h23.x, p3 - h23.y);
      }
    }
    l += psum;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      *reinterpret_cast<uint4*>(sP + sw_chunk(tid, c)) =
          make_uint4(hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
      if constexpr (kBf16) {
        *reinterpret_cast<uint4*>(sPlo + sw_chunk(tid, c)) =
            make_uint4(lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
      }
    }
    fence_proxy_async_smem();
    umma::fence_before_sync();
    __syncthreads();
    // ---- O += P V
    if (tid == 0) {
      umma::fence_after_sync();
#pragma unroll
      for (int t = 0; t < kKeys / 16; ++t) {
        const uint64_t vd = umma::smem_desc_sw128(smem_addr(sV) + t * 2048, kKeys * 128, 1024);
        umma::mma_f16(tO, umma::smem_desc_sw128(smem_addr(sP) + t * 32, 16, 1024), vd, kIdO,
                      (j > 0 || t > 0) ? 1u : 0u);
        if constexpr (kBf16) {
          umma::mma_f16(tO, umma::smem_desc_sw128(smem_addr(sPlo) + t * 32, 16, 1024), vd, kIdO,
                        1u);
        }
      }
      umma::commit(smem_addr(bars + 3));
    }
  }

  ok &= mbar_wait_bounded(smem_addr(bars + 3), (nchunks - 1) & 1);
  umma::fence_after_sync();
  launch_dependents();
  // ---- out row = O / l
  const float inv = (row_valid && l > 0.f) ? 1.0f / l : 0.f;
  uint16_t* out = static_cast<uint16_t*>(p.out) +
                  (static_cast<size_t>(q0 + t0 + (row_valid ? my_t : 0)) * p.num_q_heads +
                   kvh * G + my_g) *
                      D;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    float o[32];
    umma::ld32(tO + lane_base + c * 32, o);
    umma::wait_ld();
    if (row_valid) {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint4 w;
        w.x = pack2<kBf16>(o[8 * q4] * inv, o[8 * q4 + 1] * inv);
        w.y = pack2<kBf16>(o[8 * q4 + 2] * inv, o[8 * q4 + 3] * inv);
        w.z = pack2<kBf16>(o[8 * q4 + 4] * inv, o[8 * q4 + 5] * inv);
        w.w = pack2<kBf16>(o[8 * q4 + 6] * inv, o[8 * q4 + 7] * inv);
        *reinterpret_cast<uint4*>(out + c * 32 + 8 * q4) = w;
      }
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 0) umma::dealloc(tmem, L::kTmemCols);
  if (!__syncthreads_and(ok) && tid == 0) set_status(p.status, kErrTimeout);
}

template <bool kBf16, int D>
cudaError_t launch_prefill_t(const PrefillParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                             int grid_x, cudaStream_t s) {
  constexpr size_t smem = PrefillLayout<kBf16, D>::kSmem;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(&prefill_kernel<kBf16, D>), smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(grid_x, p.num_kv_heads, p.batch);
  return launch_pdl(prefill_kernel<kBf16, D>, grid, dim3(kThreads), smem, s, p, tk, tv);
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                           bool bf16, int grid_x, cudaStream_t s) {
  if (!bf16 && p.head_dim == 64) return launch_prefill_t<false, 64>(p, tk, tv, grid_x, s);
  if (!bf16 && p.head_dim == 128) return launch_prefill_t<false, 128>(p, tk, tv, grid_x, s);
  if (bf16 && p.head_dim == 64) return launch_prefill_t<true, 64>(p, tk, tv, grid_x, s);
  if (bf16 && p.head_dim == 128) return launch_prefill_t<true, 128>(p, tk, tv, grid_x, s);
  return cudaErrorInvalidValue;
}

}  // namespace kvp

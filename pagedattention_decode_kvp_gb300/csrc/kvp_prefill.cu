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
//   * K/V arrive in 64-key chunks (4 blocks) through separate K and V rings
//     in shared memory: TMA copies (128-byte swizzle, the layout the tensor
//     core reads directly) issued by four producer warps, one per block slot
//     of a chunk, so copy issue is spread over several threads.
//   * One thread issues the tensor-core work: S = Q K^T (tcgen05.mma, M=128,
//     N=64, K=D) into TMEM score buffers two chunks ahead of the softmax, and
//     O += P V (M=128, N=D, K=64) into a TMEM accumulator, so the tensor core
//     works while the CUDA cores exponentiate.
//   * Thread r owns TMEM lane r, i.e. query row r: it loads its 64 scores,
//     applies the causal mask and the scale, and keeps the row's running max
//     and sum in registers -- no shuffles.  The running max is updated lazily:
//     only when a row's max grows by more than 2^8 are its O columns rescaled
//     in TMEM (exact, since numerator and denominator share the stale max).
//   * P goes to shared memory (fp16; bf16 as a high part plus a bf16 residual
//     so P keeps ~16 bits).
//   * At the end each thread divides its O row by its sum and writes it out.
#include "kvp_device.cuh"
#include "kvp_internal.h"
#include "kvp_umma.cuh"

namespace kvp {
namespace {

constexpr int kRows = 128;                            // M: query rows per CTA
constexpr int kKeys = 64;                             // key tokens per chunk
constexpr int kSoftmaxWarps = 8;                      // two per TMEM lane quarter
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kMmaWarp = kSoftmaxWarps;               // issues the tensor-core work
constexpr int kProducerWarps = 4;                     // TMA issue, one per block of a chunk
constexpr int kThreads = kSoftmaxThreads + 32 + kProducerWarps * 32;
constexpr int kSmemPerSm = 233472;                    // shared memory of one SM (bytes)
constexpr int kTableCap = 1024;                       // block ids staged on chip per tile

template <bool kBf16, int D>
struct PrefillLayout {
  static constexpr int kHalves = D / 64;                  // 64-element K-major halves
  static constexpr uint32_t kQ = kRows * D * 2;           // Q tile
  static constexpr uint32_t kKV = kKeys * D * 2;          // one K or V tile
  static constexpr uint32_t kP = kRows * kKeys * 2;       // one P tile
  static constexpr uint32_t kPBuf = kBf16 ? 2 * kP : kP;  // P (and its bf16 residual)
  // Separate K and V rings: a K stage is free once its S is computed, a V
  // stage once its P V is; depths fill the shared memory left by Q and P.
  static constexpr int kKStages = D == 64 ? 6 : (kBf16 ? 4 : 5);
  static constexpr int kVStages = D == 64 ? 5 : (kBf16 ? 3 : 4);
  static constexpr int kAhead = 2;                        // S computed 2 chunks ahead
  static constexpr int kSBufs = kAhead + 1;               // TMEM score buffers
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKOff = kQ;
  static constexpr uint32_t kVOff = kKOff + kKStages * kKV;
  static constexpr uint32_t kPOff = kVOff + kVStages * kKV;  // 2 P buffers
  static constexpr uint32_t kRedOff = kPOff + 2 * kPBuf;  // [2][2][kRows] float
  static constexpr uint32_t kTblOff = kRedOff + 2 * 2 * kRows * 4;  // [kTableCap] int32
  static constexpr uint32_t kBarOff = kTblOff + kTableCap * 4;
  // kfull[], vfull[], kempty[], vempty[], s[], pv[2], p[2]
  static constexpr int kBars = 2 * (kKStages + kVStages) + kSBufs + 4;
  // + 1024 bytes of alignment slack, the barriers and the TMEM address slot
  static constexpr size_t kSmem = 1024 + kBarOff + kBars * 8 + 16;
  // TMEM columns: score buffer i at [64 i, 64 i + 64), O at [256, 256 + D).
  // The shared memory keeps a second CTA off the SM, so all 512 columns are free.
  static constexpr uint32_t kOCol = 256;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kSBufs * kKeys <= static_cast<int>(kOCol), "score buffers overlap O");
  static_assert(2 * (kSmem + 1024) > kSmemPerSm, "TMEM budget assumes one CTA per SM");
  static_assert(kSmem <= 232448, "exceeds the per-block shared-memory limit");
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

// Warp roles: warps 0-7 run the softmax -- warp w serves query rows
// 32*(w%4) .. +31 (the TMEM lanes it may access) for keys [32*(w/4), +32) of
// each chunk and O columns [D/2*(w/4), +D/2); warp 8 (one thread) issues the
// tensor-core instructions; warps 9-12 are producers -- producer i copies
// block i of every chunk (its lane 0 the K tile, lane 1 the V tile).
// Hand-offs (mbarriers; every wait is at most one phase behind its barrier):
//   kfull[c % kKStages]   producers -> MMA    chunk c's K landed (4 arrivals + bytes)
//   vfull[c % kVStages]   producers -> MMA    chunk c's V landed
//   kempty[c % kKStages]  MMA -> producers    S(c) done: K stage free
//   vempty[c % kVStages]  MMA -> producers    P V(c) done: V stage free
//   s[c % kSBufs]         MMA -> softmax      S of chunk c in score buffer c % kSBufs
//   p[c % 2]              softmax -> MMA      P of chunk c in P buffer c % 2 (8 arrivals)
//   pv[c % 2]             MMA -> softmax      O += P V of chunk c complete
// Per chunk j the MMA thread waits p(j) and V(j), issues P V(j), then S(j +
// kAhead).  The softmax of chunk j needs only S(j) -- P buffer j%2 was freed
// by P V(j-2), and O is touched (lazy rescale, after P V(j-1)) only when a
// row's max jumps.
template <bool kBf16, int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv) {
  using namespace dev;
  using L = PrefillLayout<kBf16, D>;
  constexpr int kKStages = L::kKStages;
  constexpr int kVStages = L::kVStages;
  constexpr int kSBufs = L::kSBufs;
  constexpr int kAhead = L::kAhead;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sQ = sm + L::kQOff;
  float* red = reinterpret_cast<float*>(sm + L::kRedOff);
  int32_t* stbl = reinterpret_cast<int32_t*>(sm + L::kTblOff);
  uint64_t* kf_bar = reinterpret_cast<uint64_t*>(sm + L::kBarOff);  // [kKStages]
  uint64_t* vf_bar = kf_bar + kKStages;                              // [kVStages]
  uint64_t* ke_bar = vf_bar + kVStages;                              // [kKStages]
  uint64_t* ve_bar = ke_bar + kKStages;                              // [kVStages]
  uint64_t* s_bar = ve_bar + kVStages;                               // [kSBufs]
  uint64_t* pv_bar = s_bar + kSBufs;                                 // [2]
  uint64_t* p_bar = pv_bar + 2;                                      // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(p_bar + 2);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool mma_warp = warp == kMmaWarp;
  const bool producer = warp > kMmaWarp;
  const int quarter = warp & 3;
  const int half = (warp >> 2) & 1;
  const int row = quarter * 32 + lane;
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
  // range-check every block id the tile reads; the first kTableCap are kept on
  // chip so the copy issuer never waits on a global load
  bool bad = false;
  for (int i = tid; i < nblk; i += kThreads) {
    const int id = tbl[i];
    bad |= (id < 0) || (id >= p.num_blocks);
    if (i < kTableCap) stbl[i] = id;
  }
  if (__syncthreads_or(bad)) {
    zero_tile_rows<D>(p, kvh, q0, t0, ntok);
    if (tid == 0) set_status(p.status, kErrBadBlock);
    return;
  }

  // ---- Q tile: row r = (query token r / G, query head r % G), K-major
  // swizzled; softmax thread (row, half) stores half of its row
  const int my_t = row / G;
  const int my_g = row % G;
  const bool row_valid = warp < kSoftmaxWarps && my_t < ntok;
  if (warp < kSoftmaxWarps) {
    const uint4* src =
        reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                       (static_cast<size_t>(q0 + t0 + (row_valid ? my_t : 0)) *
                                            p.num_q_heads +
                                        kvh * G + my_g) *
                                           D);
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      const int c = half * (D / 16) + i;
      const uint4 v = row_valid ? src[c] : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(sQ + (c >> 3) * (kRows * 128) + sw_chunk(row, c)) = v;
    }
    fence_proxy_async_smem();  // Q is read by the tensor core (async proxy)
  } else if (mma_warp) {
    if (lane == 0) {
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
      for (int i = 0; i < kKStages + kVStages; ++i)
        mbar_init(smem_addr(kf_bar + i), kProducerWarps);
      for (int i = kKStages + kVStages; i < 2 * (kKStages + kVStages) + kSBufs + 2; ++i)
        mbar_init(smem_addr(kf_bar + i), 1);
      mbar_init(smem_addr(p_bar), kSoftmaxWarps);
      mbar_init(smem_addr(p_bar + 1), kSoftmaxWarps);
      fence_barrier_init();
    }
    __syncwarp();
    umma::alloc(smem_addr(tmem_slot), L::kTmemCols);
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (producer) {
    if (lane < 2) {
      // lane 0 streams K tiles, lane 1 V tiles: block `slot` of every chunk
      const int slot = warp - kMmaWarp - 1;
      const bool is_k = lane == 0;
      const CUtensorMap* map = is_k ? &tmk : &tmv;
      const int nst = is_k ? kKStages : kVStages;
      uint64_t* full = is_k ? kf_bar : vf_bar;
      uint64_t* empty = is_k ? ke_bar : ve_bar;
      uint8_t* ring = sm + (is_k ? L::kKOff : L::kVOff);
      for (int c = 0; c < nchunks; ++c) {
        const int st = c % nst;
        if (c >= nst) ok &= mbar_wait_bounded(smem_addr(empty + st), ((c / nst) - 1) & 1);
        const int blk = c * (kKeys / kBlockSize) + slot;
        const bool has = blk < nblk;
        const uint32_t bar = smem_addr(full + st);
        mbar_arrive_expect_tx(bar, has ? static_cast<uint32_t>(L::kHalves * 2048) : 0u);
        if (has) {
          const int id = blk < kTableCap ? stbl[blk] : tbl[blk];
          const int y = (id * p.num_kv_heads + kvh) * kBlockSize;
          uint8_t* dst = ring + st * L::kKV + slot * 2048;
#pragma unroll
          for (int hf = 0; hf < L::kHalves; ++hf)
            tma_load_2d(smem_addr(dst + hf * (kKeys * 128)), map, hf * 64, y, bar);
        }
      }
    }
    __syncwarp();
  } else if (mma_warp) {
    if (lane == 0) {
      auto k_tile = [&](int c) { return sm + L::kKOff + (c % kKStages) * L::kKV; };
      auto v_tile = [&](int c) { return sm + L::kVOff + (c % kVStages) * L::kKV; };
      constexpr uint32_t kIdS = umma::instr_desc_f16(kRows, kKeys, kBf16, false, false);
      constexpr uint32_t kIdO = umma::instr_desc_f16(kRows, D, kBf16, false, true);
      const uint32_t qa = smem_addr(sQ);
      auto issue_s = [&](int c) {  // wait for chunk c's K, S(c) = Q K(c)^T, free the K stage
        ok &= mbar_wait_bounded(smem_addr(kf_bar + c % kKStages), (c / kKStages) & 1);
        umma::fence_after_sync();
        const uint32_t ka = smem_addr(k_tile(c));
        const uint32_t d = tmem + (c % kSBufs) * kKeys;
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint32_t qoff = (s >> 2) * (kRows * 128) + (s & 3) * 32;
          const uint32_t koff = (s >> 2) * (kKeys * 128) + (s & 3) * 32;
          umma::mma_f16(d, umma::smem_desc_sw128(qa + qoff, 16, 1024),
                        umma::smem_desc_sw128(ka + koff, 16, 1024), kIdS, s > 0 ? 1u : 0u);
        }
        umma::commit(smem_addr(s_bar + c % kSBufs));
        umma::commit(smem_addr(ke_bar + c % kKStages));
      };

      for (int c = 0; c < min(kAhead, nchunks); ++c) issue_s(c);
      for (int j = 0; j < nchunks; ++j) {
        ok &= mbar_wait_bounded(smem_addr(p_bar + (j & 1)), (j >> 1) & 1);
        ok &= mbar_wait_bounded(smem_addr(vf_bar + j % kVStages), (j / kVStages) & 1);
        umma::fence_after_sync();
        const uint32_t pa = smem_addr(sm + L::kPOff + (j & 1) * L::kPBuf);
        const uint32_t va = smem_addr(v_tile(j));
#pragma unroll
        for (int t = 0; t < kKeys / 16; ++t) {
          const uint64_t vd = umma::smem_desc_sw128(va + t * 2048, kKeys * 128, 1024);
          umma::mma_f16(tmem + L::kOCol, umma::smem_desc_sw128(pa + t * 32, 16, 1024), vd, kIdO,
                        (j > 0 || t > 0) ? 1u : 0u);
          if constexpr (kBf16) {
            umma::mma_f16(tmem + L::kOCol, umma::smem_desc_sw128(pa + L::kP + t * 32, 16, 1024),
                          vd, kIdO, 1u);
          }
        }
        umma::commit(smem_addr(pv_bar + (j & 1)));
        umma::commit(smem_addr(ve_bar + j % kVStages));
        // S(j+kAhead): its score buffer was last read by the softmax of chunk
        // j-1, which handed off before P V(j-1) was issued
        if (j + kAhead < nchunks) issue_s(j + kAhead);
      }
    }
    __syncwarp();
    launch_dependents();
  } else {
    const int qpos = pos0 + my_t;
    const float sl2 = p.scale_log2;
    // scores are scaled inside the exponent's FMA when the scale is positive
    // (max and mask commute with it); otherwise they are scaled first
    const bool pos_scale = sl2 > 0.f;
    const float mul = pos_scale ? sl2 : 1.0f;
    float m = -INFINITY, l = 0.f;  // running max (log2 units) and this half's sum
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tOh = tmem + L::kOCol + half * (D / 2) + lane_base;
    for (int j = 0; j < nchunks; ++j) {
      ok &= mbar_wait_bounded(smem_addr(s_bar + j % kSBufs), (j / kSBufs) & 1);
      umma::fence_after_sync();
      float s[32];
      umma::ld32(tmem + (j % kSBufs) * kKeys + half * 32 + lane_base, s);
      umma::wait_ld();
      const int kbase = j * kKeys + half * 32;
      if (j * kKeys + kKeys - 1 > pos0) {  // chunk reaches past some row's position
#pragma unroll
        for (int k = 0; k < 32; ++k) s[k] = (row_valid && kbase + k <= qpos) ? s[k] : -INFINITY;
      }
      if (!pos_scale) {
#pragma unroll
        for (int k = 0; k < 32; ++k) s[k] = s[k] == -INFINITY ? -INFINITY : s[k] * sl2;
      }
      float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]);
      float mx2 = fmaxf(s[4], s[5]), mx3 = fmaxf(s[6], s[7]);
#pragma unroll
      for (int k = 8; k < 32; k += 8) {
        mx0 = fmaxf(mx0, fmaxf(s[k], s[k + 1]));
        mx1 = fmaxf(mx1, fmaxf(s[k + 2], s[k + 3]));
        mx2 = fmaxf(mx2, fmaxf(s[k + 4], s[k + 5]));
        mx3 = fmaxf(mx3, fmaxf(s[k + 6], s[k + 7]));
      }
      float rowmax = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * mul;
      // the partner warp holds the row's other 32 keys
      float* rb = red + (j & 1) * (2 * kRows);
      rb[half * kRows + row] = rowmax;
      named_bar_sync(1 + quarter, 64);
      rowmax = fmaxf(rowmax, rb[(1 - half) * kRows + row]);
      const float mnew = fmaxf(m, rowmax);
      const bool grow = mnew > m + 8.0f;  // lazy: rescale only when the max grows by > 2^8
      const float alpha = grow ? ex2_approx(m - mnew) : 1.0f;
      if (grow) {
        l *= alpha;
        m = mnew;
      }
      // ---- this half of the P row (32 keys), into registers
      const float negm = -m;
      float ps0 = 0.f, ps1 = 0.f, ps2 = 0.f, ps3 = 0.f;
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int k = 0; k < 32; k += 4) {
        const float p0 = ex2_approx(fmaf(s[k], mul, negm));
        const float p1 = ex2_approx(fmaf(s[k + 1], mul, negm));
        const float p2 = ex2_approx(fmaf(s[k + 2], mul, negm));
        const float p3 = ex2_approx(fmaf(s[k + 3], mul, negm));
        ps0 += p0;
        ps1 += p1;
        ps2 += p2;
        ps3 += p3;
        hi[k / 2] = pack2<kBf16>(p0, p1);
        hi[k / 2 + 1] = pack2<kBf16>(p2, p3);
        if constexpr (kBf16) {
          const float2 h01 = unpack2<true>(hi[k / 2]);
          const float2 h23 = unpack2<true>(hi[k / 2 + 1]);
          lo[k / 2] = pack2<true>(p0 - h01.x, p1 - h01.y);
          lo[k / 2 + 1] = pack2<true>(p2 - h23.x, p3 - h23.y);
        }
      }
      l += (ps0 + ps1) + (ps2 + ps3);
      // ---- O: rescale the rows whose max jumped, once P V(j-1) is in it
      if (__any_sync(0xffffffffu, grow && j > 0)) {
        ok &= mbar_wait_bounded(smem_addr(pv_bar + ((j - 1) & 1)), ((j - 1) >> 1) & 1);
        umma::fence_after_sync();
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          float o[32];
          umma::ld32(tOh + c * 32, o);
          umma::wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          umma::st32(tOh + c * 32, o);
        }
        umma::wait_st();
      }
      // ---- P buffer j%2 is free once P V(j-2) is done
      if (j >= 2) ok &= mbar_wait_bounded(smem_addr(pv_bar + (j & 1)), ((j - 2) >> 1) & 1);
      uint8_t* sP = sm + L::kPOff + (j & 1) * L::kPBuf;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        *reinterpret_cast<uint4*>(sP + sw_chunk(row, 4 * half + c)) =
            make_uint4(hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
        if constexpr (kBf16) {
          *reinterpret_cast<uint4*>(sP + L::kP + sw_chunk(row, 4 * half + c)) =
              make_uint4(lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
        }
      }
      if (j == nchunks - 1 && nkeys - j * kKeys < kKeys) {
        // V rows of keys >= nkeys are never attended (P = 0) but may hold
        // non-finite bytes (slots past the context, blocks not loaded): clear
        // them once the chunk's copies have landed
        ok &= mbar_wait_bounded(smem_addr(vf_bar + j % kVStages), (j / kVStages) & 1);
        uint8_t* sV = sm + L::kVOff + (j % kVStages) * L::kKV;
        const int first = nkeys - j * kKeys;
        for (int idx = tid; idx < (kKeys - first) * L::kHalves * 8; idx += kSoftmaxThreads) {
          const int r = first + idx / (L::kHalves * 8);
          const int rem = idx % (L::kHalves * 8);
          *reinterpret_cast<uint4*>(sV + (rem >> 3) * (kKeys * 128) + r * 128 +
                                    ((rem & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      umma::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(p_bar + (j & 1)));
    }

    ok &= mbar_wait_bounded(smem_addr(pv_bar + ((nchunks - 1) & 1)), ((nchunks - 1) >> 1) & 1);
    umma::fence_after_sync();
    launch_dependents();
    // ---- the row's sum over both key halves, then out = O / l
    float* rb = red + (nchunks & 1) * (2 * kRows);
    rb[half * kRows + row] = l;
    named_bar_sync(1 + quarter, 64);
    const float lt = l + rb[(1 - half) * kRows + row];
    const float inv = (row_valid && lt > 0.f) ? 1.0f / lt : 0.f;
    uint16_t* out = static_cast<uint16_t*>(p.out) +
                    (static_cast<size_t>(q0 + t0 + (row_valid ? my_t : 0)) * p.num_q_heads +
                     kvh * G + my_g) *
                        D +
                    half * (D / 2);
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      float o[32];
      umma::ld32(tOh + c * 32, o);
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
  }
  umma::fence_before_sync();
  __syncthreads();
  if (mma_warp) umma::dealloc(tmem, L::kTmemCols);
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

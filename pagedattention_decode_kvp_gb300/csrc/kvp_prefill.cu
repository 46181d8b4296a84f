// kvp_prefill.cu -- multi-query (prefill / chunked-prefill) paged attention on
// the 5th-generation tensor cores.
//
// What is computed ("ATB KV Cache management", "Prefix Caching": requests that
// share a system prompt reuse its cached K/V and only their own part is new):
// request b holds n = context_lens[b] cached tokens whose last L are this
// chunk's queries (their K/V already appended); query i of the chunk sits at
// position n - L + i and attends causally to positions 0 .. n - L + i through
// the block table.  Unlike the decode, this is a dense contraction: a 128-row
// query tile against 128-key tiles.
//
// Design (one CTA of 11 warps per (request, kv head, 128-row query tile)):
//   * Tile rows are (query token, query head of the kv head's group) pairs, so
//     every K/V byte a tile reads serves the whole GQA group.
//   * K/V arrive in 128-key chunks (8 blocks) through separate K and V rings
//     in shared memory: TMA copies (128-byte swizzle, the layout the tensor
//     core reads directly) issued by two producer warps, one per tensor.
//   * One thread issues the tensor-core work: S = Q K^T (tcgen05.mma, M=128,
//     N=128, K=D; Q held in TMEM so only K is read from shared memory) into
//     one of two TMEM score buffers -- S of chunk j+1 is issued before the
//     softmax of chunk j is awaited -- and O += P V (M=128, N=D, K=128) into
//     a TMEM accumulator, so the tensor core works while the CUDA cores
//     exponentiate.
//   * Two threads own each query row (TMEM lane): each takes 64 of every
//     chunk's 128 keys, applies the causal mask and the scale; the two
//     exchange their chunk max once per chunk, keep the row's running max and
//     their partial sums in registers, and share one O accumulator in TMEM
//     (each rescales half of its columns).  The running max is updated
//     lazily: only when it grows by more than 2^8 is O rescaled (exact:
//     numerator and denominator share the stale max).
//   * P stays in tensor memory: each thread writes its 64 probabilities,
//     packed as 16-bit pairs, over the scores it has read (fp16; bf16 as a
//     high part plus a bf16 residual so P keeps ~16 bits), and P V takes its
//     A operand from TMEM -- no shared-memory round trip, no proxy fence.
//   * At the end the two threads of a row add their sums and each writes half
//     of the output row.
#include "kvp_device.cuh"
#include "kvp_internal.h"
#include "kvp_umma.cuh"

namespace kvp {
namespace {

constexpr int kRows = 128;                            // M: query rows per CTA
constexpr int kKeys = 128;                            // key tokens per chunk (8 blocks)
// (64-key chunks were measured slower: an N = 64 score MMA costs nearly as
// much as an N = 128 one, so per key the single issuing thread does more)
constexpr int kSplit = 2;                             // softmax threads per query row
constexpr int kKeysPerThread = kKeys / kSplit;        // keys of each chunk per thread
constexpr int kSoftmaxWarps = 4 * kSplit;             // kSplit per TMEM lane quarter
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kMmaWarp = kSoftmaxWarps;               // issues the tensor-core work
// TMA issue: one warp streams K tiles, one V tiles
constexpr int kProducerWarps = 2;
constexpr int kThreads = kSoftmaxThreads + 32 + kProducerWarps * 32;
constexpr int kSmemPerSm = 233472;                    // shared memory of one SM (bytes)
constexpr int kTableCap = 1024;                       // block ids staged on chip per tile

template <bool kBf16, int D>
struct PrefillLayout {
  static constexpr int kHalves = D / 64;                  // 64-element K-major halves
  static constexpr uint32_t kQ = kRows * D * 2;           // Q tile
  static constexpr uint32_t kKV = kKeys * D * 2;          // one K or V tile
  // Separate K and V rings: a K stage is free once its S is computed, a V
  // stage once its P V is; depths fill the shared memory left by Q.
  static constexpr int kKStages = D == 64 ? 5 : 3;
  static constexpr int kVStages = D == 64 ? 5 : 2;
  // S runs one chunk ahead of the softmax: the MMA thread issues S(j + 1)
  // before it waits for the softmax of chunk j
  static constexpr int kAhead = 1;
  static constexpr int kSBufs = kAhead + 1;               // TMEM score (then P) buffers
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKOff = kQ;
  static constexpr uint32_t kVOff = kKOff + kKStages * kKV;
  static constexpr uint32_t kRedOff = kVOff + kVStages * kKV;  // [4][kSplit][kRows] float
  static constexpr uint32_t kTblOff = kRedOff + 4 * kSplit * kRows * 4;  // [kTableCap] int32
  static constexpr uint32_t kBarOff = kTblOff + kTableCap * 4;
  // kfull[], vfull[], kempty[], vempty[], s[], p[], pv[2], q, q in TMEM
  static constexpr int kBars = 2 * (kKStages + kVStages) + 2 * kSBufs + 4;
  // + 1024 bytes of alignment slack, the barriers and the TMEM address slot
  static constexpr size_t kSmem = 1024 + kBarOff + kBars * 8 + 16;
  // TMEM columns: score buffer i at [128 i, 128 (i+1)) (key half h's P is
  // written over its own scores at [128 i + 64 h, +32), its bf16 residual
  // right after); the Q tile (16-bit pairs) at [256, 256 + D/2), so the score
  // MMAs read only K from shared memory; the O accumulator, shared by a row's
  // two threads, at [512 - D, 512).  The shared memory keeps a second CTA off
  // the SM, so all 512 columns are free.
  static constexpr uint32_t kQCol = kSBufs * kKeys;
  static constexpr uint32_t kOCol = 512 - D;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kQCol + D / 2 <= kOCol, "score buffers and Q overlap O");
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
// 32*(w%4) .. +31 (the TMEM lanes it may access) for keys [64*(w/4), +64) of
// each chunk and O columns [D/2*(w/4), +D/2); warp 8 issues the tensor-core
// instructions; warps 9 and 10 are producers of the K and the V tiles.  The MMA and producer warps run their loops converged (waits and
// address arithmetic warp-uniform) and issue from one elected lane.
// Hand-offs (mbarriers; every wait is at most one phase behind its barrier):
//   kfull[c % kKStages]   producer -> MMA     chunk c's K landed (1 arrival + bytes)
//   vfull[c % kVStages]   producers -> MMA    chunk c's V landed
//   kempty[c % kKStages]  MMA -> producers    S(c) done: K stage free
//   vempty[c % kVStages]  MMA -> producers    P V(c) done: V stage free
//   s[c % kSBufs]         MMA -> softmax      S of chunk c in TMEM buffer c % kSBufs
//   p[c % kSBufs]         softmax -> MMA      P of chunk c written over it (8 arrivals)
//   pv[c % 2]             MMA -> softmax, MMA O += P V of chunk c complete
// Per chunk j the MMA thread -- once P V(j-1) has read its P -- issues
// S(j + kAhead) into chunk j-1's buffer, then waits p(j) and V(j) and issues
// P V(j).  The softmax of chunk j needs only S(j); O is touched (lazy rescale,
// after P V(j-1)) only when a row's max jumps.  The producers start as soon as the
// block table is on chip, while the softmax warps load Q.
template <bool kBf16, int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmq,
                   const __grid_constant__ CUtensorMap tmk,
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
  uint64_t* p_bar = s_bar + kSBufs;                                  // [kSBufs]
  uint64_t* pv_bar = p_bar + kSBufs;                                 // [2]
  uint64_t* q_bar = pv_bar + 2;      // Q tile landed in shared memory
  uint64_t* qt_bar = q_bar + 1;      // Q copied into TMEM (8 arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(qt_bar + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool mma_warp = warp == kMmaWarp;
  const bool producer = warp > kMmaWarp;
  const int quarter = warp & 3;
  const int part = (warp >> 2) & (kSplit - 1);  // which key half / O accumulator
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
  if (q0 < 0 || q0 + qlen > p.num_tokens) {  // rows outside q / out: touch nothing
    if (tid == 0) set_status(p.status, kErrBadBlock);
    return;
  }
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
  if (mma_warp && lane == 0) {
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
    for (int i = 0; i < 2 * (kKStages + kVStages) + kSBufs; ++i)
      mbar_init(smem_addr(kf_bar + i), 1);
    for (int i = 0; i < kSBufs; ++i) mbar_init(smem_addr(p_bar + i), kSoftmaxWarps);
    mbar_init(smem_addr(pv_bar), 1);
    mbar_init(smem_addr(pv_bar + 1), 1);
    mbar_init(smem_addr(q_bar), 1);
    mbar_init(smem_addr(qt_bar), kSoftmaxWarps);
    fence_barrier_init();
    // ---- Q tile by TMA, straight into the K-major swizzled layout: a box of
    // (64 elements, G heads, 128 / G tokens) puts (token t, head g) at row
    // t * G + g.  Tokens past T read as zeros; rows past the tile's own tokens
    // are never used.
    const uint32_t qb = smem_addr(q_bar);
    mbar_arrive_expect_tx(
        qb, static_cast<uint32_t>(L::kHalves * 64 * G * p.q_box_tokens * 2));
#pragma unroll
    for (int hf = 0; hf < L::kHalves; ++hf)
      tma_load_3d(smem_addr(sQ + hf * (kRows * 128)), &tmq, hf * 64, kvh * G, q0 + t0, qb);
  }
  // range-check every block id the tile reads; the first kTableCap are kept on
  // chip so the copy issuers never wait on a global load
  bool bad = false;
  for (int i = tid; i < nblk; i += kThreads) {
    const int id = tbl[i];
    bad |= (id < 0) || (id >= p.num_blocks);
    if (i < kTableCap) stbl[i] = id;
  }
  if (__syncthreads_or(bad)) {
    zero_tile_rows<D>(p, kvh, q0, t0, ntok);
    if (tid == 0) set_status(p.status, kErrBadBlock);
    mbar_wait_bounded(smem_addr(q_bar), 0);  // no copy may land after the exit
    return;
  }

  // ---- producers: warp 9 streams the K tiles, warp 10 the V tiles
  const bool is_k = warp == kMmaWarp + 1;
  const CUtensorMap* map = is_k ? &tmk : &tmv;
  const int nst = is_k ? kKStages : kVStages;
  uint64_t* full = is_k ? kf_bar : vf_bar;
  uint64_t* empty = is_k ? ke_bar : ve_bar;
  const uint32_t ring = smem_addr(sm + (is_k ? L::kKOff : L::kVOff));
  auto produce = [&](int c) {  // the whole warp; one lane issues the copies
    const int st = c % nst;
    bool fine = true;
    if (c >= nst) fine = mbar_wait_bounded(smem_addr(empty + st), ((c / nst) - 1) & 1);
    const int blk0 = c * (kKeys / kBlockSize);
    const int nb = min(kKeys / kBlockSize, nblk - blk0);
    int my_id = 0;
    if (lane < nb) my_id = blk0 + lane < kTableCap ? stbl[blk0 + lane] : tbl[blk0 + lane];
    int ids[kKeys / kBlockSize];
#pragma unroll
    for (int i = 0; i < kKeys / kBlockSize; ++i) ids[i] = __shfl_sync(0xffffffffu, my_id, i);
    if (elect_one()) {
      const uint32_t bar = smem_addr(full + st);
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nb * L::kHalves * 2048));
#pragma unroll
      for (int i = 0; i < kKeys / kBlockSize; ++i) {
        if (i < nb) {
          const int y = (ids[i] * p.num_kv_heads + kvh) * kBlockSize;
#pragma unroll
          for (int hf = 0; hf < L::kHalves; ++hf)
            tma_load_2d(ring + st * L::kKV + i * 2048 + hf * (kKeys * 128), map, hf * 64, y, bar);
        }
      }
    }
    __syncwarp();
    return fine;
  };
  // chunk 0 goes out at once; the rest waits until Q is staged, so the first
  // copies do not queue ahead of the Q loads
  if (producer) produce(0);

  // ---- tile row r = (query token r / G, query head r % G)
  const int my_t = row / G;
  const int my_g = row % G;
  const bool row_valid = warp < kSoftmaxWarps && my_t < ntok;
  if (mma_warp) {
    umma::alloc(smem_addr(tmem_slot), L::kTmemCols);
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (producer) {
    for (int c = 1; c < nchunks; ++c) ok &= produce(c);
  } else if (mma_warp) {
    // the whole warp runs this loop (waits and descriptor arithmetic stay
    // warp-uniform); one elected lane issues each group of tensor instructions
    {
      constexpr uint32_t kIdS = umma::instr_desc_f16(kRows, kKeys, kBf16, false, false);
      constexpr uint32_t kIdO = umma::instr_desc_f16(kRows, D, kBf16, false, true);
      // shared-memory descriptors are built once; an operand at byte offset o
      // from a base is the base descriptor plus o >> 4 (the start-address
      // field, which never carries: every address is below 256 KB)
      const uint64_t k_desc = umma::smem_desc_sw128(smem_addr(sm + L::kKOff), 16, 1024);
      const uint64_t v_desc = umma::smem_desc_sw128(smem_addr(sm + L::kVOff), kKeys * 128, 1024);
      auto issue_s = [&](int c) {  // wait for chunk c's K, S(c) = Q K(c)^T, free the K stage
        ok &= mbar_wait_bounded(smem_addr(kf_bar + c % kKStages), (c / kKStages) & 1);
        umma::fence_after_sync();
        const uint64_t kd = k_desc + (((c % kKStages) * L::kKV) >> 4);
        const uint32_t d = tmem + (c % kSBufs) * kKeys;
        if (elect_one()) {
#pragma unroll
          for (int s = 0; s < D / 16; ++s) {
            const uint32_t koff = (s >> 2) * (kKeys * 128) + (s & 3) * 32;
            umma::mma_f16_tmem_a(d, tmem + L::kQCol + s * 8, kd + (koff >> 4), kIdS,
                                 s > 0 ? 1u : 0u);
          }
          umma::commit(smem_addr(s_bar + c % kSBufs));
          umma::commit(smem_addr(ke_bar + c % kKStages));
        }
        __syncwarp();
      };

      ok &= mbar_wait_bounded(smem_addr(qt_bar), 0);
      umma::fence_after_sync();
      for (int c = 0; c < min(kAhead, nchunks); ++c) issue_s(c);
      for (int j = 0; j < nchunks; ++j) {
        // S(j+kAhead) goes over chunk j-1's P: once P V(j-1) has read it, the
        // tensor core computes it while the softmax works on chunk j
        if (j + kAhead < nchunks) {
          if (j >= 1)
            ok &= mbar_wait_bounded(smem_addr(pv_bar + ((j - 1) & 1)), ((j - 1) >> 1) & 1);
          issue_s(j + kAhead);
        }
        ok &= mbar_wait_bounded(smem_addr(p_bar + j % kSBufs), (j / kSBufs) & 1);
        ok &= mbar_wait_bounded(smem_addr(vf_bar + j % kVStages), (j / kVStages) & 1);
        umma::fence_after_sync();
        const uint32_t pa = tmem + (j % kSBufs) * kKeys;  // P of chunk j (TMEM)
        const uint64_t vd = v_desc + (((j % kVStages) * L::kKV) >> 4);
        if (elect_one()) {
          // key half h (16-key steps t), P read where thread (row, h) wrote it
#pragma unroll
          for (int h = 0; h < kSplit; ++h) {
#pragma unroll
            for (int t = 0; t < kKeysPerThread / 16; ++t) {
              const uint32_t o_acc = tmem + L::kOCol;
              const uint32_t a = pa + h * kKeysPerThread + t * 8;
              const uint64_t b = vd + (((h * kKeysPerThread + t * 16) * 128) >> 4);
              const bool first = j == 0 && h == 0 && t == 0;
              umma::mma_f16_tmem_a(o_acc, a, b, kIdO, first ? 0u : 1u);
              if constexpr (kBf16)
                umma::mma_f16_tmem_a(o_acc, a + kKeysPerThread / 2, b, kIdO, 1u);
            }
          }
          umma::commit(smem_addr(pv_bar + (j & 1)));
          umma::commit(smem_addr(ve_bar + j % kVStages));
        }
        __syncwarp();
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
    float m = -INFINITY, l = 0.f;  // this key half's running max (log2 units) and sum
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    // the O columns this thread rescales and writes: its half of the row
    constexpr int kOCols = D / 2;
    const uint32_t tOp = tmem + L::kOCol + part * (D / 2) + lane_base;
    {
      // Q row `row`, elements [part * D/2, +D/2), from the swizzled tile into
      // TMEM as 16-bit pairs (the A operand of S = Q K^T)
      ok &= mbar_wait_bounded(smem_addr(q_bar), 0);
#pragma unroll
      for (int g = 0; g < D / 64; ++g) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = part * (D / 16) + g * 4 + i;  // 16-byte chunk of the row
          const uint4 v =
              *reinterpret_cast<const uint4*>(sQ + (c >> 3) * (kRows * 128) + sw_chunk(row, c));
          w[4 * i] = v.x;
          w[4 * i + 1] = v.y;
          w[4 * i + 2] = v.z;
          w[4 * i + 3] = v.w;
        }
        umma::st16_bits(tmem + L::kQCol + part * (D / 4) + g * 16 + lane_base, w);
      }
      umma::wait_st();
      umma::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(qt_bar));
    }
    auto o_scale = [&](float alpha) {  // this thread's O columns *= alpha
#pragma unroll
      for (int c = 0; c < kOCols / 32; ++c) {
        float o[32];
        umma::ld32(tOp + c * 32, o);
        umma::wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] *= alpha;
        umma::st32(tOp + c * 32, o);
      }
      umma::wait_st();
    };
    for (int j = 0; j < nchunks; ++j) {
      ok &= mbar_wait_bounded(smem_addr(s_bar + j % kSBufs), (j / kSBufs) & 1);
      umma::fence_after_sync();
      float s[kKeysPerThread];
      const uint32_t tS = tmem + (j % kSBufs) * kKeys + part * kKeysPerThread + lane_base;
#pragma unroll
      for (int c = 0; c < kKeysPerThread / 32; ++c)
        umma::ld32(tS + c * 32, *reinterpret_cast<float(*)[32]>(s + c * 32));
      umma::wait_ld();
      const int kbase = j * kKeys + part * kKeysPerThread;
      if (j * kKeys + kKeys - 1 > pos0) {  // chunk reaches past some row's position
#pragma unroll
        for (int k = 0; k < kKeysPerThread; ++k)
          s[k] = (row_valid && kbase + k <= qpos) ? s[k] : -INFINITY;
      }
      if (!pos_scale) {
#pragma unroll
        for (int k = 0; k < kKeysPerThread; ++k)
          s[k] = s[k] == -INFINITY ? -INFINITY : s[k] * sl2;
      }
      float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]);
      float mx2 = fmaxf(s[4], s[5]), mx3 = fmaxf(s[6], s[7]);
#pragma unroll
      for (int k = 8; k < kKeysPerThread; k += 8) {
        mx0 = fmaxf(mx0, fmaxf(s[k], s[k + 1]));
        mx1 = fmaxf(mx1, fmaxf(s[k + 2], s[k + 3]));
        mx2 = fmaxf(mx2, fmaxf(s[k + 4], s[k + 5]));
        mx3 = fmaxf(mx3, fmaxf(s[k + 6], s[k + 7]));
      }
      float rowmax = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * mul;
      {  // one max per row: the partner thread holds the row's other keys
        float* rb = red + (j & 1) * (kSplit * kRows);
        rb[part * kRows + row] = rowmax;
        named_bar_sync(1 + quarter, 32 * kSplit);
        rowmax = fmaxf(rowmax, rb[(1 - part) * kRows + row]);
      }
      const float mnew = fmaxf(m, rowmax);
      const bool grow = mnew > m + 8.0f;  // lazy: rescale only when the max grows by > 2^8
      const float alpha = grow ? ex2_approx(m - mnew) : 1.0f;
      if (grow) {
        l *= alpha;
        m = mnew;
      }
      // ---- P over this thread's scores in TMEM (it has read them all); a
      // half whose keys are all masked so far (m = -inf) gets P = 0
      const float negm = m == -INFINITY ? 0.f : -m;
      float ps0 = 0.f, ps1 = 0.f, ps2 = 0.f, ps3 = 0.f;
#pragma unroll
      for (int sub = 0; sub < kKeysPerThread / 32; ++sub) {
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
          const float* sk = s + sub * 32 + k;
          const float p0 = ex2_approx(fmaf(sk[0], mul, negm));
          const float p1 = ex2_approx(fmaf(sk[1], mul, negm));
          const float p2 = ex2_approx(fmaf(sk[2], mul, negm));
          const float p3 = ex2_approx(fmaf(sk[3], mul, negm));
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
        umma::st16_bits(tS + sub * 16, hi);
        if constexpr (kBf16) umma::st16_bits(tS + kKeysPerThread / 2 + sub * 16, lo);
      }
      l += (ps0 + ps1) + (ps2 + ps3);
      // ---- O: rescale the rows whose max jumped, once P V(j-1) is in it
      if (__any_sync(0xffffffffu, grow && j > 0)) {
        ok &= mbar_wait_bounded(smem_addr(pv_bar + ((j - 1) & 1)), ((j - 1) >> 1) & 1);
        umma::fence_after_sync();
        o_scale(alpha);
      }
      umma::wait_st();
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
        fence_proxy_async_smem();
      }
      umma::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(p_bar + j % kSBufs));
    }

    ok &= mbar_wait_bounded(smem_addr(pv_bar + ((nchunks - 1) & 1)), ((nchunks - 1) >> 1) & 1);
    umma::fence_after_sync();
    launch_dependents();
    // ---- the row's sum over both key halves (their max is shared), then
    // out = O / l; thread (row, part) writes output columns [part * D/2, +D/2)
    float* rb = red + 2 * kSplit * kRows;
    rb[part * kRows + row] = l;
    named_bar_sync(1 + quarter, 32 * kSplit);
    const float lt = rb[row] + rb[kRows + row];
    const float inv = (row_valid && lt > 0.f) ? 1.0f / lt : 0.f;
    uint16_t* out = static_cast<uint16_t*>(p.out) +
                    (static_cast<size_t>(q0 + t0 + (row_valid ? my_t : 0)) * p.num_q_heads +
                     kvh * G + my_g) *
                        D +
                    part * (D / 2);
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      float o[32];
      umma::ld32(tOp + c * 32, o);
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
cudaError_t launch_prefill_t(const PrefillParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                             const CUtensorMap& tv, int grid_x, cudaStream_t s) {
  constexpr size_t smem = PrefillLayout<kBf16, D>::kSmem;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(&prefill_kernel<kBf16, D>), smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(grid_x, p.num_kv_heads, p.batch);
  return launch_pdl(prefill_kernel<kBf16, D>, grid, dim3(kThreads), smem, s, p, tq, tk, tv);
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, bool bf16, int grid_x, cudaStream_t s) {
  if (!bf16 && p.head_dim == 64) return launch_prefill_t<false, 64>(p, tq, tk, tv, grid_x, s);
  if (!bf16 && p.head_dim == 128) return launch_prefill_t<false, 128>(p, tq, tk, tv, grid_x, s);
  if (bf16 && p.head_dim == 64) return launch_prefill_t<true, 64>(p, tq, tk, tv, grid_x, s);
  if (bf16 && p.head_dim == 128) return launch_prefill_t<true, 128>(p, tq, tk, tv, grid_x, s);
  return cudaErrorInvalidValue;
}

}  // namespace kvp

// kvp_decode_fp8_umma.cu -- paged decode attention over FP8 (E4M3) pools on the
// 5th-generation tensor cores (tcgen05.mma kind::f8f6f4), head_dim 128.
//
// What is computed is the decode of kvp_decode.cuh over FP8 codes with per
// token-and-head fp32 scales ("KV Cache 优化与显存管理", 二: K/V quantised to
// FP8 halve the bytes the decode reads; "ATB PagedAttention", "PagedAttention
// 的 Attention 计算修改": score, online softmax, weighted V).  The warp-level
// consumer widens every code to fp16 before its mma and is bound by those
// conversions; here no code is converted at all -- the tensor core multiplies
// the stored E4M3 bytes:
//   * One CTA per (request, kv head, query group of <= 8 heads, partition)
//     walks its blocks in chunks of 128 tokens (8 blocks).
//   * S^T[128 tokens x 16] = K . Q'^T: the chunk's K tile (as TMA lays it
//     down, K-major, 128-byte swizzle) is the A operand; Q' = q * 2^sigma (a
//     power of two putting the group's |q|max in [128, 256)) is split into
//     three E4M3 terms, each the E4M3 value nearest to what the earlier ones
//     leave (about 12 significant bits in all), and the three products
//     accumulate in one TMEM tile.  Columns past the group's heads are zero.
//   * Softmax: one thread per token (its TMEM lane).  With u the true score
//     (log2 units) and w = log2(v_scale) of the token, P' = 2^(u + w - m)
//     folds the V scale into the weight, m being the CTA's running max of
//     u + w per head (exchanged once per chunk; O is rescaled lazily, only
//     when m grows by more than 2^8, so P' <= 2^8); the row sum takes
//     2^(u - m).  P' is split into three E4M3 terms whose residuals are
//     scaled by 2^4 and 2^8 before rounding, so each stays in E4M3's normal
//     range near the largest weights (P' ~ 1), where the output is most
//     sensitive.
//   * O_t^T[128 d x 16] += V^T . P'_t^T, one TMEM accumulator per term: the
//     chunk's V tile, as stored, is the MN-major A operand (rows along the
//     token index); the P' terms, written by the softmax threads in shared
//     memory, are the B operand.  O = O_1 + O_2 / 2^4 + O_3 / 2^8.
//   * Warp roles: warps 0-3 softmax, warp 4 streams K tiles and both scale
//     rows, warp 5 streams V tiles, warp 6 issues the tensor-core work; all
//     hand-offs are mbarriers with bounded waits.
// The result (or this partition's (m, l, o)) is written like the other
// decode kernels', so the split-context reduce merges it unchanged.
#include "kvp_decode.cuh"
#include "kvp_umma.cuh"

namespace kvp {
namespace {

constexpr int kD = 128;
constexpr int kChunk = 128;                      // tokens per chunk
constexpr int kChunkBlocks = kChunk / kBlockSize;
constexpr int kSoftWarps = 4;
constexpr int kThreadsU = (kSoftWarps + 3) * 32;  // + K producer, V producer, MMA
constexpr int kTerms = 3;                        // E4M3 terms of Q' and P'
constexpr int kN = 16;                           // MMA N: query heads (8) padded
constexpr int kMaxHeads = 8;

// Shared memory (1024-byte aligned base).  K runs a stage deeper than V: it
// is needed first (S, then the softmax), V only by P V.
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr uint32_t kTile = kChunk * kD;                   // one K or V chunk, 16 KB
constexpr uint32_t kKOff = 0;                             // K ring
constexpr uint32_t kVOff = kKOff + kKStages * kTile;      // V ring
constexpr uint32_t kScOff = kVOff + kVStages * kTile;     // per K stage: 128 K, 128 V scales
constexpr uint32_t kQOff = kScOff + kKStages * 1024;      // Q' terms [3][16 rows][128 B]
constexpr uint32_t kPOff = kQOff + kTerms * 2048;   // P' terms [2 buffers][3][16][128 B]
constexpr uint32_t kRedOff = kPOff + 2 * kTerms * 2048;  // [4 warps][8] floats, + [4]
constexpr uint32_t kBarOff = kRedOff + 512;
// kfull[3], vfull[2], sfull[2], pfull[2], pvdone[2], kfree[3], qready, done
constexpr int kNumBars = 2 * kKStages + 4 * 2 + 2;
constexpr uint32_t kSlotOff = kBarOff + kNumBars * 8;
constexpr uint32_t kTblOff = kSlotOff + 16;
static_assert(kQOff % 1024 == 0 && kPOff % 1024 == 0, "operand tiles need 1024-byte alignment");

constexpr size_t umma_smem_for(int part_blocks) {
  return 1024 + kTblOff + static_cast<size_t>(part_blocks) * 4;
}

// TMEM columns: S^T buffers [0, 16) and [16, 32); O_t^T (term t) at
// [32 + 16 t, 48 + 16 t).
constexpr uint32_t kSCol = 0;
constexpr uint32_t kOCol = 2 * kN;
constexpr uint32_t kTmemCols = 128;

// Instruction descriptors (kind::f8f6f4, E4M3 x E4M3 -> f32, M = 128, N = 16):
// S^T with both operands K-major; O^T with A (V^T) MN-major.
constexpr uint32_t kIdS = umma::instr_desc_f16(kChunk, kN, false, false, false);
constexpr uint32_t kIdO = umma::instr_desc_f16(kD, kN, false, true, false);

// byte (row r, column c) of a 128-byte-row tile with the 128-byte swizzle
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t c) {
  return r * 128 + ((((c >> 4) ^ r) & 7u) << 4) + (c & 15u);
}

// 8 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void st8(uint32_t taddr, const float (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem] over E4M3 codes; issued by one thread.
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// log2 on the special-function unit (the lg2.approx PTX instruction).
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Three E4M3 terms of two values (x0, x1), each term the E4M3 value nearest
// to what the earlier ones leave (times 2^kShift per term: x = t_0 +
// t_1 / 2^kShift + t_2 / 2^(2 kShift)); term t of the pair as a 16-bit code
// pair.  (The residuals are exact: a term is the value rounded to 4
// significant bits.)
template <int kShift>
__device__ __forceinline__ void split3(float x0, float x1, uint16_t (&t)[kTerms]) {
  constexpr float kUp = static_cast<float>(1 << kShift);
#pragma unroll
  for (int i = 0; i < kTerms; ++i) {
    t[i] = dev::f32x2_to_e4m3x2(x0, x1);
    if (i + 1 < kTerms) {
      const float2 e = dev::unpack2<false>(dev::e4m3x2_to_f16x2(t[i]));
      x0 = (x0 - e.x) * kUp;
      x1 = (x1 - e.y) * kUp;
    }
  }
}

// Max-reduction of N values held by every lane over the warp (N = 8: lane l
// ends with the max of value index (l >> 2) & 7): each step halves what a lane
// holds while folding in one lane bit.
template <int N, int BIT>
__device__ __forceinline__ void butterfly_max(float* v, int lane) {
  if constexpr (BIT >= 1) {
    if constexpr (N > 1) {
      const bool upper = (lane & BIT) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        const float send = upper ? v[i] : v[i + N / 2];
        const float keep = upper ? v[i + N / 2] : v[i];
        v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, BIT));
      }
      butterfly_max<N / 2, BIT / 2>(v, lane);
    } else {
      v[0] = fmaxf(v[0], __shfl_xor_sync(0xffffffffu, v[0], BIT));
      butterfly_max<1, BIT / 2>(v, lane);
    }
  }
}
template <int N, int BIT>
__device__ __forceinline__ void butterfly_sum(float* v, int lane) {
  if constexpr (BIT >= 1) {
    if constexpr (N > 1) {
      const bool upper = (lane & BIT) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        const float send = upper ? v[i] : v[i + N / 2];
        const float keep = upper ? v[i + N / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, BIT);
      }
      butterfly_sum<N / 2, BIT / 2>(v, lane);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], BIT);
      butterfly_sum<1, BIT / 2>(v, lane);
    }
  }
}

// The 8-bit pool shape for the shared decode prologue.
struct Fp8UmmaShape {
  static constexpr int kD = 128;
  static constexpr int kElemBytes = 1;
};

template <bool kQBf16>
__global__ void __launch_bounds__(kThreadsU, 2)
    decode_fp8_umma_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                           const __grid_constant__ CUtensorMap tmv) {
  using namespace dev;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint64_t* kfull = reinterpret_cast<uint64_t*>(sm + kBarOff);  // [kKStages]
  uint64_t* vfull = kfull + kKStages;                              // [kVStages]
  uint64_t* sfull = vfull + kVStages;                              // [2] S buffers
  uint64_t* pfull = sfull + 2;                                     // [2] P' buffers
  uint64_t* pvdone = pfull + 2;                                    // [2]
  uint64_t* kfree = pvdone + 2;                                    // [kKStages]
  uint64_t* qready = kfree + kKStages;
  uint64_t* done = qready + 1;  // every tensor-core op of the CTA complete
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + kSlotOff);
  float* red = reinterpret_cast<float*>(sm + kRedOff);
  __shared__ int cta_flag;

  DecodeSmem dsm{};
  dsm.tbl = reinterpret_cast<int32_t*>(sm + kTblOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  DecodeCta c;
  bool any_bad = false;
  if (!decode_prologue<Fp8UmmaShape>(p, dsm, c, &any_bad, [&] {
        cta_flag = 0;
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        for (int i = 0; i < kKStages + kVStages + 2; ++i)  // kfull, vfull, sfull
          mbar_init(smem_addr(kfull + i), 1);
        mbar_init(smem_addr(pfull), kSoftWarps);
        mbar_init(smem_addr(pfull + 1), kSoftWarps);
        mbar_init(smem_addr(pvdone), 1);
        mbar_init(smem_addr(pvdone + 1), 1);
        for (int i = 0; i < kKStages; ++i) mbar_init(smem_addr(kfree + i), kSoftWarps);
        mbar_init(smem_addr(qready), kSoftWarps);
        mbar_init(smem_addr(done), 1);
      }))
    return;
  const int32_t* tbl = dsm.tbl;
  const int nchunks = (c.nb + kChunkBlocks - 1) / kChunkBlocks;
  // tokens of chunk k this partition holds (the sequence's last block may be partial)
  auto chunk_tokens = [&](int k) {
    const int nbk = min(kChunkBlocks, c.nb - k * kChunkBlocks);
    return (c.last_part && k == nchunks - 1) ? (nbk - 1) * kBlockSize + c.tail_valid
                                             : nbk * kBlockSize;
  };

  bool ok = !any_bad;
  if (warp == kSoftWarps + 2) umma::alloc(smem_addr(tslot), kTmemCols);
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tslot;

  if (ok && warp == kSoftWarps) {
    // ---- K producer: K tiles and both scale rows of each chunk; a stage is
    // refilled once the softmax of its previous chunk has read its scales
    // (after its S, computed from the K tile, landed)
    for (int k = 0; k < nchunks && ok; ++k) {
      const int st = k % kKStages;
      if (k >= kKStages)
        ok &= mbar_wait_bounded(smem_addr(kfree + st), (k / kKStages - 1) & 1);
      if (elect_one()) {
        const int nbk = min(kChunkBlocks, c.nb - k * kChunkBlocks);
        const uint32_t bar = smem_addr(kfull + st);
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nbk * (2048 + 2 * 64)));
        float* sc = reinterpret_cast<float*>(sm + kScOff + st * 1024);  // (st: K stage)
        for (int i = 0; i < nbk; ++i) {
          const int y = (tbl[k * kChunkBlocks + i] * p.num_kv_heads + c.kvh) * kBlockSize;
          tma_load_2d(smem_addr(sm + kKOff + st * kTile + i * 2048), &tmk, 0, y, bar);
          bulk_load(smem_addr(sc + i * 16), p.k_scale + y, 64, bar);
          bulk_load(smem_addr(sc + 128 + i * 16), p.v_scale + y, 64, bar);
        }
      }
      __syncwarp();
    }
    // no copy may land after the exit: wait (bounded) for the last chunks'
    for (int k = max(0, nchunks - kKStages); k < nchunks; ++k)
      mbar_wait_bounded(smem_addr(kfull + k % kKStages), (k / kKStages) & 1);
  } else if (ok && warp == kSoftWarps + 1) {
    // ---- V producer
    for (int k = 0; k < nchunks && ok; ++k) {
      const int st = k & 1;
      if (k >= 2) ok &= mbar_wait_bounded(smem_addr(pvdone + st), ((k - 2) >> 1) & 1);
      if (elect_one()) {
        const int nbk = min(kChunkBlocks, c.nb - k * kChunkBlocks);
        const uint32_t bar = smem_addr(vfull + st);
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nbk * 2048));
        for (int i = 0; i < nbk; ++i) {
          const int y = (tbl[k * kChunkBlocks + i] * p.num_kv_heads + c.kvh) * kBlockSize;
          tma_load_2d(smem_addr(sm + kVOff + st * kTile + i * 2048), &tmv, 0, y, bar);
        }
      }
      __syncwarp();
    }
    for (int k = max(0, nchunks - 2); k < nchunks; ++k)
      mbar_wait_bounded(smem_addr(vfull + (k & 1)), (k >> 1) & 1);
  } else if (ok && warp == kSoftWarps + 2) {
    // ---- MMA warp: S(0), S(1); then per chunk k: P V(k), S(k + 2)
    const uint64_t q_desc = umma::smem_desc_sw128(smem_addr(sm + kQOff), 16, 1024);
    const uint64_t p_desc = umma::smem_desc_sw128(smem_addr(sm + kPOff), 16, 1024);
    const uint64_t k_desc = umma::smem_desc_sw128(smem_addr(sm + kKOff), 16, 1024);
    const uint64_t v_desc = umma::smem_desc_sw128(smem_addr(sm + kVOff), 4096, 1024);
    ok &= mbar_wait_bounded(smem_addr(qready), 0);
    auto issue_s = [&](int k) {
      const int ks = k % kKStages;  // K stage
      const int sb = k & 1;         // S buffer
      ok &= mbar_wait_bounded(smem_addr(kfull + ks), (k / kKStages) & 1);
      umma::fence_after_sync();
      if (elect_one()) {
        const uint64_t kd = k_desc + ((ks * kTile) >> 4);
#pragma unroll
        for (int t = 0; t < kTerms; ++t)
#pragma unroll
          for (int s = 0; s < kD / 32; ++s)
            mma_f8(tmem + kSCol + sb * kN, kd + ((s * 32) >> 4),
                   q_desc + ((t * 2048 + s * 32) >> 4), kIdS, (t | s) ? 1u : 0u);
        umma::commit(smem_addr(sfull + sb));
      }
      __syncwarp();
    };
    issue_s(0);
    if (nchunks > 1) issue_s(1);
    for (int k = 0; k < nchunks && ok; ++k) {
      const int st = k & 1;
      ok &= mbar_wait_bounded(smem_addr(pfull + st), (k >> 1) & 1);
      ok &= mbar_wait_bounded(smem_addr(vfull + st), (k >> 1) & 1);
      umma::fence_after_sync();
      if (elect_one()) {
        const uint64_t vd = v_desc + ((st * kTile) >> 4);
        const uint64_t pd = p_desc + ((st * kTerms * 2048) >> 4);
#pragma unroll
        for (int t = 0; t < kTerms; ++t)
#pragma unroll
          for (int s = 0; s < kChunk / 32; ++s)
            mma_f8(tmem + kOCol + t * kN, vd + ((s * 32 * 128) >> 4),
                   pd + ((t * 2048 + s * 32) >> 4), kIdO, (k | s) ? 1u : 0u);
        umma::commit(smem_addr(pvdone + st));
      }
      __syncwarp();
      if (k + 2 < nchunks && ok) issue_s(k + 2);
    }
    // every tensor-core op issued here completes before TMEM is released
    if (elect_one()) umma::commit(smem_addr(done));
    __syncwarp();
    mbar_wait_bounded(smem_addr(done), 0);
  }

  // ---- softmax warps: one thread per token of the chunk (its TMEM lane)
  float o[kMaxHeads];
  float mrun[kMaxHeads], lpart[kMaxHeads];
  if (warp < kSoftWarps) {
    const int nh = c.nheads;
    // Q' terms: thread t converts head t / 16, columns 8 (t % 16) .. + 7
    {
      uint4* z = reinterpret_cast<uint4*>(sm + kQOff);
      for (int i = tid; i < (kTerms + 2 * kTerms) * 2048 / 16; i += kSoftWarps * 32)
        z[i] = make_uint4(0u, 0u, 0u, 0u);  // Q' and both P' buffers start zero
      const int h = tid >> 4, d0 = 8 * (tid & 15);
      uint4 raw = make_uint4(0u, 0u, 0u, 0u);
      if (h < nh && ok)
        raw = *reinterpret_cast<const uint4*>(
            static_cast<const uint16_t*>(p.q) +
            (static_cast<size_t>(c.b) * p.num_q_heads + c.head0 + h) * kD + d0);
      const uint32_t wq[4] = {raw.x, raw.y, raw.z, raw.w};
      float x[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = unpack2<kQBf16>(wq[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
      }
      float am = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(x[i]));
      am = warp_max(am);
      if (lane == 0) red[32 + warp] = am;
      named_bar_sync(1, kSoftWarps * 32);
      am = fmaxf(fmaxf(red[32], red[33]), fmaxf(red[34], red[35]));
      // a power of two putting the group's |q|max in [128, 256) (exact)
      int sigma = am > 0.f ? 7 - (static_cast<int>((__float_as_uint(am) >> 23) & 0xffu) - 127) : 0;
      sigma = max(-120, min(120, sigma));
      const float up = __uint_as_float(static_cast<uint32_t>(127 + sigma) << 23);
      const float qunscale = __uint_as_float(static_cast<uint32_t>(127 - sigma) << 23);
      uint16_t tt[4][kTerms];
#pragma unroll
      for (int i = 0; i < 4; ++i) split3<0>(x[2 * i] * up, x[2 * i + 1] * up, tt[i]);
      if (h < nh) {
#pragma unroll
        for (int t = 0; t < kTerms; ++t) {
          const uint2 wv = make_uint2(static_cast<uint32_t>(tt[0][t]) | (static_cast<uint32_t>(tt[1][t]) << 16),
                                      static_cast<uint32_t>(tt[2][t]) | (static_cast<uint32_t>(tt[3][t]) << 16));
          *reinterpret_cast<uint2*>(sm + kQOff + t * 2048 + swz(h, d0)) = wv;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(qready));
#pragma unroll
      for (int h2 = 0; h2 < kMaxHeads; ++h2) {
        mrun[h2] = -INFINITY;
        lpart[h2] = 0.f;
      }
      // the score scale of u (log2 units): softmax scale times 2^-sigma (the K
      // scale multiplies per token)
      const float cs = p.scale_log2 * qunscale;
      const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
      // (the loop ends only at the barrier where the softmax warps agree on
      // ok, so none of them is left waiting at a named barrier; a CTA with a
      // bad block id streams nothing)
      const int nloop = any_bad ? 0 : nchunks;
      for (int k = 0; k < nloop; ++k) {
        const int st = k & 1;
        const int ntk = chunk_tokens(k);
        const bool valid = tid < ntk;
        ok &= mbar_wait_bounded(smem_addr(sfull + st), (k >> 1) & 1);
        umma::fence_after_sync();
        float s[kMaxHeads];
        ld8(tmem + lane_off + kSCol + st * kN, s);
        umma::wait_ld();
        const int kst = k % kKStages;
        const float* sc = reinterpret_cast<const float*>(sm + kScOff + kst * 1024);
        const float ks = valid ? sc[tid] : 0.f;
        const float vs = valid ? sc[128 + tid] : 1.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(kfree + kst));  // K stage kst is read
        const float wv = lg2_approx(vs);
        float u[kMaxHeads], z[kMaxHeads];
#pragma unroll
        for (int h2 = 0; h2 < kMaxHeads; ++h2) {
          u[h2] = (valid && h2 < nh) ? s[h2] * ks * cs : -INFINITY;
          z[h2] = u[h2] + wv;
        }
        // ---- the chunk's max of u + w per head over the CTA's 128 tokens
        float mx[kMaxHeads];
#pragma unroll
        for (int h2 = 0; h2 < kMaxHeads; ++h2) mx[h2] = z[h2];
        butterfly_max<kMaxHeads, 16>(mx, lane);
        if ((lane & 3) == 0) red[warp * 8 + ((lane >> 2) & 7)] = mx[0];
        // the softmax warps agree here whether every wait so far succeeded
        // (a named barrier has no time limit, so all of them stop together)
        ok = named_bar_and(1, kSoftWarps * 32, ok);
        if (!ok) break;
        bool rescale = false;
        float mnew[kMaxHeads];
#pragma unroll
        for (int h2 = 0; h2 < kMaxHeads; ++h2) {
          const float cm = fmaxf(fmaxf(red[h2], red[8 + h2]), fmaxf(red[16 + h2], red[24 + h2]));
          mnew[h2] = fmaxf(mrun[h2], cm);
          rescale |= mnew[h2] > mrun[h2] + 8.0f;
        }
        named_bar_sync(1, kSoftWarps * 32);  // red is rewritten next chunk
        if (rescale) {  // CTA-uniform: every thread sees the same maxima
          float al[kMaxHeads];
#pragma unroll
          for (int h2 = 0; h2 < kMaxHeads; ++h2) {
            const bool g = mnew[h2] > mrun[h2] + 8.0f;
            al[h2] = g ? ex2_approx(mrun[h2] - mnew[h2]) : 1.0f;
            lpart[h2] *= al[h2];
            mrun[h2] = g ? mnew[h2] : mrun[h2];
          }
          if (k > 0) {  // O holds chunks 0 .. k-1: wait for the last P V, then scale
            ok &= mbar_wait_bounded(smem_addr(pvdone + ((k - 1) & 1)), ((k - 1) >> 1) & 1);
            umma::fence_after_sync();
#pragma unroll
            for (int t = 0; t < kTerms; ++t) {
              float ov[8];
              ld8(tmem + lane_off + kOCol + t * kN, ov);
              umma::wait_ld();
#pragma unroll
              for (int h2 = 0; h2 < kMaxHeads; ++h2) ov[h2] *= al[h2];
              st8(tmem + lane_off + kOCol + t * kN, ov);
            }
            umma::wait_st();
          }
        }
        // ---- P' = 2^(u + w - m) (<= 2^8) as three E4M3 terms; l += 2^(u - m)
        float pw[kMaxHeads];
#pragma unroll
        for (int h2 = 0; h2 < kMaxHeads; ++h2) {
          const float nm = mrun[h2] == -INFINITY ? 0.f : -mrun[h2];
          pw[h2] = ex2_approx(z[h2] + nm);
          lpart[h2] += ex2_approx(u[h2] + nm);
        }
        uint16_t pt[kMaxHeads / 2][kTerms];
#pragma unroll
        for (int i = 0; i < kMaxHeads / 2; ++i) split3<4>(pw[2 * i], pw[2 * i + 1], pt[i]);
        // the P' buffer of chunk k - 2 has been read by its P V
        if (k >= 2) ok &= mbar_wait_bounded(smem_addr(pvdone + st), ((k - 2) >> 1) & 1);
        uint8_t* pb = sm + kPOff + st * kTerms * 2048;
#pragma unroll
        for (int t = 0; t < kTerms; ++t)
#pragma unroll
          for (int h2 = 0; h2 < kMaxHeads; ++h2)
            if (h2 < nh)
              pb[t * 2048 + swz(h2, tid)] =
                  static_cast<uint8_t>(pt[h2 >> 1][t] >> ((h2 & 1) * 8));
        if (!valid) {
          // a token past the chunk's context: its V row may hold NaN codes
          // (0 * NaN = NaN in the product); clear it once it has landed
          ok &= mbar_wait_bounded(smem_addr(vfull + st), (k >> 1) & 1);
          uint4* vr = reinterpret_cast<uint4*>(sm + kVOff + st * kTile + tid * 128);
#pragma unroll
          for (int i = 0; i < 8; ++i) vr[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        umma::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(pfull + st));
      }
      // ---- O^T row tid (d = tid) and the row sums over the CTA
      if (ok && nchunks > 0)
        ok &= mbar_wait_bounded(smem_addr(pvdone + ((nchunks - 1) & 1)), ((nchunks - 1) >> 1) & 1);
      umma::fence_after_sync();
      {
        float o1[8], o2[8], o3[8];
        ld8(tmem + lane_off + kOCol, o1);
        ld8(tmem + lane_off + kOCol + kN, o2);
        ld8(tmem + lane_off + kOCol + 2 * kN, o3);
        umma::wait_ld();
#pragma unroll
        for (int h2 = 0; h2 < kMaxHeads; ++h2)
          o[h2] = o1[h2] + o2[h2] * (1.0f / 16.0f) + o3[h2] * (1.0f / 256.0f);
      }
      butterfly_sum<kMaxHeads, 16>(lpart, lane);
      named_bar_sync(1, kSoftWarps * 32);
      if ((lane & 3) == 0) red[warp * 8 + ((lane >> 2) & 7)] = lpart[0];
      named_bar_sync(1, kSoftWarps * 32);
#pragma unroll
      for (int h2 = 0; h2 < kMaxHeads; ++h2)
        lpart[h2] = red[h2] + red[8 + h2] + red[16 + h2] + red[24 + h2];
      if (!ok) atomicExch(&cta_flag, 1);
    }
  }

  // ---- teardown: every tensor-core op done (the softmax warps waited for the
  // last P V, or gave up), then the output
  umma::fence_before_sync();
  __syncthreads();
  launch_dependents();
  if (warp == kSoftWarps + 2) umma::dealloc(tmem, kTmemCols);
  const bool bad = any_bad || cta_flag != 0;
  if (threadIdx.x == 0) {
    if (any_bad) set_status(p.status, kErrBadBlock);
    else if (cta_flag != 0) set_status(p.status, kErrTimeout);
  }
  if (warp >= kSoftWarps) return;
  const size_t rowbase = static_cast<size_t>(c.b) * p.num_q_heads + c.head0;
  for (int h2 = 0; h2 < c.nheads && h2 < kMaxHeads; ++h2) {
    if (c.nparts == 1) {
      const float res = (!bad && lpart[h2] > 0.f) ? o[h2] / lpart[h2] : 0.f;
      uint16_t* out = static_cast<uint16_t*>(p.out) + (rowbase + h2) * kD;
      out[tid] = p.q_bf16 ? from_float<true>(res) : from_float<false>(res);
    } else {
      const size_t prow = (rowbase + h2) * p.max_parts + c.part;
      p.ws_o[prow * kD + tid] = bad ? 0.f : o[h2];
      if (tid == 0) {
        p.ws_ml[2 * prow] = bad ? -INFINITY : mrun[h2];
        p.ws_ml[2 * prow + 1] = bad ? -1.f : lpart[h2];  // L < 0: a failed partition
      }
    }
  }
}

}  // namespace

cudaError_t launch_decode_fp8_umma(const DecodeParams& p, const CUtensorMap& tk,
                                   const CUtensorMap& tv, int grid_x, cudaStream_t s) {
  const size_t smem = umma_smem_for(p.part_blocks);
  const dim3 grid(grid_x, p.num_kv_heads * p.qgroups, p.batch);
  if (p.head_dim != kD || p.heads_per_cta > kMaxHeads) return cudaErrorInvalidValue;
  if (p.q_bf16) {
    const cudaError_t e = ensure_smem_attr(
        reinterpret_cast<const void*>(&decode_fp8_umma_kernel<true>), umma_smem_for(kMaxPartBlocks));
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_fp8_umma_kernel<true>, grid, dim3(kThreadsU), smem, s, p, tk, tv);
  }
  const cudaError_t e = ensure_smem_attr(
      reinterpret_cast<const void*>(&decode_fp8_umma_kernel<false>), umma_smem_for(kMaxPartBlocks));
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_fp8_umma_kernel<false>, grid, dim3(kThreadsU), smem, s, p, tk, tv);
}

}  // namespace kvp

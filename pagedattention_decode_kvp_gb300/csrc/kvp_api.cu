// kvp_api.cu -- the extern "C" entry points declared in include/kvp.h:
// argument validation, TMA descriptor encoding, split-context sizing and
// kernel dispatch.  Nothing here allocates device memory.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "kvp_internal.h"

using namespace kvp;

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// KVP_OK, or why the cache description is not usable.
kvp_status check_desc(const kvp_cache_desc& c) {
  if (c.num_blocks <= 0 || c.num_kv_heads <= 0 || c.block_size <= 0 || c.head_dim <= 0)
    return KVP_ERR_INVALID_ARG;
  if (c.block_size != kBlockSize) return KVP_ERR_UNSUPPORTED;
  if (c.head_dim != 64 && c.head_dim != 128) return KVP_ERR_UNSUPPORTED;
  // TMA row coordinates are 32-bit signed
  if (static_cast<long long>(c.num_blocks) * c.num_kv_heads * kBlockSize >= (1ll << 31))
    return KVP_ERR_UNSUPPORTED;
  return KVP_OK;
}

kvp_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KVP_OK : KVP_ERR_CUDA; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
  });
  return fn;
}

// TMA descriptor over a whole pool viewed as [NB * Hkv * 16 rows][D elements]:
// a box is 16 token rows by at most 128 bytes, written to shared memory with
// the 128-byte swizzle (a 256-byte row takes two boxes); 64-byte rows (INT8,
// D = 64) are copied unswizzled.
kvp_status make_pool_map(CUtensorMap* map, const void* base, const kvp_cache_desc& c,
                         int elem_bytes) {
  auto fn = encode_fn();
  if (fn == nullptr) return KVP_ERR_CUDA;
  const int row_bytes = c.head_dim * elem_bytes;
  const int box_bytes = row_bytes < 128 ? row_bytes : 128;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(c.head_dim),
                        static_cast<cuuint64_t>(c.num_blocks) * c.num_kv_heads * kBlockSize};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_bytes / elem_bytes),
                       static_cast<cuuint32_t>(kBlockSize)};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      fn(map, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? KVP_OK : KVP_ERR_CUDA;
}

// TMA descriptor over a whole pool viewed as 5-D {row piece, 16 rows, pieces
// per row, Hkv, NB} (a row piece is <= 128 bytes of a token row), whose box
// {piece, 16, pieces, 1, run} lands `run` consecutive blocks' tiles of one kv
// head in shared memory back to back, each laid out as a per-block box would
// put it ([piece][16 rows][bytes], 128-byte swizzle for 128-byte pieces).
kvp_status make_pool_run_map(CUtensorMap* map, const void* base, const kvp_cache_desc& c,
                             int elem_bytes, int run) {
  auto fn = encode_fn();
  if (fn == nullptr) return KVP_ERR_CUDA;
  const int row_bytes = c.head_dim * elem_bytes;
  const int piece_bytes = row_bytes < 128 ? row_bytes : 128;
  const int pieces = row_bytes / piece_bytes;
  cuuint64_t dims[5] = {static_cast<cuuint64_t>(piece_bytes / elem_bytes),
                        static_cast<cuuint64_t>(kBlockSize), static_cast<cuuint64_t>(pieces),
                        static_cast<cuuint64_t>(c.num_kv_heads),
                        static_cast<cuuint64_t>(c.num_blocks)};
  cuuint64_t strides[4] = {static_cast<cuuint64_t>(row_bytes),
                           static_cast<cuuint64_t>(piece_bytes),
                           static_cast<cuuint64_t>(row_bytes) * kBlockSize,
                           static_cast<cuuint64_t>(row_bytes) * kBlockSize * c.num_kv_heads};
  cuuint32_t box[5] = {static_cast<cuuint32_t>(piece_bytes / elem_bytes),
                       static_cast<cuuint32_t>(kBlockSize), static_cast<cuuint32_t>(pieces), 1,
                       static_cast<cuuint32_t>(run)};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r =
      fn(map, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 5,
         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         piece_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? KVP_OK : KVP_ERR_CUDA;
}

// TMA descriptor over q viewed as [T tokens][Hq heads][D]: a box of 64
// elements x `group` heads x `box_tokens` tokens lands in shared memory as
// 128-byte swizzled rows ordered (token, head) -- the K-major operand layout.
kvp_status make_q_map(CUtensorMap* map, const void* q, int num_tokens, int num_q_heads,
                      int head_dim, int group, int box_tokens) {
  auto fn = encode_fn();
  if (fn == nullptr) return KVP_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(num_q_heads),
                        static_cast<cuuint64_t>(num_tokens)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                           static_cast<cuuint64_t>(num_q_heads) * head_dim * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(box_tokens)};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(q), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? KVP_OK : KVP_ERR_CUDA;
}

struct DecodeShape {
  DecodePath path;
  int heads_per_cta;
  int qgroups;
  int part_blocks;
  int max_parts;
  size_t ws_bytes;
};

// Split-context rule.  Each (request, kv head, query group) unit is cut into
// `parts` partitions of ceil(MB / parts) blocks, run as independent CTAs on
// GB300's 152 SMs (3 resident decode CTAs per SM for 16-bit tiles, 4 for INT8
// tiles, from their shared-memory and register use).  The count of parts
// minimises a simple makespan model: waves * (blocks per CTA + a fixed
// per-CTA cost of about 4 blocks of streaming), plus a small cost for the
// reduce pass when parts > 1.  Partitions stay >= 16 blocks (256 tokens) and
// <= kMaxPartBlocks (the table slice staged on chip).  The model sees only the
// table width MB, not the actual lengths, so it is exact for uniform contexts
// and conservative for ragged ones.
constexpr int kSms = 152;
constexpr double kCtaOverheadBlocks = 4.0;
constexpr double kReduceCostBlocks = 2.0;

int resident_ctas(DecodePath path) {
  switch (path) {
    case DecodePath::kMmaInt8: return 4;
    case DecodePath::kUmmaFp8: return 2;
    default: return 3;
  }
}

int auto_partition(DecodePath path, long long units, int max_blocks) {
  const long long slots = static_cast<long long>(kSms) * resident_ctas(path);
  int best_pb = max_blocks <= kMaxPartBlocks ? max_blocks : kMaxPartBlocks;
  double best = 1e300;
  for (int parts = 1; parts <= max_blocks; ++parts) {
    const int pb = (max_blocks + parts - 1) / parts;
    if (parts > 1 && pb < 16) break;
    if (pb > kMaxPartBlocks) continue;
    if ((max_blocks + pb - 1) / pb != parts) continue;  // same split as a smaller count
    const long long ctas = units * parts;
    const long long waves = (ctas + slots - 1) / slots;
    const double cost = static_cast<double>(waves) * (pb + kCtaOverheadBlocks) +
                        (parts > 1 ? kReduceCostBlocks : 0.0);
    if (cost < best * 0.999) {
      best = cost;
      best_pb = pb;
    }
  }
  return best_pb;
}

// kv_8bit: 0 for 16-bit pools, 1 for INT8 codes, 2 for FP8 (E4M3) codes.
kvp_status shape_decode(int batch, int num_q_heads, const kvp_cache_desc& c, int max_blocks,
                        int partition_blocks, int kv_8bit, DecodeShape* out) {
  if (batch < 0 || num_q_heads <= 0 || max_blocks <= 0) return KVP_ERR_INVALID_ARG;
  const kvp_status ds = check_desc(c);
  if (ds != KVP_OK) return ds;
  if (num_q_heads % c.num_kv_heads != 0) return KVP_ERR_INVALID_ARG;
  if (partition_blocks < 0 || partition_blocks > kMaxPartBlocks) return KVP_ERR_INVALID_ARG;
  const int G = num_q_heads / c.num_kv_heads;
  DecodeShape s;
  if (kv_8bit == 2 && c.head_dim == 128) {
    s.path = DecodePath::kUmmaFp8;  // FP8 codes straight into the tensor core
    s.heads_per_cta = G < kHeadsPerCta ? G : kHeadsPerCta;
  } else if (kv_8bit) {
    s.path = DecodePath::kMmaInt8;  // INT8, and FP8 at head_dim 64 (8-bit tiles)
    s.heads_per_cta = G < kHeadsPerCta ? G : kHeadsPerCta;
  } else if (G <= 2) {
    s.path = DecodePath::kSimt;
    s.heads_per_cta = G;
  } else {
    s.path = DecodePath::kMma;
    s.heads_per_cta = G < kHeadsPerCta ? G : kHeadsPerCta;
  }
  s.qgroups = (G + s.heads_per_cta - 1) / s.heads_per_cta;
  const long long units = static_cast<long long>(batch) * c.num_kv_heads * s.qgroups;
  int pb = partition_blocks > 0 ? partition_blocks : auto_partition(s.path, units, max_blocks);
  if (pb >= max_blocks) pb = max_blocks;
  if (pb > kMaxPartBlocks) return KVP_ERR_UNSUPPORTED;  // one partition must fit on chip
  s.part_blocks = pb;
  s.max_parts = (max_blocks + pb - 1) / pb;
  s.ws_bytes = s.max_parts > 1 ? static_cast<size_t>(batch) * num_q_heads * s.max_parts *
                                     (static_cast<size_t>(c.head_dim) + 2) * sizeof(float)
                               : 0;
  *out = s;
  return KVP_OK;
}

kvp_status decode_common(void* out, const void* q, bool q_bf16, int kv_kind, const void* kc,
                         const void* vc, const float* ks, const float* vs, const int32_t* tables,
                         int32_t max_blocks, const int32_t* lens, int32_t batch, int32_t hq,
                         float scale, kvp_cache_desc c, int32_t partition_blocks, void* ws,
                         size_t ws_bytes, int32_t phases, int32_t* status, kvp_stream_t stream,
                         const void* new_k = nullptr, const void* new_v = nullptr) {
  const bool int8 = kv_kind >= 2;  // 8-bit codes with scales: INT8 (2) or FP8 E4M3 (3)
  DecodeShape sh;
  const kvp_status st =
      shape_decode(batch, hq, c, max_blocks, partition_blocks, int8 ? kv_kind - 1 : 0, &sh);
  if (st != KVP_OK) return st;
  const bool merge_runs = (phases & KVP_DECODE_MERGE_RUNS) != 0;
  phases &= ~KVP_DECODE_MERGE_RUNS;
  if (phases < 1 || phases > 3) return KVP_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return KVP_ERR_INVALID_ARG;
  if (batch == 0) return KVP_OK;
  if (!out || !q || !kc || !vc || !tables || !lens) return KVP_ERR_INVALID_ARG;
  if (int8 && (!ks || !vs)) return KVP_ERR_INVALID_ARG;
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(kc, 16) || !aligned(vc, 16))
    return KVP_ERR_INVALID_ARG;
  if (int8 && (!aligned(ks, 16) || !aligned(vs, 16))) return KVP_ERR_INVALID_ARG;
  if (sh.ws_bytes > 0 && (ws == nullptr || ws_bytes < sh.ws_bytes || !aligned(ws, 16)))
    return KVP_ERR_INVALID_ARG;

  DecodeParams p{};
  p.out = out;
  p.q = q;
  p.k_scale = ks;
  p.v_scale = vs;
  p.block_tables = tables;
  p.context_lens = lens;
  p.ws_o = static_cast<float*>(ws);
  p.ws_ml = sh.ws_bytes ? static_cast<float*>(ws) + static_cast<size_t>(batch) * hq *
                                                        sh.max_parts * c.head_dim
                        : nullptr;
  p.status = status;
  p.batch = batch;
  p.num_q_heads = hq;
  p.num_kv_heads = c.num_kv_heads;
  p.head_dim = c.head_dim;
  p.num_blocks = c.num_blocks;
  p.max_blocks = max_blocks;
  p.group = hq / c.num_kv_heads;
  p.qgroups = sh.qgroups;
  p.heads_per_cta = sh.heads_per_cta;
  p.part_blocks = sh.part_blocks;
  p.max_parts = sh.max_parts;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.q_bf16 = q_bf16 ? 1 : 0;
  p.new_k = new_k;
  p.new_v = new_v;
  p.k_pool = kc;
  p.v_pool = vc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  if (static_cast<long long>(c.num_kv_heads) * sh.qgroups > 65535 || batch > 65535)
    return KVP_ERR_UNSUPPORTED;

  if (phases & KVP_PHASE_PARTIAL) {
    const int eb = int8 ? 1 : 2;
    DecodeMaps maps;
    maps.merged = merge_runs && sh.path != DecodePath::kUmmaFp8;  // (per-block fetch only)
    kvp_status r = KVP_OK;
    if (maps.merged) {
      const int runs[3] = {1, 2, 4};
      for (int i = 0; i < 3 && r == KVP_OK; ++i) {
        r = make_pool_run_map(&maps.runs.k[i], kc, c, eb, runs[i]);
        if (r == KVP_OK) r = make_pool_run_map(&maps.runs.v[i], vc, c, eb, runs[i]);
      }
    } else {
      r = make_pool_map(&maps.k, kc, c, eb);
      if (r == KVP_OK) r = make_pool_map(&maps.v, vc, c, eb);
    }
    if (r != KVP_OK) return r;
    cudaError_t e;
    switch (sh.path) {
      case DecodePath::kSimt:
        e = launch_decode_simt(p, maps, kv_kind == 1, sh.max_parts, s);
        break;
      case DecodePath::kMma:
        e = launch_decode_mma(p, maps, kv_kind == 1, sh.max_parts, s);
        break;
      case DecodePath::kUmmaFp8:
        e = launch_decode_fp8_umma(p, maps.k, maps.v, sh.max_parts, s);
        break;
      default:
        e = kv_kind == 3 ? launch_decode_mma_fp8(p, maps, sh.max_parts, s)
                         : launch_decode_mma_int8(p, maps, sh.max_parts, s);
        break;
    }
    if (e != cudaSuccess) return KVP_ERR_CUDA;
  }
  if ((phases & KVP_PHASE_REDUCE) && sh.max_parts > 1) {
    if (launch_decode_reduce(p, s) != cudaSuccess) return KVP_ERR_CUDA;
  }
  return KVP_OK;
}

// A decode whose requests share their first `shared` table entries: the
// prefix's full 128-token chunks (skip = 8 * floor(shared / 8) blocks) are one
// dense pass per kv head over every request's query (tensor cores), written
// as partition 0 of the workspace; the rest of each context is the ordinary
// split decode over blocks skip .. n - 1, written as partitions 1 ...; the
// reduce merges them.  skip == 0 (a prefix shorter than one chunk) or a group
// that does not divide the 128-row tile: the ordinary decode.
struct PrefixShape {
  int skip;          // blocks covered by the prefix pass (0: ordinary decode)
  DecodeShape suf;   // the split decode over the suffix (max_parts: its partitions)
  int max_parts;     // workspace partitions per row: 1 + suf.max_parts
  size_t ws_bytes;
};

kvp_status shape_prefix_decode(int batch, int hq, const kvp_cache_desc& c, int max_blocks,
                               int shared, int partition_blocks, PrefixShape* out) {
  if (shared < 0 || shared > max_blocks) return KVP_ERR_INVALID_ARG;
  const kvp_status ds = check_desc(c);
  if (ds != KVP_OK) return ds;
  if (hq <= 0 || hq % c.num_kv_heads != 0) return KVP_ERR_INVALID_ARG;
  const int group = hq / c.num_kv_heads;
  PrefixShape s{};
  s.skip = (128 % group == 0) ? shared / 8 * 8 : 0;
  if (s.skip == max_blocks) s.skip -= 8;  // keep a suffix width of at least one block
  if (s.skip <= 0) {
    s.skip = 0;
    const kvp_status r = shape_decode(batch, hq, c, max_blocks, partition_blocks, 0, &s.suf);
    if (r != KVP_OK) return r;
    s.max_parts = s.suf.max_parts;
    s.ws_bytes = s.suf.ws_bytes;
  } else {
    const kvp_status r =
        shape_decode(batch, hq, c, max_blocks - s.skip, partition_blocks, 0, &s.suf);
    if (r != KVP_OK) return r;
    s.max_parts = 1 + s.suf.max_parts;
    s.ws_bytes = static_cast<size_t>(batch) * hq * s.max_parts *
                 (static_cast<size_t>(c.head_dim) + 2) * sizeof(float);
  }
  *out = s;
  return KVP_OK;
}

}  // namespace

extern "C" {

const char* kvp_status_string(kvp_status status) {
  switch (status) {
    case KVP_OK: return "KVP_OK";
    case KVP_ERR_INVALID_ARG: return "KVP_ERR_INVALID_ARG";
    case KVP_ERR_UNSUPPORTED: return "KVP_ERR_UNSUPPORTED";
    case KVP_ERR_CUDA: return "KVP_ERR_CUDA";
    case KVP_ERR_BAD_BLOCK: return "KVP_ERR_BAD_BLOCK";
    case KVP_ERR_TIMEOUT: return "KVP_ERR_TIMEOUT";
    case KVP_ERR_OOM: return "KVP_ERR_OOM";
    case KVP_ERR_REFCOUNT: return "KVP_ERR_REFCOUNT";
    case KVP_ERR_NOT_FOUND: return "KVP_ERR_NOT_FOUND";
    case KVP_ERR_SCRATCH_LIMIT: return "KVP_ERR_SCRATCH_LIMIT";
  }
  return "KVP_ERR_UNKNOWN";
}

int32_t kvp_version(void) { return 100; }  // 0.1.0

kvp_status kvp_append(const void* key, const void* value, void* k_cache, void* v_cache,
                      const int32_t* slot_mapping, int32_t num_tokens, kvp_cache_desc cache,
                      kvp_dtype dtype, int32_t* dev_status, kvp_stream_t stream) {
  KVP_NVTX_RANGE("kvp_append");
  const kvp_status ds = check_desc(cache);
  if (ds != KVP_OK) return ds;
  if (num_tokens < 0 || (dtype != KVP_F16 && dtype != KVP_BF16)) return KVP_ERR_INVALID_ARG;
  if (num_tokens == 0) return KVP_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return KVP_ERR_INVALID_ARG;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return KVP_ERR_INVALID_ARG;
  return from_cuda(launch_append(key, value, k_cache, v_cache, slot_mapping, num_tokens, cache, 2,
                                 dev_status, reinterpret_cast<cudaStream_t>(stream)));
}

kvp_status kvp_append_int8(const void* key, const void* value, kvp_dtype src_dtype,
                           int8_t* k_cache, int8_t* v_cache, float* k_scale, float* v_scale,
                           const int32_t* slot_mapping, int32_t num_tokens, kvp_cache_desc cache,
                           int32_t* dev_status, kvp_stream_t stream) {
  KVP_NVTX_RANGE("kvp_append_int8");
  const kvp_status ds = check_desc(cache);
  if (ds != KVP_OK) return ds;
  if (num_tokens < 0 || (src_dtype != KVP_F16 && src_dtype != KVP_BF16))
    return KVP_ERR_INVALID_ARG;
  if (num_tokens == 0) return KVP_OK;
  if (!key || !value || !k_cache || !v_cache || !k_scale || !v_scale || !slot_mapping)
    return KVP_ERR_INVALID_ARG;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 8) || !aligned(v_cache, 8) ||
      !aligned(k_scale, 4) || !aligned(v_scale, 4))
    return KVP_ERR_INVALID_ARG;
  return from_cuda(launch_append_int8(key, value, src_dtype == KVP_BF16, k_cache, v_cache, k_scale,
                                      v_scale, slot_mapping, num_tokens, cache, dev_status,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

kvp_status kvp_append_int8_fixed(const void* key, const void* value, kvp_dtype src_dtype,
                                 int8_t* k_cache, int8_t* v_cache, float* k_scale_pool,
                                 float* v_scale_pool, float k_scale, float v_scale,
                                 const int32_t* slot_mapping, int32_t num_tokens,
                                 kvp_cache_desc cache, int32_t* dev_status, kvp_stream_t stream) {
  KVP_NVTX_RANGE("kvp_append_int8_fixed");
  const kvp_status ds = check_desc(cache);
  if (ds != KVP_OK) return ds;
  if (num_tokens < 0 || (src_dtype != KVP_F16 && src_dtype != KVP_BF16))
    return KVP_ERR_INVALID_ARG;
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return KVP_ERR_INVALID_ARG;
  if (num_tokens == 0) return KVP_OK;
  if (!key || !value || !k_cache || !v_cache || !k_scale_pool || !v_scale_pool || !slot_mapping)
    return KVP_ERR_INVALID_ARG;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 8) || !aligned(v_cache, 8) ||
      !aligned(k_scale_pool, 4) || !aligned(v_scale_pool, 4))
    return KVP_ERR_INVALID_ARG;
  return from_cuda(launch_append_int8_fixed(key, value, src_dtype == KVP_BF16, k_cache, v_cache,
                                            k_scale_pool, v_scale_pool, k_scale, v_scale,
                                            slot_mapping, num_tokens, cache, dev_status,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

kvp_status kvp_append_fp8(const void* key, const void* value, kvp_dtype src_dtype,
                          uint8_t* k_cache, uint8_t* v_cache, float* k_scale, float* v_scale,
                          const int32_t* slot_mapping, int32_t num_tokens, kvp_cache_desc cache,
                          int32_t* dev_status, kvp_stream_t stream) {
  KVP_NVTX_RANGE("kvp_append_fp8");
  const kvp_status ds = check_desc(cache);
  if (ds != KVP_OK) return ds;
  if (num_tokens < 0 || (src_dtype != KVP_F16 && src_dtype != KVP_BF16))
    return KVP_ERR_INVALID_ARG;
  if (num_tokens == 0) return KVP_OK;
  if (!key || !value || !k_cache || !v_cache || !k_scale || !v_scale || !slot_mapping)
    return KVP_ERR_INVALID_ARG;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 8) || !aligned(v_cache, 8) ||
      !aligned(k_scale, 4) || !aligned(v_scale, 4))
    return KVP_ERR_INVALID_ARG;
  return from_cuda(launch_append_fp8(key, value, src_dtype == KVP_BF16, k_cache, v_cache, k_scale,
                                     v_scale, slot_mapping, num_tokens, cache, dev_status,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

kvp_status kvp_copy_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                           int32_t cache_elem_bytes, const int32_t* pairs, int32_t num_pairs,
                           kvp_cache_desc cache, int32_t* dev_status, kvp_stream_t stream) {
  KVP_NVTX_RANGE("kvp_copy_blocks");
  const kvp_status ds = check_desc(cache);
  if (ds != KVP_OK) return ds;
  if (num_pairs < 0 || (cache_elem_bytes != 1 && cache_elem_bytes != 2))
    return KVP_ERR_INVALID_ARG;
  if ((k_scale == nullptr) != (v_scale == nullptr)) return KVP_ERR_INVALID_ARG;
  if (num_pairs == 0) return KVP_OK;
  if (!k_cache || !v_cache || !pairs) return KVP_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return KVP_ERR_INVALID_ARG;
  if (k_scale && (!aligned(k_scale, 16) || !aligned(v_scale, 16))) return KVP_ERR_INVALID_ARG;
  return from_cuda(launch_copy_blocks(k_cache, v_cache, k_scale, v_scale, cache_elem_bytes, pairs,
                                      num_pairs, cache, dev_status,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

int32_t kvp_decode_partition_blocks(int32_t batch, int32_t num_q_heads, kvp_cache_desc cache,
                                    int32_t max_blocks_per_seq, int32_t kv_int8) {
  DecodeShape sh;
  if (kv_int8 < 0 || kv_int8 > 2 ||
      shape_decode(batch, num_q_heads, cache, max_blocks_per_seq, 0, kv_int8, &sh) != KVP_OK)
    return 0;
  return sh.part_blocks;
}

size_t kvp_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, kvp_cache_desc cache,
                                  int32_t max_blocks_per_seq, int32_t partition_blocks,
                                  int32_t kv_int8) {
  DecodeShape sh;
  if (kv_int8 < 0 || kv_int8 > 2 ||
      shape_decode(batch, num_q_heads, cache, max_blocks_per_seq, partition_blocks, kv_int8,
                   &sh) != KVP_OK)
    return 0;
  return sh.ws_bytes;
}

kvp_status kvp_attention_decode(void* out, const void* q, const void* k_cache,
                                const void* v_cache, const int32_t* block_tables,
                                int32_t max_blocks_per_seq, const int32_t* context_lens,
                                int32_t batch, int32_t num_q_heads, float scale,
                                kvp_cache_desc cache, kvp_dtype dtype, int32_t partition_blocks,
                                void* workspace, size_t workspace_bytes, int32_t phases,
                                int32_t* dev_status, kvp_stream_t stream) {
  KVP_NVTX_RANGE("kvp_attention_decode");
  if (dtype != KVP_F16 && dtype != KVP_BF16) return KVP_ERR_INVALID_ARG;
  return decode_common(out, q, dtype == KVP_BF16, dtype == KVP_BF16 ? 1 : 0, k_cache, v_cache,
                       nullptr, nullptr, block_tables, max_blocks_per_seq, context_lens, batch,
                       num_q_heads, scale, cache, partition_blocks, workspace, workspace_bytes,
                       phases, dev_status, stream);
}

kvp_status kvp_append_attention_decode(const void* key, const void* value, void* out,
                                       const void* q, void* k_cache, void* v_cache,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, int32_t batch,
                                       int32_t num_q_heads, float scale, kvp_cache_desc cache,
                                       kvp_dtype dtype, int32_t partition_blocks,
                                       void* workspace, size_t workspace_bytes,
                                       int32_t phases, int32_t* dev_status,
                                       kvp_stream_t stream) {
  KVP_NVTX_RANGE("kvp_append_attention_decode");
  if (dtype != KVP_F16 && dtype != KVP_BF16) return KVP_ERR_INVALID_ARG;
  if (batch > 0 && (!key || !value || !aligned(key, 16) || !aligned(value, 16)))
    return KVP_ERR_INVALID_ARG;
  return decode_common(out, q, dtype == KVP_BF16, dtype == KVP_BF16 ? 1 : 0, k_cache, v_cache,
                       nullptr, nullptr, block_tables, max_blocks_per_seq, context_lens, batch,
                       num_q_heads, scale, cache, partition_blocks, workspace, workspace_bytes,
                       phases, dev_status, stream, key, value);
}

kvp_status kvp_attention_decode_int8(void* out, const void* q, kvp_dtype q_dtype,
                                     const int8_t* k_cache, const int8_t* v_cache,
                                     const float* k_scale, const float* v_scale,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* context_lens, int32_t batch,
                                     int32_t num_q_heads, float scale, kvp_cache_desc cache,
                                     int32_t partition_blocks, void* workspace,
                                     size_t workspace_bytes, int32_t phases,
                                     int32_t* dev_status, kvp_stream_t stream) {
  KVP_NVTX_RANGE("kvp_attention_decode_int8");
  if (q_dtype != KVP_F16 && q_dtype != KVP_BF16) return KVP_ERR_INVALID_ARG;
  return decode_common(out, q, q_dtype == KVP_BF16, 2, k_cache, v_cache, k_scale, v_scale,
                       block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads, scale,
                       cache, partition_blocks, workspace, workspace_bytes, phases, dev_status,
                       stream);
}

kvp_status kvp_attention_decode_fp8(void* out, const void* q, kvp_dtype q_dtype,
                                    const uint8_t* k_cache, const uint8_t* v_cache,
                                    const float* k_scale, const float* v_scale,
                                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                                    const int32_t* context_lens, int32_t batch,
                                    int32_t num_q_heads, float scale, kvp_cache_desc cache,
                                    int32_t partition_blocks, void* workspace,
                                    size_t workspace_bytes, int32_t phases, int32_t* dev_status,
                                    kvp_stream_t stream) {
  KVP_NVTX_RANGE("kvp_attention_decode_fp8");
  if (q_dtype != KVP_F16 && q_dtype != KVP_BF16) return KVP_ERR_INVALID_ARG;
  return decode_common(out, q, q_dtype == KVP_BF16, 3, k_cache, v_cache, k_scale, v_scale,
                       block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads, scale,
                       cache, partition_blocks, workspace, workspace_bytes, phases, dev_status,
                       stream);
}

kvp_status kvp_attention_prefill(void* out, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* context_lens,
                                 const int32_t* query_start, int32_t num_query_tokens,
                                 int32_t batch, int32_t num_q_heads, int32_t max_query_len,
                                 int32_t shared_prefix_blocks, float scale,
                                 kvp_cache_desc cache, kvp_dtype dtype, int32_t* dev_status,
                                 kvp_stream_t stream) {
  KVP_NVTX_RANGE("kvp_attention_prefill");
  const kvp_status st = check_desc(cache);
  if (st != KVP_OK) return st;
  if (dtype != KVP_F16 && dtype != KVP_BF16) return KVP_ERR_INVALID_ARG;
  if (batch < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || max_query_len < 0 ||
      num_query_tokens < 0 || shared_prefix_blocks < 0 ||
      shared_prefix_blocks > max_blocks_per_seq)
    return KVP_ERR_INVALID_ARG;
  if (num_q_heads % cache.num_kv_heads != 0) return KVP_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return KVP_ERR_INVALID_ARG;
  const int group = num_q_heads / cache.num_kv_heads;
  if (128 % group != 0) return KVP_ERR_UNSUPPORTED;  // a 128-row tile holds whole groups
  if (batch == 0 || max_query_len == 0 || num_query_tokens == 0) return KVP_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start)
    return KVP_ERR_INVALID_ARG;
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return KVP_ERR_INVALID_ARG;
  // work items: per-request 128-row tiles, or (a shared prefix) dense tiles
  // over the whole batch's query rows
  const bool dense = shared_prefix_blocks > 0;
  const long long tiles = dense ? (static_cast<long long>(num_query_tokens) * group + 127) / 128
                                : (static_cast<long long>(max_query_len) * group + 127) / 128;
  if (tiles * (dense ? 1 : batch) * cache.num_kv_heads > 0x7fffffffll)
    return KVP_ERR_UNSUPPORTED;

  const int box_tokens = std::min(128 / group, static_cast<int>(num_query_tokens));
  CUtensorMap tq, tk, tv;
  kvp_status r = make_q_map(&tq, q, num_query_tokens, num_q_heads, cache.head_dim, group,
                            box_tokens);
  if (r != KVP_OK) return r;
  r = make_pool_map(&tk, k_cache, cache, 2);
  if (r != KVP_OK) return r;
  r = make_pool_map(&tv, v_cache, cache, 2);
  if (r != KVP_OK) return r;
  // out has q's shape [T, Hq, D]: full tiles leave through the same box
  CUtensorMap to;
  r = make_q_map(&to, out, num_query_tokens, num_q_heads, cache.head_dim, group, box_tokens);
  if (r != KVP_OK) return r;
  PrefillParams p{};
  p.out = out;
  p.q = q;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.query_start = query_start;
  p.status = dev_status;
  p.batch = batch;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = cache.num_kv_heads;
  p.head_dim = cache.head_dim;
  p.num_blocks = cache.num_blocks;
  p.max_blocks = max_blocks_per_seq;
  p.group = group;
  p.num_tokens = num_query_tokens;
  p.q_box_tokens = box_tokens;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.shared_blocks = shared_prefix_blocks;
  p.prefix_chunks = shared_prefix_blocks * kBlockSize / 128;
  return from_cuda(launch_prefill(p, tq, tk, tv, to, dtype == KVP_BF16, static_cast<int>(tiles),
                                  reinterpret_cast<cudaStream_t>(stream)));
}

size_t kvp_decode_shared_prefix_workspace_bytes(int32_t batch, int32_t num_q_heads,
                                                kvp_cache_desc cache, int32_t max_blocks_per_seq,
                                                int32_t shared_prefix_blocks,
                                                int32_t partition_blocks) {
  PrefixShape sh;
  if (batch < 0 || shape_prefix_decode(batch, num_q_heads, cache, max_blocks_per_seq,
                                       shared_prefix_blocks, partition_blocks, &sh) != KVP_OK)
    return 0;
  return sh.ws_bytes;
}

kvp_status kvp_attention_decode_shared_prefix(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t batch, int32_t num_q_heads, float scale, kvp_cache_desc cache, kvp_dtype dtype,
    int32_t shared_prefix_blocks, int32_t partition_blocks, void* workspace,
    size_t workspace_bytes, int32_t* dev_status, kvp_stream_t stream) {
  KVP_NVTX_RANGE("kvp_attention_decode_shared_prefix");
  if (dtype != KVP_F16 && dtype != KVP_BF16) return KVP_ERR_INVALID_ARG;
  if (batch < 0 || max_blocks_per_seq <= 0) return KVP_ERR_INVALID_ARG;
  PrefixShape sh;
  kvp_status r = shape_prefix_decode(batch, num_q_heads, cache, max_blocks_per_seq,
                                     shared_prefix_blocks, partition_blocks, &sh);
  if (r != KVP_OK) return r;
  if (sh.skip == 0)  // no whole chunk of shared prefix: the ordinary decode
    return decode_common(out, q, dtype == KVP_BF16, dtype == KVP_BF16 ? 1 : 0, k_cache,
                         v_cache, nullptr, nullptr, block_tables, max_blocks_per_seq,
                         context_lens, batch, num_q_heads, scale, cache, partition_blocks,
                         workspace, workspace_bytes, KVP_PHASE_PARTIAL | KVP_PHASE_REDUCE,
                         dev_status, stream);
  if (!std::isfinite(scale)) return KVP_ERR_INVALID_ARG;
  if (batch == 0) return KVP_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return KVP_ERR_INVALID_ARG;
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return KVP_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < sh.ws_bytes || !aligned(workspace, 16))
    return KVP_ERR_INVALID_ARG;
  const int group = num_q_heads / cache.num_kv_heads;
  if (static_cast<long long>(cache.num_kv_heads) * sh.suf.qgroups > 65535 || batch > 65535)
    return KVP_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* ws_o = static_cast<float*>(workspace);
  float* ws_ml = ws_o + static_cast<size_t>(batch) * num_q_heads * sh.max_parts * cache.head_dim;

  // 1. the prefix part: dense tiles of 128 (request, head) rows per kv head,
  // the prefix's full chunks only, into partition 0
  const int box_tokens = std::min(128 / group, static_cast<int>(batch));
  CUtensorMap tq, tk, tv;
  r = make_q_map(&tq, q, batch, num_q_heads, cache.head_dim, group, box_tokens);
  if (r != KVP_OK) return r;
  r = make_pool_map(&tk, k_cache, cache, 2);
  if (r != KVP_OK) return r;
  r = make_pool_map(&tv, v_cache, cache, 2);
  if (r != KVP_OK) return r;
  PrefillParams pp{};
  pp.q = q;
  pp.block_tables = block_tables;
  pp.context_lens = context_lens;
  pp.query_start = nullptr;  // one query per request
  pp.status = dev_status;
  pp.batch = batch;
  pp.num_q_heads = num_q_heads;
  pp.num_kv_heads = cache.num_kv_heads;
  pp.head_dim = cache.head_dim;
  pp.num_blocks = cache.num_blocks;
  pp.max_blocks = max_blocks_per_seq;
  pp.group = group;
  pp.num_tokens = batch;
  pp.q_box_tokens = box_tokens;
  pp.scale_log2 = scale * 1.4426950408889634f;
  pp.shared_blocks = shared_prefix_blocks;
  pp.prefix_chunks = sh.skip / 8;
  pp.partial = 1;
  pp.part_stride = sh.max_parts;
  pp.part_o = ws_o;
  pp.part_ml = ws_ml;
  const long long tiles = (static_cast<long long>(batch) * group + 127) / 128;
  if (launch_prefill(pp, tq, tk, tv, tq, dtype == KVP_BF16, static_cast<int>(tiles), s) !=
      cudaSuccess)
    return KVP_ERR_CUDA;

  // 2. the rest of every context: the split decode over blocks skip .. n - 1,
  // into partitions 1 ...
  DecodeParams p{};
  p.out = out;
  p.q = q;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.ws_o = ws_o;
  p.ws_ml = ws_ml;
  p.status = dev_status;
  p.batch = batch;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = cache.num_kv_heads;
  p.head_dim = cache.head_dim;
  p.num_blocks = cache.num_blocks;
  p.max_blocks = max_blocks_per_seq;
  p.group = group;
  p.qgroups = sh.suf.qgroups;
  p.heads_per_cta = sh.suf.heads_per_cta;
  p.part_blocks = sh.suf.part_blocks;
  p.max_parts = sh.max_parts;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.q_bf16 = dtype == KVP_BF16 ? 1 : 0;
  p.k_pool = k_cache;
  p.v_pool = v_cache;
  p.skip_blocks = sh.skip;
  DecodeMaps maps;
  maps.merged = false;
  maps.k = tk;
  maps.v = tv;
  cudaError_t e = sh.suf.path == DecodePath::kSimt
                      ? launch_decode_simt(p, maps, dtype == KVP_BF16, sh.suf.max_parts, s)
                      : launch_decode_mma(p, maps, dtype == KVP_BF16, sh.suf.max_parts, s);
  if (e != cudaSuccess) return KVP_ERR_CUDA;
  // 3. merge
  if (launch_decode_reduce(p, s) != cudaSuccess) return KVP_ERR_CUDA;
  return KVP_OK;
}

kvp_status kvp_selftest_wait_timeout(int32_t* dev_status, int64_t limit_ns,
                                     kvp_stream_t stream) {
  KVP_NVTX_RANGE("kvp_selftest_wait_timeout");
  if (dev_status == nullptr || limit_ns < 1000 || limit_ns > 5000000000ll)
    return KVP_ERR_INVALID_ARG;
  return from_cuda(launch_selftest_wait(dev_status, static_cast<uint64_t>(limit_ns),
                                        reinterpret_cast<cudaStream_t>(stream)));
}

kvp_status kvp_read_status(const int32_t* dev_status, kvp_stream_t stream) {
  KVP_NVTX_RANGE("kvp_read_status");
  if (dev_status == nullptr) return KVP_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, dev_status, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return KVP_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KVP_ERR_CUDA;
  if (v < KVP_OK || v > KVP_ERR_NOT_FOUND) return KVP_ERR_CUDA;
  return static_cast<kvp_status>(v);
}

}  // extern "C"

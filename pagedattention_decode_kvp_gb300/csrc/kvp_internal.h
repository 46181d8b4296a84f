// kvp_internal.h -- declarations shared by the library's translation units.
// Not part of the public ABI (see include/kvp.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include <utility>

#include "kvp.h"

namespace kvp {

// An NVTX range named after the entry point, open for the rest of the scope,
// so a profiler's timeline and its kernel filters (e.g. ncu --nvtx-include
// "kvp_attention_decode/") see each C-ABI call.  NVTX v3 is header-only; with
// no tool attached a push or pop is a check of one function pointer.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
#define KVP_NVTX_RANGE(name) ::kvp::NvtxRange kvp_nvtx_range_(name)

constexpr int kBlockSize = 16;       // tokens per cache block
constexpr int kWarps = 4;            // consumer warps per decode CTA
constexpr int kStagesPerWarp = 2;    // pipeline depth of each warp's ring
constexpr int kHeadsPerCta = 8;      // query heads one tensor-core CTA serves
constexpr int kMaxPartBlocks = 1024;  // table slice staged per CTA (4 KB)

// Decode kernel family.
enum class DecodePath : int { kSimt = 0, kMma = 1, kMmaInt8 = 2, kMmaFp8 = 3, kUmmaFp8 = 4 };

// Everything a decode launch needs besides the two tensor maps.
struct DecodeParams {
  void* out;                    // [B, Hq, D] of q dtype
  const void* q;                // [B, Hq, D]
  const float* k_scale;         // [NB, Hkv, bs] (INT8 pools only)
  const float* v_scale;
  const int32_t* block_tables;  // [B, MB]
  const int32_t* context_lens;  // [B]
  float* ws_o;                  // [B, Hq, P, D]
  float* ws_ml;                 // [B, Hq, P, 2]  (running max in log2 units, sum)
  int32_t* status;              // nullable
  int32_t batch, num_q_heads, num_kv_heads, head_dim, num_blocks, max_blocks;
  int32_t group;                // Hq / Hkv
  int32_t qgroups;              // CTAs per kv head along the query group
  int32_t heads_per_cta;        // query heads handled by one CTA
  int32_t part_blocks;          // blocks per partition
  int32_t max_parts;            // ceil(MB / part_blocks)
  float scale_log2;             // scale * log2(e)
  int32_t q_bf16;               // q / out are bf16 (else fp16)
  const void* new_k;            // fused append: [B, Hkv, D] token at position n-1, or null
  const void* new_v;
  const void* k_pool;           // pool base pointers (the fused append writes through them)
  const void* v_pool;
  int32_t skip_blocks;          // > 0: blocks [0, skip) are partition 0 of the workspace,
                                // written by another kernel (a shared prefix); this launch's
                                // partitions cover [skip, n) and are written as 1, 2, ...
};

// Everything a multi-query (prefill / chunked-prefill) launch needs besides the
// two tensor maps.  Query rows of request b are q[query_start[b] ..
// query_start[b+1]) and sit at the last positions of its context_lens[b].
struct PrefillParams {
  void* out;                     // [T, Hq, D] of the pool dtype
  const void* q;                 // [T, Hq, D]
  const int32_t* block_tables;   // [B, MB]
  const int32_t* context_lens;   // [B]
  const int32_t* query_start;    // [B + 1]
  int32_t* status;               // nullable
  int32_t batch, num_q_heads, num_kv_heads, head_dim, num_blocks, max_blocks;
  int32_t group;                 // Hq / Hkv (divides 128)
  int32_t num_tokens;            // T, rows of q and out
  int32_t q_box_tokens;          // tokens per Q tile copy: min(128 / group, T)
  float scale_log2;              // scale * log2(e)
  int32_t shared_blocks;         // > 0: leading table entries shared by all requests
                                 // (dense tiles over the whole batch's rows)
  int32_t prefix_chunks;         // full 128-key chunks inside the shared prefix
  // Decode over a shared prefix: query_start is null (one query per request,
  // rows of q / out are requests), only the prefix chunks are read, and each
  // row's unnormalised (o, m, l) goes to partition 0 of a decode workspace
  // (part_o [rows, part_stride, D], part_ml [rows, part_stride, 2]) instead of out.
  int32_t partial;
  int32_t part_stride;
  float* part_o;
  float* part_ml;
};

// Pool maps of the run-merged decode fetch: 5-D views {row piece (<= 128
// bytes), 16 rows, pieces per row, Hkv, NB} of a pool whose boxes hold whole
// (block, kv head) tiles of 1, 2 and 4 consecutive blocks (index 0, 1, 2).
struct RunMaps {
  CUtensorMap k[3];
  CUtensorMap v[3];
};

// Tensor maps of a decode launch: per-block fetch (2-D views [NB * Hkv * 16
// rows, D], a box of 16 rows x <= 128 bytes) or run-merged fetch.
struct DecodeMaps {
  bool merged;
  CUtensorMap k, v;  // per-block fetch
  RunMaps runs;      // run-merged fetch
};

// Device error codes (mirror kvp_status).
constexpr int32_t kErrBadBlock = KVP_ERR_BAD_BLOCK;
constexpr int32_t kErrTimeout = KVP_ERR_TIMEOUT;

// Host launchers implemented in the kernel translation units.  Each returns a
// cudaError_t from the launch.
cudaError_t launch_decode_simt(const DecodeParams& p, const DecodeMaps& m, bool kv_bf16,
                               int grid_x, cudaStream_t s);
cudaError_t launch_decode_mma(const DecodeParams& p, const DecodeMaps& m, bool kv_bf16,
                              int grid_x, cudaStream_t s);
cudaError_t launch_decode_mma_int8(const DecodeParams& p, const DecodeMaps& m, int grid_x,
                                   cudaStream_t s);
cudaError_t launch_decode_mma_fp8(const DecodeParams& p, const DecodeMaps& m, int grid_x,
                                  cudaStream_t s);
// FP8 pools, head_dim 128, on tcgen05 (kind::f8f6f4); per-block 2-D pool maps.
cudaError_t launch_decode_fp8_umma(const DecodeParams& p, const CUtensorMap& tk,
                                   const CUtensorMap& tv, int grid_x, cudaStream_t s);
cudaError_t launch_decode_reduce(const DecodeParams& p, cudaStream_t s);
// Self-test of the bounded wait: one block waits on a barrier nothing arrives
// on, for at most limit_ns, and records kErrTimeout when it gives up.
cudaError_t launch_selftest_wait(int32_t* status, uint64_t limit_ns, cudaStream_t s);

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& to, bool bf16, int grid_x,
                           cudaStream_t s);

// Launch `kernel` on stream `s` with programmatic stream serialisation, so its
// CTAs can be scheduled while the previous kernel drains (every kernel of this
// library starts with a grid-dependency wait, so this never lets it read data
// a predecessor is still writing).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device (once per device and kernel).
cudaError_t ensure_smem_attr(const void* kernel, size_t bytes);

cudaError_t launch_append(const void* key, const void* value, void* k_cache, void* v_cache,
                          const int32_t* slots, int num_tokens, const kvp_cache_desc& c,
                          int elem_bytes, int32_t* status, cudaStream_t s);
cudaError_t launch_append_int8(const void* key, const void* value, bool src_bf16,
                               int8_t* k_cache, int8_t* v_cache, float* k_scale,
                               float* v_scale, const int32_t* slots, int num_tokens,
                               const kvp_cache_desc& c, int32_t* status, cudaStream_t s);
cudaError_t launch_append_fp8(const void* key, const void* value, bool src_bf16,
                              uint8_t* k_cache, uint8_t* v_cache, float* k_scale, float* v_scale,
                              const int32_t* slots, int num_tokens, const kvp_cache_desc& c,
                              int32_t* status, cudaStream_t s);
cudaError_t launch_append_int8_fixed(const void* key, const void* value, bool src_bf16,
                                     int8_t* k_cache, int8_t* v_cache, float* k_scale_pool,
                                     float* v_scale_pool, float k_scale, float v_scale,
                                     const int32_t* slots, int num_tokens,
                                     const kvp_cache_desc& c, int32_t* status, cudaStream_t s);
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                               int elem_bytes, const int32_t* pairs, int num_pairs,
                               const kvp_cache_desc& c, int32_t* status, cudaStream_t s);

}  // namespace kvp

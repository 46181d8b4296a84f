/*
 * kvp.h -- C ABI of the paged-KV-cache decode library for NVIDIA GB300 (sm_103a).
 *
 * The problem, as the pages state it:
 *   - "ATB KV Cache management", "Paged KV Cache": the K/V cache is cut into
 *     fixed blocks of 16 tokens, allocated on demand and released when a
 *     request ends.
 *   - "ATB PagedAttention", "ATB 的 PagedAttention 实现": a per-request page
 *     table maps logical position i to page i / page_size, offset i % page_size.
 *   - "ATB PagedAttention", "PagedAttention 的 Attention 计算修改": decode
 *     attention of the request's query against its keys/values, walked page by
 *     page (query [batch, num_heads, head_dim], page table [request, max_pages]).
 *   - "KV Cache 优化与显存管理", 二: GQA shares one K/V head among a group of
 *     query heads; INT8 quantisation halves the cache.
 *   - "ATB PagedAttention", "踩坑三": copy-on-write of a shared last page.
 *
 * Layouts (all row-major, all device memory unless stated):
 *   q, out          [batch, num_q_heads, head_dim]        fp16 or bf16
 *   key, value      [num_tokens, num_kv_heads, head_dim]  (tokens to append)
 *   k/v cache pool  [num_blocks, num_kv_heads, block_size, head_dim]
 *   k/v scale pool  [num_blocks, num_kv_heads, block_size] float32 (INT8 pools)
 *   block_tables    [batch, max_blocks_per_seq] int32 physical block ids
 *   context_lens    [batch] int32, tokens already in the cache per request
 *   slot_mapping    [num_tokens] int32, slot = block * block_size + offset;
 *                   a negative slot marks a padding token that is skipped
 * Query head h reads K/V head h / (num_q_heads / num_kv_heads).
 *
 * Conventions:
 *   - The caller owns every buffer.  The library never allocates or frees
 *     device memory; scratch space for long contexts ("workspace") is passed
 *     in, sized by kvp_decode_workspace_bytes.
 *   - GPU entry points only enqueue work on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and return without synchronising.  Calls on
 *     the same buffers from several host threads must be serialised by the
 *     caller.
 *   - Host-checkable argument errors (null pointers, unsupported sizes,
 *     misaligned buffers, small workspace) return KVP_ERR_INVALID_ARG or
 *     KVP_ERR_UNSUPPORTED before anything is launched.  A failed launch returns
 *     KVP_ERR_CUDA.
 *   - Data errors found on the GPU (a block id outside [0, num_blocks), a slot
 *     at or past num_blocks * block_size, a context longer than
 *     max_blocks_per_seq * block_size, a pipeline wait that timed out) never
 *     fault: the offending work is skipped, affected output rows are written
 *     as zeros, and the error code is stored into *dev_status (a device int32,
 *     may be NULL) if it still holds KVP_OK (first error wins).  Read it with
 *     kvp_read_status.
 */
#ifndef KVP_H_
#define KVP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* kvp_stream_t;

typedef enum {
  KVP_OK = 0,
  KVP_ERR_INVALID_ARG = 1, /* bad pointer, size, shape or alignment            */
  KVP_ERR_UNSUPPORTED = 2, /* valid but not built (head_dim, block_size, ...)   */
  KVP_ERR_CUDA = 3,        /* a CUDA runtime / driver call failed              */
  KVP_ERR_BAD_BLOCK = 4,   /* device: block id, slot or context length invalid */
  KVP_ERR_TIMEOUT = 5,     /* device: a bounded pipeline wait gave up          */
  KVP_ERR_OOM = 6,         /* block manager: not enough free blocks            */
  KVP_ERR_REFCOUNT = 7,    /* block manager: release by a non-holder           */
  KVP_ERR_NOT_FOUND = 8,   /* block manager: unknown request id                */
  KVP_ERR_SCRATCH_LIMIT = 9 /* decode_noalloc: sizes need more than its scratch */
} kvp_status;

typedef enum { KVP_F16 = 0, KVP_BF16 = 1 } kvp_dtype;

/* Shape of one cache pool (K and V pools share it). */
typedef struct {
  int32_t num_blocks;   /* NB, physical blocks in the pool                    */
  int32_t num_kv_heads; /* Hkv                                                */
  int32_t block_size;   /* tokens per block; must be 16                       */
  int32_t head_dim;     /* D; 64 or 128                                       */
} kvp_cache_desc;

/* Which halves of a decode to run (kvp_attention_decode*, `phases`). */
enum {
  KVP_PHASE_PARTIAL = 1, /* per-partition pass: partial (m, l, o) to workspace,
                            or the final row for requests with one partition  */
  KVP_PHASE_REDUCE = 2,  /* merge of the partials into out                     */
  KVP_PHASE_ALL = 3,
  /* Flag, or'ed into `phases` of any decode entry point: fetch runs of
   * physically consecutive blocks ("ATB KV Cache management", "显存碎片问题":
   * contiguous-first allocation leaves most of a table as such runs) with one
   * copy per run of up to 4 blocks instead of one per block.  Same results,
   * bit for bit, as the default per-block fetch. */
  KVP_DECODE_MERGE_RUNS = 8
};

/* Human-readable name of a status code (static storage). */
const char* kvp_status_string(kvp_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t kvp_version(void);

/*
 * kvp_append -- scatter new tokens' K and V into their cache slots.
 * Source: "KV Cache 优化与显存管理", 三 (write_page writes a token at
 * (page, offset)); "ATB PagedAttention", "踩坑三" (WriteKV of the new token).
 * For every t < num_tokens with slot = slot_mapping[t] >= 0:
 *   k_cache[slot / bs, h, slot % bs, :] = key[t, h, :]   for all h (same for V).
 * key, value: [num_tokens, Hkv, D] of `dtype`; k_cache, v_cache: pools of `dtype`.
 * Bytes are copied unchanged.  Slots must be distinct (two tokens writing one
 * slot race).  num_tokens == 0 is a no-op.  Pools and sources must be 16-byte
 * aligned.  Device errors: KVP_ERR_BAD_BLOCK for slot >= NB * bs (token skipped).
 */
kvp_status kvp_append(const void* key, const void* value, void* k_cache, void* v_cache,
                      const int32_t* slot_mapping, int32_t num_tokens,
                      kvp_cache_desc cache, kvp_dtype dtype, int32_t* dev_status,
                      kvp_stream_t stream);

/*
 * kvp_append_int8 -- quantise new tokens per token and head, then scatter.
 * Source: "KV Cache 优化与显存管理", 三, KVCacheQuantizer, per-channel branch
 * (abs-max over the last axis / 127, zero scale replaced by 1, round half to
 * even, clip to [-128, 127]); 二 (INT8 halves the cache).  For each token t and
 * head h, with x = float32(key[t, h, :]):
 *   s = amax|x| / 127 (IEEE float division); s = 1 if s is not > 0;
 *   k_cache[blk, h, off, :] = clip(rint(x / s), -128, 127);  k_scale[blk, h, off] = s
 * and the same for V.  Results are bit-exact with that float32 definition.
 * key, value: [num_tokens, Hkv, D] of `src_dtype`; k_cache, v_cache: int8 pools;
 * k_scale, v_scale: float32 [NB, Hkv, bs].  Sources 16-byte aligned, int8 pools
 * 8-byte aligned.  Errors as kvp_append.
 */
kvp_status kvp_append_int8(const void* key, const void* value, kvp_dtype src_dtype,
                           int8_t* k_cache, int8_t* v_cache, float* k_scale,
                           float* v_scale, const int32_t* slot_mapping, int32_t num_tokens,
                           kvp_cache_desc cache, int32_t* dev_status, kvp_stream_t stream);

/*
 * kvp_append_int8_fixed -- per-tensor INT8: quantise with a given scale, scatter.
 * Source: "KV Cache 优化与显存管理", 三, KVCacheQuantizer, per_tensor branch (one
 * scale for the whole tensor, abs-max / 127).  A cache filled token by token
 * cannot see the whole tensor, so the scale is fixed ahead by the caller:
 *   k_cache[blk, h, off, :] = clip(rint(float32(key[t, h, :]) / k_scale), -128, 127)
 * (IEEE float32 division, round half to even) and k_scale is also written to
 * k_scale_pool[blk, h, off], so kvp_attention_decode_int8 reads these pools as
 * it reads per-token ones.  Same for V.  k_scale, v_scale: finite and > 0.
 * Other arguments and errors as kvp_append_int8.
 */
kvp_status kvp_append_int8_fixed(const void* key, const void* value, kvp_dtype src_dtype,
                                 int8_t* k_cache, int8_t* v_cache, float* k_scale_pool,
                                 float* v_scale_pool, float k_scale, float v_scale,
                                 const int32_t* slot_mapping, int32_t num_tokens,
                                 kvp_cache_desc cache, int32_t* dev_status, kvp_stream_t stream);

/*
 * kvp_append_fp8 -- FP8 (E4M3) per token and head quantisation, then scatter.
 * Source: "KV Cache 优化与显存管理", 二 (K and V quantised from FP16 to INT8 or
 * FP8).  The pages give the rule for INT8 only; this is the same rule with the
 * E4M3 format's largest magnitude, 448, in place of 127:
 *   s = amax|x| / 448 (IEEE float32 division); s = 1 if s is not > 0;
 *   code = E4M3 round-to-nearest-even of the float32 quotient x / s (saturating
 *          at +-448; OCP "e4m3fn" encoding: bias 7, no infinities).
 * Codes are bytes in uint8_t pools; otherwise as kvp_append_int8.
 */
kvp_status kvp_append_fp8(const void* key, const void* value, kvp_dtype src_dtype,
                          uint8_t* k_cache, uint8_t* v_cache, float* k_scale, float* v_scale,
                          const int32_t* slot_mapping, int32_t num_tokens, kvp_cache_desc cache,
                          int32_t* dev_status, kvp_stream_t stream);

/*
 * kvp_copy_blocks -- copy whole blocks (copy-on-write of a shared last block).
 * Source: "ATB PagedAttention", "踩坑三", ExtendKVPage: a page shared by
 * several requests is copied to a fresh page before a request writes to it.
 * For each pair p: block pairs[2p] (src) is copied onto block pairs[2p+1] (dst)
 * in k_cache and v_cache (all heads and slots), and in k_scale / v_scale when
 * they are non-NULL (INT8 pools).  cache_elem_bytes: 2 for fp16/bf16 pools,
 * 1 for int8.  pairs is a device array [num_pairs, 2].  A pair with src == dst
 * is skipped.  Destinations must be distinct and no destination may be the
 * source of another pair (the copies run concurrently).  Device errors:
 * KVP_ERR_BAD_BLOCK for an id outside [0, NB) (that pair is skipped).
 */
kvp_status kvp_copy_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                           int32_t cache_elem_bytes, const int32_t* pairs, int32_t num_pairs,
                           kvp_cache_desc cache, int32_t* dev_status, kvp_stream_t stream);

/*
 * kvp_decode_partition_blocks -- blocks per split-context partition that the
 * decode would use for these sizes when its `partition_blocks` argument is 0.
 * Long contexts are split into partitions that run as independent CTAs and are
 * merged by a reduce pass (flash-decoding); a return value >= max_blocks_per_seq
 * means single-pass (no workspace needed).  Returns 0 on invalid sizes.
 * kv_8bit: 0 for the fp16/bf16 decodes, 1 for the INT8 decode, 2 for the FP8
 * decode (the decodes run differently shaped CTAs).
 */
int32_t kvp_decode_partition_blocks(int32_t batch, int32_t num_q_heads, kvp_cache_desc cache,
                                    int32_t max_blocks_per_seq, int32_t kv_8bit);

/*
 * kvp_decode_workspace_bytes -- bytes of workspace the decode needs for these
 * sizes (0 when every request fits one partition).  partition_blocks as for the
 * decode (0 = automatic).  The workspace holds, per (request, query head,
 * partition), the partition's running max, sum and unnormalised output in
 * float32; it needs no initialisation and is fully rewritten by each call.
 * kv_8bit: 0 for the fp16/bf16 decodes, 1 for the INT8 decode, 2 for the FP8
 * decode; other values answer 0.
 */
size_t kvp_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, kvp_cache_desc cache,
                                  int32_t max_blocks_per_seq, int32_t partition_blocks,
                                  int32_t kv_8bit);

/*
 * kvp_attention_decode -- single-query paged attention over fp16/bf16 pools.
 * Source: "ATB PagedAttention", "PagedAttention 的 Attention 计算修改" (score
 * each cached key, online softmax page by page, weight V, normalise);
 * "ATB 的 PagedAttention 实现" (page table lookup); "踩坑一" (the page table is
 * staged on chip once); "KV Cache 优化与显存管理", 二 (GQA groups).
 * For each request b with n = context_lens[b] and query head h (g = h / G):
 *   out[b, h, :] = sum_i softmax_i(scale * q[b, h, :] . K_i) V_i,  i < n,
 *   K_i = k_cache[block_tables[b, i / 16], g, i % 16, :] (V likewise),
 * computed with float32 accumulation and written in `dtype`.  n == 0 gives a
 * zero row.  Only the first ceil(n / 16) table entries of a request are read,
 * and only its first n slots; other slots may hold anything (even NaN).
 * q, out: [batch, Hq, D] of `dtype`; pools of `dtype`; Hq % Hkv == 0.
 * partition_blocks: blocks per split-context partition (1 to 1024; values at or
 * above max_blocks_per_seq mean single pass), or 0 for the automatic choice.  workspace: >= kvp_decode_workspace_bytes(...)
 * bytes, 16-byte aligned (may be NULL when that is 0).  phases: KVP_PHASE_ALL,
 * or one of KVP_PHASE_PARTIAL / KVP_PHASE_REDUCE to run the halves as separate
 * calls (same arguments) -- e.g. to time them or to merge partials elsewhere.
 * Pools and q/out must be 16-byte aligned (pools 128-byte aligned).
 */
kvp_status kvp_attention_decode(void* out, const void* q, const void* k_cache,
                                const void* v_cache, const int32_t* block_tables,
                                int32_t max_blocks_per_seq, const int32_t* context_lens,
                                int32_t batch, int32_t num_q_heads, float scale,
                                kvp_cache_desc cache, kvp_dtype dtype,
                                int32_t partition_blocks, void* workspace,
                                size_t workspace_bytes, int32_t phases, int32_t* dev_status,
                                kvp_stream_t stream);

/*
 * kvp_append_attention_decode -- one decode step in one pass: append each
 * request's new token, then decode (fp16/bf16 pools).
 * Sources: as kvp_append and kvp_attention_decode.  key, value: [batch, Hkv, D]
 * of `dtype`, the K/V of request b's new token, which is written at position
 * context_lens[b] - 1 (slot = block_tables[b][(n-1)/16] * 16 + (n-1) % 16);
 * requests with context_lens[b] == 0 append nothing.  The result equals
 * kvp_append with those slots followed by kvp_attention_decode (KVP_PHASE_ALL),
 * but the append is done by the decode CTAs that read the request's last block,
 * saving a kernel launch and a pass over the new rows.  key/value 16-byte
 * aligned.  The append happens in the KVP_PHASE_PARTIAL pass.  Other arguments
 * and errors as kvp_attention_decode.
 */
kvp_status kvp_append_attention_decode(const void* key, const void* value, void* out,
                                       const void* q, void* k_cache, void* v_cache,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, int32_t batch,
                                       int32_t num_q_heads, float scale, kvp_cache_desc cache,
                                       kvp_dtype dtype, int32_t partition_blocks,
                                       void* workspace, size_t workspace_bytes, int32_t phases,
                                       int32_t* dev_status, kvp_stream_t stream);

/*
 * kvp_attention_decode_int8 -- as kvp_attention_decode over INT8 pools.
 * Source: "KV Cache 优化与显存管理", 三 (dequantize: code * scale), 二.
 * K_i = k_cache[...] * k_scale[blk, g, off] (V likewise); q and out are of
 * `q_dtype`.  Arguments otherwise as kvp_attention_decode.
 */
kvp_status kvp_attention_decode_int8(void* out, const void* q, kvp_dtype q_dtype,
                                     const int8_t* k_cache, const int8_t* v_cache,
                                     const float* k_scale, const float* v_scale,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* context_lens, int32_t batch,
                                     int32_t num_q_heads, float scale, kvp_cache_desc cache,
                                     int32_t partition_blocks, void* workspace,
                                     size_t workspace_bytes, int32_t phases,
                                     int32_t* dev_status, kvp_stream_t stream);

/*
 * kvp_attention_decode_fp8 -- as kvp_attention_decode_int8 over FP8 (E4M3)
 * pools: K_i = e4m3(k_cache[...]) * k_scale[blk, g, off] (V likewise), exact
 * widening of the codes, float32 accumulation.  Source: "KV Cache 优化与显存管理",
 * 二 (FP8 KV) and 三 (dequantize: code * scale).
 */
kvp_status kvp_attention_decode_fp8(void* out, const void* q, kvp_dtype q_dtype,
                                    const uint8_t* k_cache, const uint8_t* v_cache,
                                    const float* k_scale, const float* v_scale,
                                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                                    const int32_t* context_lens, int32_t batch,
                                    int32_t num_q_heads, float scale, kvp_cache_desc cache,
                                    int32_t partition_blocks, void* workspace,
                                    size_t workspace_bytes, int32_t phases, int32_t* dev_status,
                                    kvp_stream_t stream);

/*
 * kvp_attention_prefill -- causal multi-query paged attention over fp16/bf16
 * pools: the prompt (prefill) or a chunk of it (chunked prefill) attends to
 * the request's cached K/V through its block table.
 * Sources: "ATB KV Cache management", "Prefix Caching" (requests that share a
 * system prompt reuse its cached K/V, and only their own tokens are computed);
 * "ATB PagedAttention", "ATB 的 PagedAttention 实现" (the page-table walk).
 *   q, out        [T, num_q_heads, D] of `dtype`, T = num_query_tokens rows;
 *                 16-byte aligned.  out rows outside every request's range
 *                 are not written.
 *   query_start   [batch + 1] int32 (device), non-decreasing, query_start[0]
 *                 = 0: request b's query rows are query_start[b] ..
 *                 query_start[b+1] - 1, all below num_query_tokens.
 *   context_lens  [batch] int32 (device): n, the request's tokens in the cache
 *                 INCLUDING this chunk (append the chunk's K/V first).  Query
 *                 row i of request b (L = its row count) sits at position
 *                 n - L + i and attends to positions 0 .. n - L + i:
 *                 out = sum_j softmax_j(scale * q.K_j) V_j (causal mask).
 *   max_query_len an upper bound on every request's L; with the batch and
 *                 the kv heads it sizes the list of 128-row work items
 *                 (ceil(max_query_len * G / 128) per request and kv head),
 *                 which must stay below 2^31 (KVP_ERR_UNSUPPORTED otherwise).
 *   shared_prefix_blocks  S >= 0.  S > 0 states that the first S entries of
 *                 every request's block table (of the requests with query
 *                 rows) name the same physical blocks -- a prompt prefix
 *                 cached once and shared ("Prefix Caching") -- and that each
 *                 such request holds n >= 16 * S tokens.  The rows of all
 *                 requests are then packed into 128-row tiles of consecutive
 *                 query tokens (no tile is padded at a request's end) and the
 *                 prefix's whole 128-key chunks are read through one table;
 *                 each request's other keys through its own.  Results are
 *                 those of S = 0, bit for bit.  A table that disagrees on the
 *                 first S entries, or n < 16 * S, is a data error
 *                 (KVP_ERR_BAD_BLOCK; the tiles holding that request's rows
 *                 are written as zeros).  With S > 0 the work items are
 *                 ceil(num_query_tokens * G / 128) per kv head and
 *                 max_query_len is not used to size them.
 *   k/v cache, block_tables, max_blocks_per_seq, cache: as kvp_attention_decode.
 * num_q_heads / num_kv_heads must divide 128 (KVP_ERR_UNSUPPORTED otherwise).
 * Device-side errors (*dev_status): KVP_ERR_BAD_BLOCK when a block id is out of
 * range (every 128-row tile that reads one is written as zeros), when L > n,
 * n > max_blocks_per_seq * 16 or L > max_query_len (the request's rows that
 * are reached are written as zeros), or when a request's rows reach past
 * num_query_tokens (nothing of it is written); KVP_ERR_TIMEOUT when a pipeline
 * wait gave up; KVP_ERR_UNSUPPORTED if the device placed the kernel's shared
 * memory off a 1024-byte boundary (nothing is computed; not expected).
 * Computed on the tensor cores with float32 accumulation by one persistent
 * block per SM; no workspace.
 */
kvp_status kvp_attention_prefill(void* out, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* context_lens,
                                 const int32_t* query_start, int32_t num_query_tokens,
                                 int32_t batch, int32_t num_q_heads, int32_t max_query_len,
                                 int32_t shared_prefix_blocks, float scale,
                                 kvp_cache_desc cache, kvp_dtype dtype, int32_t* dev_status,
                                 kvp_stream_t stream);

/*
 * kvp_decode_shared_prefix_workspace_bytes -- bytes of workspace
 * kvp_attention_decode_shared_prefix needs for these sizes (0 for invalid
 * sizes).  Same layout as the decode's workspace, with one more partition per
 * (request, query head): the shared prefix's part.
 */
size_t kvp_decode_shared_prefix_workspace_bytes(int32_t batch, int32_t num_q_heads,
                                                kvp_cache_desc cache, int32_t max_blocks_per_seq,
                                                int32_t shared_prefix_blocks,
                                                int32_t partition_blocks);

/*
 * kvp_attention_decode_shared_prefix -- kvp_attention_decode for a batch whose
 * requests share a cached prompt prefix: the first shared_prefix_blocks table
 * entries of every request name the same physical blocks ("ATB KV Cache
 * management", "Prefix Caching": the shared prefix's K/V is cached once and
 * reused by every request).  The result is the decode's (same definition, same
 * tolerance); only the order of the sums differs.  The prefix's whole 128-token
 * chunks are attended once per kv head for every request's query together, on
 * the tensor cores, instead of once per request; the rest of each context runs
 * as the ordinary split-context decode; a reduce merges the two.  Every
 * context_lens[b] must cover the shared prefix (>= 16 * shared_prefix_blocks),
 * and every request's table must name the first request's prefix blocks:
 * otherwise the rows of the 128-row tile holding that request (128 / G
 * requests of one kv head, G = Hq / Hkv) are zeros and *dev_status gets
 * KVP_ERR_BAD_BLOCK.  A prefix shorter than 128 tokens, or a query group that
 * does not divide 128, runs the ordinary decode.  fp16/bf16 pools only;
 * workspace: >= kvp_decode_shared_prefix_workspace_bytes(...) bytes, 16-byte
 * aligned (required).  Other arguments as kvp_attention_decode.
 */
kvp_status kvp_attention_decode_shared_prefix(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t batch, int32_t num_q_heads, float scale, kvp_cache_desc cache, kvp_dtype dtype,
    int32_t shared_prefix_blocks, int32_t partition_blocks, void* workspace,
    size_t workspace_bytes, int32_t* dev_status, kvp_stream_t stream);

/*
 * kvp_attention_decode_noalloc -- kvp_attention_decode for callers that cannot
 * allocate device memory.  (The pages have no counterpart: this entry point
 * exists for integration, not for the method.)
 *
 * Long contexts need a workspace for their split-context partial results, and
 * kvp_attention_decode takes it from the caller.  Callers that cannot allocate
 * -- a plugin whose host framework owns all device memory and hands it only
 * input and output buffers, or a serving loop that gave nearly all free HBM to
 * the KV pool and must not risk a failing or synchronising cudaMalloc in the
 * middle of a step -- call this instead: it uses a scratch array built into
 * the library (KVP_NOALLOC_SCRATCH_BYTES of device memory that every GPU which
 * loads the library holds until the process exits) and calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *   - Arguments and results are those of kvp_attention_decode (fp16/bf16 pools,
 *     all phases) without the workspace arguments.
 *   - Returns KVP_ERR_SCRATCH_LIMIT, before launching anything, when these sizes
 *     need more than KVP_NOALLOC_SCRATCH_BYTES of workspace
 *     (kvp_decode_workspace_bytes tells how much they need).
 *   - The first call on each device that needs partials looks up the scratch
 *     array's device address (cudaGetSymbolAddress, with that device current);
 *     make that first call before any stream capture.  The address is cached
 *     per device and per context: after a device reset (or from a new context)
 *     the next such call looks it up again, so it too belongs before any
 *     capture.  Calls whose contexts fit one partition, and calls with
 *     arguments the decode rejects, never look it up.
 *   - Every call, on any stream, shares the one array: calls that overlap on the
 *     GPU race and corrupt each other's results.  Serialise them (one stream, or
 *     events).  The array keeps the last call's contents; nothing in it needs to
 *     start at zero, each call rewrites what it reads.
 */
#define KVP_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
kvp_status kvp_attention_decode_noalloc(void* out, const void* q, const void* k_cache,
                                        const void* v_cache, const int32_t* block_tables,
                                        int32_t max_blocks_per_seq, const int32_t* context_lens,
                                        int32_t batch, int32_t num_q_heads, float scale,
                                        kvp_cache_desc cache, kvp_dtype dtype,
                                        int32_t partition_blocks, int32_t* dev_status,
                                        kvp_stream_t stream);

/*
 * kvp_selftest_wait_timeout -- a diagnostic (the pages have no counterpart):
 * launches one block whose two warps wait, through the same bounded mbarrier
 * wait every pipeline of this library uses, on barriers that nothing arrives
 * on: the first gives up after `limit_ns` nanoseconds of wall-clock time
 * (1e3 .. 5e9), as the kernels do after 2 s when a copy or a hand-off never
 * comes, and sets the block's abort flag; the second, waiting with the
 * default 2 s limit, sees the flag and gives up within 16 tries (about a
 * third of a millisecond), as every wait that polls the flag does.  The
 * waits record KVP_ERR_TIMEOUT in *dev_status (if it still holds KVP_OK);
 * nothing faults and the stream stays usable.  Returns KVP_ERR_INVALID_ARG for a null
 * status or a limit outside the range, KVP_ERR_CUDA if the launch fails.
 */
kvp_status kvp_selftest_wait_timeout(int32_t* dev_status, int64_t limit_ns, kvp_stream_t stream);

/*
 * kvp_read_status -- synchronise `stream`, read the device status word and
 * return it as a kvp_status (KVP_ERR_CUDA if the read fails).  Does not reset
 * the word; write 0 to it to clear.
 */
kvp_status kvp_read_status(const int32_t* dev_status, kvp_stream_t stream);

/* ------------------------------------------------------------------------
 * Host block manager (plain C++, no CUDA).  Keeps the free pool, per-request
 * block tables and per-block reference counts.
 * Sources: "ATB KV Cache management", "BlockManager 的调度" (free list,
 * ceil(tokens / block_size) blocks per request, blocks returned on free) and
 * "显存碎片问题" (prefer a contiguous run from the largest free range, else
 * scatter); "KV Cache 优化与显存管理", 三 (allocation fails cleanly when short,
 * a new block when tokens exceed capacity, memory statistics); "ATB
 * PagedAttention", "ATB 的 PagedAttention 实现" (reference counts, OUT_OF_MEMORY),
 * "踩坑二" (release decrements, frees at zero; release by a non-holder is an
 * error) and "踩坑三" (copy-on-write when the last block is shared).
 * Not thread-safe: one manager per thread, or external locking.
 * ---------------------------------------------------------------------- */
typedef struct kvp_bm kvp_bm;

typedef struct {
  int32_t total_blocks;
  int32_t used_blocks;      /* blocks with reference count > 0                 */
  int32_t free_blocks;
  int32_t active_requests;
  int64_t block_refs;       /* sum of reference counts = table entries held    */
  double utilization;       /* used / total, in [0, 1]                         */
  int64_t bytes_per_block;  /* as given to kvp_bm_create                       */
  double total_memory_gb;   /* total_blocks * bytes_per_block / 1e9            */
} kvp_bm_stats_t;

/* A pool of num_blocks blocks of block_size tokens (bytes_per_block only feeds
 * the statistics).  Returns NULL on invalid sizes or allocation failure. */
kvp_bm* kvp_bm_create(int32_t num_blocks, int32_t block_size, int64_t bytes_per_block);
void kvp_bm_destroy(kvp_bm* bm);

/* Give request `req` (a new id) ceil(num_tokens / block_size) + reserve_blocks
 * blocks, contiguous when a free range that long exists (the largest such
 * range is used), otherwise the lowest free ids.  KVP_ERR_OOM leaves the
 * manager unchanged; KVP_ERR_INVALID_ARG if req exists or sizes are negative. */
kvp_status kvp_bm_allocate(kvp_bm* bm, int64_t req, int32_t num_tokens, int32_t reserve_blocks);

/* New request `dst` shares the blocks holding the first num_tokens tokens of
 * `src` (reference counts incremented); dst's length becomes num_tokens. */
kvp_status kvp_bm_share_prefix(kvp_bm* bm, int64_t src, int64_t dst, int32_t num_tokens);

/* Reserve the slot of request req's next token.  Takes a new block when the
 * request's blocks are full.  If the block receiving the token is shared
 * (reference count > 1), a fresh block replaces it in req's table and
 * (*cow_src, *cow_dst) name the copy to run first (kvp_copy_blocks); otherwise
 * both are -1.  *slot = block * block_size + offset. */
kvp_status kvp_bm_append_slot(kvp_bm* bm, int64_t req, int32_t* slot, int32_t* cow_src,
                              int32_t* cow_dst);

/* Release every block reference of `req` (a block returns to the free pool
 * when its count reaches zero) and forget the request. */
kvp_status kvp_bm_free(kvp_bm* bm, int64_t req);

/* Drop request req's reference to one physical block.  KVP_ERR_REFCOUNT if
 * req does not hold it. */
kvp_status kvp_bm_release_block(kvp_bm* bm, int64_t req, int32_t block);

/* Copy up to cap block ids of req's table into out; returns the table length,
 * or -1 for an unknown request. */
int32_t kvp_bm_block_table(const kvp_bm* bm, int64_t req, int32_t* out, int32_t cap);

/* Tokens currently held by req, or -1 for an unknown request. */
int32_t kvp_bm_num_tokens(const kvp_bm* bm, int64_t req);

/* Reference count of a block (0 = free), -1 for an id out of range. */
int32_t kvp_bm_ref_count(const kvp_bm* bm, int32_t block);

void kvp_bm_stats(const kvp_bm* bm, kvp_bm_stats_t* out);

#ifdef __cplusplus
}
#endif

#endif /* KVP_H_ */

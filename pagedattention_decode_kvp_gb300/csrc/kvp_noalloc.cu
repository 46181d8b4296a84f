// kvp_noalloc.cu -- decode for callers that cannot allocate device memory.
//
// kvp_attention_decode splits long contexts into partitions whose partial
// results live in a caller-provided workspace.  Some callers cannot provide
// one: a plugin inside a host framework that owns all device memory and hands
// the plugin only its input and output buffers, or a serving loop that has
// given nearly all free HBM to the KV pool and cannot risk a cudaMalloc (which
// may fail, or synchronise the device) in the middle of a decode step.
// kvp_attention_decode_noalloc serves them from a scratch array compiled into
// this library instead: g_decode_scratch below, KVP_NOALLOC_SCRATCH_BYTES
// (64 MiB) of device memory that every GPU which loads the library keeps
// until the process exits.  No cudaMalloc, cudaFree or allocating library
// routine is called.
#include <cudaTypedefs.h>

#include <mutex>

#include "kvp_internal.h"

namespace {

__device__ __align__(256) unsigned char g_decode_scratch[KVP_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
struct ScratchEntry {
  void* addr;                 // device address of g_decode_scratch
  unsigned long long ctx_id;  // the context it belongs to (0: none yet)
};
ScratchEntry g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Unique id of the calling thread's current context (0 when there is none, or
// when the driver cannot say).  A device reset or a new context on the same
// device loads the library's device code again, possibly at another address,
// and gets a new id, so a cached address is only reused within its context.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr) return 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_decode_scratch on the current device.  In host code the
// symbol itself is only a host-side stand-in, so its address is looked up with
// the device current (cudaGetSymbolAddress, which allocates nothing) and cached
// per device together with the context it was found in; a call from another
// context (after a device reset, say) looks it up again.
kvp_status scratch_address(void** out) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return KVP_ERR_CUDA;
  if (device < 0 || device >= kMaxDevices) return KVP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchEntry& e = g_scratch[device];
  const unsigned long long id = current_context_id();
  if (e.addr == nullptr || id == 0 || e.ctx_id != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return KVP_ERR_CUDA;
    e.addr = p;
    e.ctx_id = current_context_id();  // the lookup made the primary context current
  }
  *out = e.addr;
  return KVP_OK;
}

}  // namespace

extern "C" kvp_status kvp_attention_decode_noalloc(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t batch, int32_t num_q_heads, float scale, kvp_cache_desc cache, kvp_dtype dtype,
    int32_t partition_blocks, int32_t* dev_status, kvp_stream_t stream) {
  KVP_NVTX_RANGE("kvp_attention_decode_noalloc");
  const size_t need = kvp_decode_workspace_bytes(batch, num_q_heads, cache, max_blocks_per_seq,
                                                 partition_blocks, 0);
  if (need > static_cast<size_t>(KVP_NOALLOC_SCRATCH_BYTES)) return KVP_ERR_SCRATCH_LIMIT;
  // Calls that need no partials (short contexts, or arguments the decode
  // rejects, for which the size is 0) never touch the scratch array.
  void* scratch = nullptr;
  if (need > 0) {
    const kvp_status st = scratch_address(&scratch);
    if (st != KVP_OK) return st;
  }
  // The partial results are fully rewritten by every call before they are
  // read, so nothing in the scratch array needs clearing between calls.
  return kvp_attention_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                              context_lens, batch, num_q_heads, scale, cache, dtype,
                              partition_blocks, scratch,
                              static_cast<size_t>(KVP_NOALLOC_SCRATCH_BYTES), KVP_PHASE_ALL,
                              dev_status, stream);
}

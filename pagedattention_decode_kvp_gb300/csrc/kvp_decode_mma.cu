// Instantiations of the tensor-core decode consumer for fp16/bf16 pools.
#include "kvp_decode.cuh"

namespace kvp {

cudaError_t launch_decode_mma(const DecodeParams& p, const DecodeMaps& m, bool kv_bf16,
                              int grid_x, cudaStream_t s) {
  if (!kv_bf16 && p.head_dim == 64) return launch_partial<MmaPath<false, 64>>(p, m, grid_x, s);
  if (!kv_bf16 && p.head_dim == 128) return launch_partial<MmaPath<false, 128>>(p, m, grid_x, s);
  if (kv_bf16 && p.head_dim == 64) return launch_partial<MmaPath<true, 64>>(p, m, grid_x, s);
  if (kv_bf16 && p.head_dim == 128) return launch_partial<MmaPath<true, 128>>(p, m, grid_x, s);
  return cudaErrorInvalidValue;
}

}  // namespace kvp

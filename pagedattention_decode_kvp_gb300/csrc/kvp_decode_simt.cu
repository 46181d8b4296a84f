// Instantiations of the CUDA-core decode consumer (1-2 query heads per kv head).
#include "kvp_decode.cuh"

namespace kvp {

cudaError_t launch_decode_simt(const DecodeParams& p, const DecodeMaps& m, bool kv_bf16,
                               int grid_x, cudaStream_t s) {
#define KVP_SIMT_CASE(BF, DD, GG)                                              \
  if (kv_bf16 == BF && p.head_dim == DD && p.heads_per_cta == GG)              \
    return launch_partial<SimtPath<BF, DD, GG>>(p, m, grid_x, s);
  KVP_SIMT_CASE(false, 64, 1)
  KVP_SIMT_CASE(false, 64, 2)
  KVP_SIMT_CASE(false, 128, 1)
  KVP_SIMT_CASE(false, 128, 2)
  KVP_SIMT_CASE(true, 64, 1)
  KVP_SIMT_CASE(true, 64, 2)
  KVP_SIMT_CASE(true, 128, 1)
  KVP_SIMT_CASE(true, 128, 2)
#undef KVP_SIMT_CASE
  return cudaErrorInvalidValue;
}

}  // namespace kvp

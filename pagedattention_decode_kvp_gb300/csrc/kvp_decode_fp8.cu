// Instantiations of the tensor-core decode consumer for FP8 (E4M3) pools.
#include "kvp_decode.cuh"

namespace kvp {

cudaError_t launch_decode_mma_fp8(const DecodeParams& p, const DecodeMaps& m, int grid_x,
                                  cudaStream_t s) {
  const bool qbf = p.q_bf16 != 0;
  if (!qbf && p.head_dim == 64)
    return launch_partial<MmaInt8Path<false, 64, true>>(p, m, grid_x, s);
  if (!qbf && p.head_dim == 128)
    return launch_partial<MmaInt8Path<false, 128, true>>(p, m, grid_x, s);
  if (qbf && p.head_dim == 64)
    return launch_partial<MmaInt8Path<true, 64, true>>(p, m, grid_x, s);
  if (qbf && p.head_dim == 128)
    return launch_partial<MmaInt8Path<true, 128, true>>(p, m, grid_x, s);
  return cudaErrorInvalidValue;
}

}  // namespace kvp

// Split-context reduce: merge the per-partition (m, l, o) of each (request,
// query head) into the final output row (flash-decoding's second pass).
//   M = max_p m_p;  w_p = 2^(m_p - M);  out = sum_p w_p o_p / sum_p w_p l_p
// (m_p is kept in log2 units, o_p unnormalised).  A partition that failed its
// checks is marked with l_p < 0 and turns the whole row into zeros.
#include <mutex>
#include <set>
#include <utility>

#include "kvp_device.cuh"
#include "kvp_internal.h"

namespace kvp {

template <int D, bool kBf16Out>
__global__ void __launch_bounds__(128) decode_reduce_kernel(const DecodeParams p) {
  constexpr int E = D / 32;  // output elements per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + warp;  // (b, h) flattened
  if (row >= p.batch * p.num_q_heads) return;
  const int b = row / p.num_q_heads;
  const int n = p.context_lens[b];
  if (n <= 0 || n > p.max_blocks * kBlockSize) return;  // written by the partition pass
  const int nblk = (n + kBlockSize - 1) / kBlockSize;
  const int nparts = (nblk + p.part_blocks - 1) / p.part_blocks;
  if (nparts <= 1) return;

  const float* ml = p.ws_ml + static_cast<size_t>(row) * p.max_parts * 2;
  const float* wo = p.ws_o + static_cast<size_t>(row) * p.max_parts * D + lane * E;
  float M = -INFINITY;
  bool bad = false;
  for (int i = lane; i < nparts; i += 32) {
    const float2 v = *reinterpret_cast<const float2*>(ml + 2 * i);
    M = fmaxf(M, v.x);
    bad |= v.y < 0.f;
  }
  M = dev::warp_max(M);
  bad = __any_sync(0xffffffffu, bad);

  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float L = 0.f;
  if (!bad) {
#pragma unroll 4
    for (int i = 0; i < nparts; ++i) {
      const float2 v = *reinterpret_cast<const float2*>(ml + 2 * i);
      const float f = exp2f(v.x - M);
      L = fmaf(f, v.y, L);
      if constexpr (E == 4) {
        const float4 x = *reinterpret_cast<const float4*>(wo + static_cast<size_t>(i) * D);
        acc[0] = fmaf(f, x.x, acc[0]);
        acc[1] = fmaf(f, x.y, acc[1]);
        acc[2] = fmaf(f, x.z, acc[2]);
        acc[3] = fmaf(f, x.w, acc[3]);
      } else {
        const float2 x = *reinterpret_cast<const float2*>(wo + static_cast<size_t>(i) * D);
        acc[0] = fmaf(f, x.x, acc[0]);
        acc[1] = fmaf(f, x.y, acc[1]);
      }
    }
  }
  uint16_t* out = static_cast<uint16_t*>(p.out) + static_cast<size_t>(row) * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const float r = (!bad && L > 0.f) ? acc[e] / L : 0.f;
    out[e] = dev::from_float<kBf16Out>(r);
  }
}

cudaError_t launch_decode_reduce(const DecodeParams& p, cudaStream_t s) {
  const int rows = p.batch * p.num_q_heads;
  const dim3 grid((rows + 3) / 4);
  if (p.head_dim == 64) {
    if (p.q_bf16) decode_reduce_kernel<64, true><<<grid, 128, 0, s>>>(p);
    else decode_reduce_kernel<64, false><<<grid, 128, 0, s>>>(p);
  } else if (p.head_dim == 128) {
    if (p.q_bf16) decode_reduce_kernel<128, true><<<grid, 128, 0, s>>>(p);
    else decode_reduce_kernel<128, false><<<grid, 128, 0, s>>>(p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t ensure_smem_attr(const void* kernel, size_t bytes) {
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({kernel, device})) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes));
  if (e == cudaSuccess) done.insert({kernel, device});
  return e;
}

}  // namespace kvp

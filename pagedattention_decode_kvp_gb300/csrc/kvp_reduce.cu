// Split-context reduce: merge the per-partition (m, l, o) of each (request,
// query head) into the final output row (flash-decoding's second pass).
//   M = max_p m_p;  w_p = 2^(m_p - M);  out = sum_p w_p o_p / sum_p w_p l_p
// (m_p is kept in log2 units, o_p unnormalised).  A partition that failed its
// checks is marked with l_p < 0 and turns the whole row into zeros.  The
// partials were written moments before, so they are read mostly from L2.
#include <mutex>
#include <set>
#include <utility>

#include "kvp_device.cuh"
#include "kvp_internal.h"

namespace kvp {

// One CTA of 8 warps per (request, query head) row: all threads find the
// largest partition max, warp w accumulates partitions w, w+8, ... (one lane
// per D/32 output elements, independent loads), shared memory sums the warps.
template <int D, bool kBf16Out>
__global__ void __launch_bounds__(256) decode_reduce_kernel(const DecodeParams p) {
  constexpr int E = D / 32;  // output elements per lane
  constexpr int W = 8;
  __shared__ __align__(16) float s_acc[W][D];
  __shared__ float s_m[W];
  __shared__ float s_l[W];
  dev::grid_dependency_wait();  // the partition pass has written the workspace
  dev::launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x;  // (b, h) flattened
  const int b = row / p.num_q_heads;
  const int n = p.context_lens[b];
  if (n <= 0 || n > p.max_blocks * kBlockSize) return;  // written by the partition pass
  const int nblk = (n + kBlockSize - 1) / kBlockSize;
  // with a shared prefix (skip_blocks > 0) partition 0 holds the prefix part
  // and the rest cover blocks skip .. nblk - 1; the row is always merged here
  const int nparts = p.skip_blocks > 0
                         ? 1 + (max(nblk - p.skip_blocks, 0) + p.part_blocks - 1) / p.part_blocks
                         : (nblk + p.part_blocks - 1) / p.part_blocks;
  if (nparts <= 1 && p.skip_blocks == 0) return;

  const float* ml = p.ws_ml + static_cast<size_t>(row) * p.max_parts * 2;
  const float* wo = p.ws_o + static_cast<size_t>(row) * p.max_parts * D + lane * E;
  float M = -INFINITY;
  bool bad = false;
  for (int i = threadIdx.x; i < nparts; i += blockDim.x) {
    const float2 v = *reinterpret_cast<const float2*>(ml + 2 * i);
    M = fmaxf(M, v.x);
    bad |= v.y < 0.f;
  }
  M = dev::warp_max(M);
  if (lane == 0) s_m[warp] = M;
  bad = __syncthreads_or(bad);
  M = s_m[0];
#pragma unroll
  for (int w = 1; w < W; ++w) M = fmaxf(M, s_m[w]);

  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float L = 0.f;
  if (!bad) {
#pragma unroll 4
    for (int i = warp; i < nparts; i += W) {
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
  if constexpr (E == 4) {
    *reinterpret_cast<float4*>(&s_acc[warp][lane * 4]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
  } else {
    *reinterpret_cast<float2*>(&s_acc[warp][lane * 2]) = make_float2(acc[0], acc[1]);
  }
  if (lane == 0) s_l[warp] = L;
  __syncthreads();
  if (threadIdx.x < D) {
    float a = 0.f, lt = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      a += s_acc[w][threadIdx.x];
      lt += s_l[w];
    }
    const float r = (!bad && lt > 0.f) ? a / lt : 0.f;
    static_cast<uint16_t*>(p.out)[static_cast<size_t>(row) * D + threadIdx.x] =
        dev::from_float<kBf16Out>(r);
  }
}

cudaError_t launch_decode_reduce(const DecodeParams& p, cudaStream_t s) {
  const dim3 grid(p.batch * p.num_q_heads);
  const dim3 block(256);
  if (p.head_dim == 64) {
    return p.q_bf16 ? launch_pdl(decode_reduce_kernel<64, true>, grid, block, 0, s, p)
                    : launch_pdl(decode_reduce_kernel<64, false>, grid, block, 0, s, p);
  }
  if (p.head_dim == 128) {
    return p.q_bf16 ? launch_pdl(decode_reduce_kernel<128, true>, grid, block, 0, s, p)
                    : launch_pdl(decode_reduce_kernel<128, false>, grid, block, 0, s, p);
  }
  return cudaErrorInvalidValue;
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

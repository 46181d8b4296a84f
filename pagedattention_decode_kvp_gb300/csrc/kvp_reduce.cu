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

// One warp per row, for splits of at most 8 partitions (most rows of a
// short or medium context), eight rows per CTA: a block of 256 threads per row
// would spend its time being scheduled and synchronised.  Lane i holds
// partition i's (m, l); every lane accumulates its D/32 output elements over
// the partitions in order (independent loads), multiplying and adding
// separately, so a row comes out bit for bit as decode_reduce_kernel writes
// it (one partition per warp there, summed in warp order).
template <int D, bool kBf16Out>
__global__ void __launch_bounds__(256) decode_reduce_warp_kernel(const DecodeParams p) {
  constexpr int E = D / 32;  // output elements per lane
  constexpr int kMaxParts = 8;
  dev::grid_dependency_wait();  // the partition pass has written the workspace
  dev::launch_dependents();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);  // (b, h) flattened
  if (row >= p.batch * p.num_q_heads) return;
  const int b = row / p.num_q_heads;
  const int n = p.context_lens[b];
  if (n <= 0 || n > p.max_blocks * kBlockSize) return;  // written by the partition pass
  const int nblk = (n + kBlockSize - 1) / kBlockSize;
  const int nparts = p.skip_blocks > 0
                         ? 1 + (max(nblk - p.skip_blocks, 0) + p.part_blocks - 1) / p.part_blocks
                         : (nblk + p.part_blocks - 1) / p.part_blocks;
  if (nparts <= 1 && p.skip_blocks == 0) return;

  const float* ml = p.ws_ml + static_cast<size_t>(row) * p.max_parts * 2;
  const float* wo = p.ws_o + static_cast<size_t>(row) * p.max_parts * D + lane * E;
  float2 v = make_float2(-INFINITY, 0.f);
  if (lane < nparts) v = *reinterpret_cast<const float2*>(ml + 2 * lane);
  const float M = dev::warp_max(v.x);
  const bool bad = __any_sync(0xffffffffu, lane < nparts && v.y < 0.f);

  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float L = 0.f;
  if (!bad) {
#pragma unroll
    for (int i = 0; i < kMaxParts; ++i) {
      if (i < nparts) {
        const float f = exp2f(__shfl_sync(0xffffffffu, v.x, i) - M);
        L = __fadd_rn(L, __fmul_rn(f, __shfl_sync(0xffffffffu, v.y, i)));
        float x[E];
        if constexpr (E == 4) {
          const float4 t = *reinterpret_cast<const float4*>(wo + static_cast<size_t>(i) * D);
          x[0] = t.x;
          x[1] = t.y;
          x[2] = t.z;
          x[3] = t.w;
        } else {
          const float2 t = *reinterpret_cast<const float2*>(wo + static_cast<size_t>(i) * D);
          x[0] = t.x;
          x[1] = t.y;
        }
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = __fadd_rn(acc[e], __fmul_rn(f, x[e]));
      }
    }
  }
  uint16_t* out = static_cast<uint16_t*>(p.out) + static_cast<size_t>(row) * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e)
    out[e] = dev::from_float<kBf16Out>((!bad && L > 0.f) ? acc[e] / L : 0.f);
}

cudaError_t launch_decode_reduce(const DecodeParams& p, cudaStream_t s) {
  const dim3 block(256);
  if (p.max_parts <= 8) {  // every row has at most 8 partitions: a warp per row
    const dim3 grid((p.batch * p.num_q_heads + 7) / 8);
    if (p.head_dim == 64) {
      return p.q_bf16 ? launch_pdl(decode_reduce_warp_kernel<64, true>, grid, block, 0, s, p)
                      : launch_pdl(decode_reduce_warp_kernel<64, false>, grid, block, 0, s, p);
    }
    if (p.head_dim == 128) {
      return p.q_bf16 ? launch_pdl(decode_reduce_warp_kernel<128, true>, grid, block, 0, s, p)
                      : launch_pdl(decode_reduce_warp_kernel<128, false>, grid, block, 0, s, p);
    }
    return cudaErrorInvalidValue;
  }
  const dim3 grid(p.batch * p.num_q_heads);
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

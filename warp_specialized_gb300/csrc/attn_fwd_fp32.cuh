// attn_fwd_fp32.cuh - the fp32 forward pass on the FP32 CUDA-core pipes.
//
// Same online-softmax recurrence as the tensor-core kernel ("Warp
// specialization" concept card, section "Implementation sketch": running
// max, rescale of the old sum and output by exp(m_old - m_new), O / l and
// m + log l at the end), in exact fp32 arithmetic.  fp32 inputs do not go
// through tcgen05: its tf32 form reads only 10 mantissa bits of each
// operand (at d = 64 that alone moves the LSE by about 1e-3), and it does
// not accept an MN-major B operand, which V's [keys, d] layout needs.
//
// One warp per query row.  Keys are taken 32 at a time: lane l computes the
// score of key j0 + l, the warp reduces max and sum with shuffles, and each
// lane accumulates d/32 output columns from the 32 broadcast probabilities.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace wsattn {

constexpr int kFp32WarpsPerBlock = 8;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kFp32WarpsPerBlock * 32)
    attn_fwd_fp32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                         const float* __restrict__ v, float* __restrict__ o,
                         float* __restrict__ lse, int N, long long total_rows, float scale_log2) {
  constexpr int kPer = D / 32;
  __shared__ __align__(16) float sq[kFp32WarpsPerBlock][D];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kFp32WarpsPerBlock + warp;
  if (row >= total_rows) return;  // uniform per warp
  const long long bh = row / N;
  const int i = static_cast<int>(row - bh * N);
  const float* kh = k + bh * N * D;
  const float* vh = v + bh * N * D;
#pragma unroll
  for (int t = 0; t < kPer; ++t) sq[warp][lane + 32 * t] = q[row * D + lane + 32 * t];
  __syncwarp();

  float m = -INFINITY;  // running max, log2 units of the scaled scores
  float l = 0.f;
  float acc[kPer];
#pragma unroll
  for (int t = 0; t < kPer; ++t) acc[t] = 0.f;
  const int nkeys = CAUSAL ? i + 1 : N;
  for (int j0 = 0; j0 < nkeys; j0 += 32) {
    const int j = j0 + lane;
    float s = -INFINITY;
    if (j < nkeys) {
      const float4* kr = reinterpret_cast<const float4*>(kh + static_cast<long long>(j) * D);
      float dot = 0.f;
#pragma unroll 8
      for (int c = 0; c < D / 4; ++c) {
        const float4 kk = kr[c];
        dot = fmaf(sq[warp][4 * c + 0], kk.x, dot);
        dot = fmaf(sq[warp][4 * c + 1], kk.y, dot);
        dot = fmaf(sq[warp][4 * c + 2], kk.z, dot);
        dot = fmaf(sq[warp][4 * c + 3], kk.w, dot);
      }
      s = dot * scale_log2;
    }
    const float m_new = fmaxf(m, warp_max(s));  // finite: key 0 is always visible
    const float alpha = exp2f(m - m_new);        // 0 on the first chunk
    const float p = exp2f(s - m_new);            // 0 for masked keys
    l = alpha * l + warp_sum(p);
#pragma unroll
    for (int t = 0; t < kPer; ++t) acc[t] *= alpha;
    const int jn = min(32, nkeys - j0);
    for (int jj = 0; jj < jn; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
      const float* vr = vh + static_cast<long long>(j0 + jj) * D;
#pragma unroll
      for (int t = 0; t < kPer; ++t) acc[t] = fmaf(pj, vr[lane + 32 * t], acc[t]);
    }
    m = m_new;
  }
  const float inv = 1.0f / l;
#pragma unroll
  for (int t = 0; t < kPer; ++t) o[row * D + lane + 32 * t] = acc[t] * inv;
  if (lane == 0) lse[row] = (m + log2f(l)) * 0.6931471805599453f;
}

}  // namespace wsattn

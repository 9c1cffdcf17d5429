// attn_quant.cu - e4m3 block quantisation of Q or K, optionally after the
// 16 x 16 Walsh-Hadamard rotation ("Inside FlashAttention-3 &
// Warp-Specialized CUDA Kernels", section 5: Q' = Q H and K' = K H keep
// Q' K'^T = Q K^T while spreading outlier channels over 16 channels, and
// block scales replace one per-tensor scale).
//
// One CTA per (b, h, 128-row tile): each thread holds one row in registers,
// rotates each group of 16 channels with the fast butterfly (h = 1, 2, 4, 8:
// (a, b) -> (a + b, a - b) in fp32, then * 1/4), the block's absolute
// maximum is reduced over the CTA, scale = amax / 448 (IEEE division; 1 for
// an all-zero block) and code = e4m3(value / scale), round to nearest even,
// saturating.  HBM-bound: it reads the tensor once and writes one byte per
// element plus one scale per block.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn.h"
#include "attn_launch.h"

namespace wsattn {
namespace {

// Group g of 16 channels of a row held as raw 16-byte words, as fp32
template <typename T>
__device__ __forceinline__ void unpack16(const uint4* raw, int g, float (&v)[16]);

template <>
__device__ __forceinline__ void unpack16<float>(const uint4* raw, int g, float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 x = raw[4 * g + i];
    v[4 * i] = __uint_as_float(x.x);
    v[4 * i + 1] = __uint_as_float(x.y);
    v[4 * i + 2] = __uint_as_float(x.z);
    v[4 * i + 3] = __uint_as_float(x.w);
  }
}

template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4* raw, int g, float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 x = raw[2 * g + i];
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
      v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
}

template <>
__device__ __forceinline__ void unpack16<__half>(const uint4* raw, int g, float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 x = raw[2 * g + i];
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __half2 h = *reinterpret_cast<const __half2*>(&w[j]);
      const float2 f = __half22float2(h);
      v[8 * i + 2 * j] = f.x;
      v[8 * i + 2 * j + 1] = f.y;
    }
  }
}

// 16-point Walsh-Hadamard butterfly on v[0 .. 15], fp32, then * 1/4
__device__ __forceinline__ void wht16(float (&v)[16]) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = __fadd_rn(a, b);
        v[i + h] = __fsub_rn(a, b);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(v[i], 0.25f);
}

// One CTA per (b, h, 128-row tile), one thread per row.  The row stays in
// registers as the raw words it was loaded as (64 registers for a bf16 row
// of 128 channels), so that small CTAs keep several tiles of loads in
// flight on each SM; for 16-bit inputs the rotation of each group of 16
// channels is computed once for the block maximum and again, identically,
// for the codes (fp32 rows keep the rotated values in place).
template <typename T, int D>
__global__ void __launch_bounds__(128) quant_fp8_kernel(const T* __restrict__ x,
                                                       uint8_t* __restrict__ codes,
                                                       float* __restrict__ scales, int N, int nt,
                                                       int hadamard) {
  constexpr int kWords = D * static_cast<int>(sizeof(T)) / 16;  // 16-byte words per row
  __shared__ float red[4];
  const long long blk = blockIdx.x;
  const long long bh = blk / nt;
  const int tile = static_cast<int>(blk - bh * nt);
  const int row = tile * 128 + static_cast<int>(threadIdx.x);
  const bool valid = row < N;
  const size_t off = (static_cast<size_t>(bh) * N + (valid ? row : 0)) * D;
  uint4 raw[kWords];
  const uint4* src = reinterpret_cast<const uint4*>(x + off);
#pragma unroll
  for (int i = 0; i < kWords; ++i) raw[i] = valid ? src[i] : make_uint4(0u, 0u, 0u, 0u);
  float amax = 0.f;
  constexpr bool kInPlace = sizeof(T) == 4;  // fp32 rows keep the rotated values themselves
#pragma unroll
  for (int g = 0; g < D / 16; ++g) {
    float v[16];
    unpack16<T>(raw, g, v);
    if (hadamard) wht16(v);
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    if constexpr (kInPlace) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        raw[4 * g + i] = make_uint4(__float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
                                    __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3]));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  if (threadIdx.x == 0) scales[blk] = scale;
  if (!valid) return;
#pragma unroll
  for (int g = 0; g < D / 16; ++g) {
    float v[16];
    unpack16<T>(raw, g, v);
    if (hadamard && !kInPlace) wht16(v);
    uint32_t pk[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
          make_float2(__fdiv_rn(v[4 * i], scale), __fdiv_rn(v[4 * i + 1], scale)),
          __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
          make_float2(__fdiv_rn(v[4 * i + 2], scale), __fdiv_rn(v[4 * i + 3], scale)),
          __NV_SATFINITE, __NV_E4M3);
      pk[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    }
    *reinterpret_cast<uint4*>(codes + off + 16 * g) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
}

template <typename T, int D>
int launch_quant(const void* x, void* codes, float* scales, int B, int H, int N, int hadamard,
                 cudaStream_t stream) {
  const int nt = (N + 127) / 128;
  const long long blocks = static_cast<long long>(B) * H * nt;
  quant_fp8_kernel<T, D><<<static_cast<unsigned>(blocks), 128, 0, stream>>>(
      static_cast<const T*>(x), static_cast<uint8_t*>(codes), scales, N, nt, hadamard);
  return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

}  // namespace
}  // namespace wsattn

extern "C" int attn_quantize_fp8(const void* x, void* codes, float* scales, int B, int H, int N,
                                 int d, int dtype, int hadamard, struct CUstream_st* stream) {
  using namespace wsattn;
  if (!x || !codes || !scales || B < 1 || H < 1 || N < 1) return kErrInvalidArg;
  const long long bh = static_cast<long long>(B) * H;
  if (bh > (1LL << 24) || N > (1 << 24) || bh * ((N + 127) / 128) > 0x7FFFFFFFLL)
    return kErrInvalidArg;
  if (hadamard != 0 && hadamard != 1) return kErrInvalidArg;
  if (dtype < ATTN_FP32 || dtype > ATTN_FP8_E4M3) return kErrInvalidArg;
  if (dtype == ATTN_FP8_E4M3 || (d != 64 && d != 128)) return kErrUnsupported;
  if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(codes) % 16 ||
      reinterpret_cast<uintptr_t>(scales) % 4)
    return kErrMisaligned;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return kErrDevice;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (dtype) {
    case ATTN_FP32:
      return d == 64 ? launch_quant<float, 64>(x, codes, scales, B, H, N, hadamard, s)
                     : launch_quant<float, 128>(x, codes, scales, B, H, N, hadamard, s);
    case ATTN_FP16:
      return d == 64 ? launch_quant<__half, 64>(x, codes, scales, B, H, N, hadamard, s)
                     : launch_quant<__half, 128>(x, codes, scales, B, H, N, hadamard, s);
    default:
      return d == 64 ? launch_quant<__nv_bfloat16, 64>(x, codes, scales, B, H, N, hadamard, s)
                     : launch_quant<__nv_bfloat16, 128>(x, codes, scales, B, H, N, hadamard, s);
  }
}

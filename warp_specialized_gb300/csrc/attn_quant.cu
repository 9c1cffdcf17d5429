// attn_quant.cu - e4m3 block quantisation of Q or K, optionally after the
// 16 x 16 Walsh-Hadamard rotation ("Inside FlashAttention-3 &
// Warp-Specialized CUDA Kernels", section 5: Q' = Q H and K' = K H keep
// Q' K'^T = Q K^T while spreading outlier channels over 16 channels, and
// block scales replace one per-tensor scale).
//
// One CTA per (b, h, 128-row tile), reading the tile with coalesced 16-byte
// loads: each group of 16 channels is rotated with the fast butterfly
// (h = 1, 2, 4, 8: (a, b) -> (a + b, a - b) in fp32, then * 1/4), the
// block's absolute maximum is reduced over the CTA, scale = amax / 448 (IEEE
// division; 1 for an all-zero block) and code = e4m3(value / scale), the
// quotient correctly rounded in fp32, then to e4m3 nearest even,
// saturating.  HBM-bound: it reads the tensor once and writes one byte per
// element plus one scale per block.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "attn.h"
#include "attn_launch.h"
#include "ptx_sm103.cuh"

namespace wsattn {
namespace {

// A 16-byte chunk of a row (8 elements of a 16-bit type, 4 of fp32) as fp32
template <typename T>
__device__ __forceinline__ void unpack_chunk(const uint4 x, float (&v)[16 / sizeof(T)]);

template <>
__device__ __forceinline__ void unpack_chunk<float>(const uint4 x, float (&v)[4]) {
  v[0] = __uint_as_float(x.x);
  v[1] = __uint_as_float(x.y);
  v[2] = __uint_as_float(x.z);
  v[3] = __uint_as_float(x.w);
}

template <>
__device__ __forceinline__ void unpack_chunk<__nv_bfloat16>(const uint4 x, float (&v)[8]) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    v[2 * j] = __uint_as_float(w[j] << 16);
    v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}

template <>
__device__ __forceinline__ void unpack_chunk<__half>(const uint4 x, float (&v)[8]) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
    v[2 * j] = f.x;
    v[2 * j + 1] = f.y;
  }
}

// The 16-point Walsh-Hadamard butterfly on a group of 16 channels spread
// over 16 / E adjacent lanes, E channels each (v = this lane's E channels,
// lane bit h / E of the lane index says which part of the group it holds).
// Stages h = 1, 2, 4, 8 in that order, each (a, b) -> (a + b, a - b) in fp32
// for the pair (i, i + h): stages below E pair channels inside a lane, the
// others pair a lane with lane ^ (h / E), where the lane holding i keeps
// a + b and the lane holding i + h keeps a - b.  The final * 1/4 is left to
// the caller (it is exact, and folds into the block scale).
template <int E>
__device__ __forceinline__ void wht16_lanes(float (&v)[E]) {
  static_assert(E % 2 == 0, "pairs of channels per thread");
  // stage h = 1 pairs neighbours: scalar adds and subtracts
#pragma unroll
  for (int i = 0; i < E; i += 2) {
    const float a = v[i], b = v[i + 1];
    v[i] = __fadd_rn(a, b);
    v[i + 1] = __fsub_rn(a, b);
  }
  // stages h = 2 .. E/2 pair (i, i + 1) with (i + h, i + h + 1): two channels
  // per packed f32x2 add, and a - b as the packed fma b * (-1) + a, which
  // rounds once exactly as the scalar subtraction
  const uint64_t minus1 = f2_pack(-1.0f, -1.0f);
#pragma unroll
  for (int h = 2; h < E; h <<= 1) {
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      if ((i & h) == 0) {
        const uint64_t a = f2_pack(v[i], v[i + 1]), b = f2_pack(v[i + h], v[i + h + 1]);
        f2_unpack(f2_add(a, b), v[i], v[i + 1]);
        f2_unpack(f2_fma(b, minus1, a), v[i + h], v[i + h + 1]);
      }
    }
  }
  if constexpr (E >= 16) return;  // the whole group in this thread
  const int lane = static_cast<int>(threadIdx.x & 31);
#pragma unroll
  for (int h = E; h < 16; h <<= 1) {
    // other + v or other - v, rounded once: fma with a multiplier of +-1
    const float sgn = (lane & (h / E)) != 0 ? -1.0f : 1.0f;
    const uint64_t sgn2 = f2_pack(sgn, sgn);
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      const float o0 = __shfl_xor_sync(0xffffffffu, v[i], h / E);
      const float o1 = __shfl_xor_sync(0xffffffffu, v[i + 1], h / E);
      f2_unpack(f2_fma(sgn2, f2_pack(v[i], v[i + 1]), f2_pack(o0, o1)), v[i], v[i + 1]);
    }
  }
}

// e4m3 codes of one chunk's E values, stored as E bytes.
//
// With REFINE, value / b is correctly rounded from y = 1 / b correctly
// rounded by Markstein's refinement (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): with r = a - q b computed exactly by an fma,
// RN(q + r y) is the correctly rounded quotient whenever q is within one ulp
// of a / b.  q = RN(a y) can be off by up to 1.5 ulp, so one refinement
// first makes it faithful and a second rounds it correctly.  Valid while
// neither the quotient's ulp times b nor y leaves the normal range: the
// caller takes this path only for 2^-60 <= scale <= 2^60 (b = scale or
// 4 scale) with |value| <= 448 scale, where every quotient that can reach a
// nonzero e4m3 code (|a / b| > 2^-10) has an exact remainder, and smaller
// ones round to a zero code whatever their last bits; copysign keeps the
// sign of a zero quotient.  The quotients are formed two at a time with
// the packed f32x2 multiply and fma, each lane rounded exactly as the scalar
// instruction.
template <int E, bool REFINE>
__device__ __forceinline__ void store_codes(const float (&v)[E], float b, float y,
                                            uint8_t* dst) {
  float q[E];
  if constexpr (REFINE) {
    const uint64_t y2 = f2_pack(y, y);
    const uint64_t nb2 = f2_pack(-b, -b);
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      const uint64_t a2 = f2_pack(v[i], v[i + 1]);
      uint64_t q2 = f2_mul(a2, y2);
      uint64_t r2 = f2_fma(q2, nb2, a2);
      q2 = f2_fma(r2, y2, q2);
      r2 = f2_fma(q2, nb2, a2);
      q2 = f2_fma(r2, y2, q2);
      f2_unpack(q2, q[i], q[i + 1]);
      q[i] = copysignf(q[i], v[i]);
      q[i + 1] = copysignf(q[i + 1], v[i + 1]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) q[i] = __fdiv_rn(v[i], b);
  }
  uint32_t pk[E / 4];
#pragma unroll
  for (int j = 0; j < E / 4; ++j) {
    const __nv_fp8x2_storage_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(q[4 * j], q[4 * j + 1]), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi =
        __nv_cvt_float2_to_fp8x2(make_float2(q[4 * j + 2], q[4 * j + 3]), __NV_SATFINITE, __NV_E4M3);
    pk[j] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  if constexpr (E == 16)
    *reinterpret_cast<uint4*>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  else if constexpr (E == 8)
    *reinterpret_cast<uint2*>(dst) = make_uint2(pk[0], pk[1]);
  else
    *reinterpret_cast<uint32_t*>(dst) = pk[0];
}

// One CTA of NT threads per (b, h, 128-row tile).  The tile's rows are one
// contiguous span of memory, cut into 16-byte chunks; thread t takes chunks
// t, t + NT, t + 2 NT, ..., so that every warp-wide load and store covers
// one contiguous run.  NT is a multiple of the W chunks of a row, so a
// thread always holds the same E channels (chunk t mod W) of its rows, and
// the 16 / E chunks of a group of 16 channels sit in adjacent lanes.  The
// tile is read once and kept in registers (raw words, or the rotated fp32
// values) until the block maximum is known.
//
// With the rotation and 16-bit inputs a thread's chunk is 32 bytes (two
// adjacent 16-byte loads): a whole group of 16 channels, so that the
// butterfly runs without shuffles.
template <typename T, int D, int NT, bool HAD>
__global__ void __launch_bounds__(NT) quant_fp8_kernel(const T* __restrict__ x,
                                                      uint8_t* __restrict__ codes,
                                                      float* __restrict__ scales, int N,
                                                      int nt) {
  constexpr int kCV = HAD && sizeof(T) == 2 ? 2 : 1;    // 16-byte words per chunk
  constexpr int E = 16 * kCV / static_cast<int>(sizeof(T));  // channels per chunk
  constexpr int W = D / E;                              // chunks per row
  constexpr int C = 128 * W / NT;                       // chunks per thread
  constexpr int kRowStep = NT / W;                      // rows between a thread's chunks
  static_assert(NT % W == 0 && (128 * W) % NT == 0 && 16 % E == 0, "chunk layout");
  __shared__ float red[NT / 32];
  const long long blk = blockIdx.x;
  const long long bh = blk / nt;
  const int tile = static_cast<int>(blk - bh * nt);
  const int row0 = tile * 128 + static_cast<int>(threadIdx.x) / W;
  const size_t base = (static_cast<size_t>(bh) * N + static_cast<size_t>(tile) * 128) * D;
  const uint4* src = reinterpret_cast<const uint4*>(x + base) + threadIdx.x * kCV;
  uint4 raw[C][kCV];
#pragma unroll
  for (int k = 0; k < C; ++k)
#pragma unroll
    for (int u = 0; u < kCV; ++u)
      raw[k][u] = row0 + k * kRowStep < N ? src[k * NT * kCV + u] : make_uint4(0u, 0u, 0u, 0u);
  // the chunk's E values as fp32
  constexpr int kPerWord = 16 / static_cast<int>(sizeof(T));
  auto unpack = [&](int k, float (&v)[E]) {
#pragma unroll
    for (int u = 0; u < kCV; ++u) {
      float w[kPerWord];
      unpack_chunk<T>(raw[k][u], w);
#pragma unroll
      for (int i = 0; i < kPerWord; ++i) v[u * kPerWord + i] = w[i];
    }
  };
  // With 16-bit inputs the rotation's exact * 1/4 moves into the divisor:
  // value / scale = w / (4 scale) for value = w / 4, both exact, since w is
  // a multiple of the type's smallest step and stays far from fp32's
  // subnormal floor.  fp32 inputs keep the multiply.
  constexpr bool kFold = HAD && sizeof(T) == 2;
  float rot[HAD ? C : 1][E];
  float amax = 0.f;
  if constexpr (!HAD && sizeof(T) == 2) {
    // |x| of two 16-bit values per word is the word with its sign bits
    // cleared, and magnitudes order like their bit patterns: the block
    // maximum is an unsigned 16-bit maximum, two lanes per instruction
    uint32_t m2 = 0u;
#pragma unroll
    for (int k = 0; k < C; ++k) {
      m2 = __vmaxu2(m2, raw[k][0].x & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, raw[k][0].y & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, raw[k][0].z & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, raw[k][0].w & 0x7FFF7FFFu);
    }
    const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    if constexpr (std::is_same<T, __half>::value)
      amax = __half2float(__ushort_as_half(static_cast<unsigned short>(m)));
    else
      amax = __uint_as_float(m << 16);
  } else {
#pragma unroll
    for (int k = 0; k < C; ++k) {
      float v[E];
      unpack(k, v);
      if constexpr (HAD) {
        wht16_lanes<E>(v);
#pragma unroll
        for (int i = 0; i < E; ++i) rot[k][i] = kFold ? v[i] : __fmul_rn(v[i], 0.25f);
      }
#pragma unroll
      for (int i = 0; i < E; ++i) amax = fmaxf(amax, fabsf(HAD ? rot[k][i] : v[i]));
    }
    if constexpr (kFold) amax *= 0.25f;  // the rotated values' maximum
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) amax = fmaxf(amax, red[w]);
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  const bool refine = scale >= 0x1p-60f && scale <= 0x1p60f;  // same for the whole block
  if (threadIdx.x == 0) scales[blk] = scale;
  // the divisor the codes are formed with (4 scale when the rotation's
  // * 1/4 is folded in) and its correctly rounded reciprocal
  const float div = kFold ? scale * 4.0f : scale;
  const float y = __frcp_rn(div);
  uint8_t* dst = codes + base + static_cast<size_t>(threadIdx.x) * E;
  // one branch for the block, so that the per-element code has none
  auto store_all = [&](auto refine_tag) {
    constexpr bool kRefine = decltype(refine_tag)::value;
#pragma unroll
    for (int k = 0; k < C; ++k) {
      if (row0 + k * kRowStep >= N) break;
      float v[E];
      if constexpr (HAD) {
#pragma unroll
        for (int i = 0; i < E; ++i) v[i] = rot[k][i];
      } else {
        unpack(k, v);
      }
      store_codes<E, kRefine>(v, div, y, dst + static_cast<size_t>(k) * NT * E);
    }
  };
  if (refine)
    store_all(std::true_type{});
  else
    store_all(std::false_type{});
}

template <typename T, int D>
int launch_quant(const void* x, void* codes, float* scales, int B, int H, int N, int hadamard,
                 cudaStream_t stream) {
  // Four 16-byte chunks per thread for 16-bit rows and eight for fp32 rows
  // (capped at 512 threads) measured fastest: bf16 d = 128 takes 512
  // threads, d = 64 takes 256.  (With the rotation a 16-bit thread holds the
  // same bytes as two 32-byte chunks.)
  constexpr int kW = D * static_cast<int>(sizeof(T)) / 16;
  constexpr int kPerThread = sizeof(T) == 4 ? 8 : 4;
  constexpr int kNT = 128 * kW / kPerThread > 512 ? 512 : 128 * kW / kPerThread;
  const int nt = (N + 127) / 128;
  const long long blocks = static_cast<long long>(B) * H * nt;
  const auto* xp = static_cast<const T*>(x);
  auto* cp = static_cast<uint8_t*>(codes);
  if (hadamard)
    quant_fp8_kernel<T, D, kNT, true><<<static_cast<unsigned>(blocks), kNT, 0, stream>>>(
        xp, cp, scales, N, nt);
  else
    quant_fp8_kernel<T, D, kNT, false><<<static_cast<unsigned>(blocks), kNT, 0, stream>>>(
        xp, cp, scales, N, nt);
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
  if (!on_device(x, dev) || !on_device(codes, dev) || !on_device(scales, dev))
    return kErrInvalidArg;
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

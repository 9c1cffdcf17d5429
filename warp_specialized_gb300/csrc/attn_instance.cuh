// attn_instance.cuh - host launch of one kernel instance (element type,
// head dim, mask); included by the inst_*.cu units only.
#pragma once

#include <atomic>

#include "attn_fwd_kernel.cuh"
#include "attn_launch.h"

namespace wsattn {

inline CUtensorMapDataType tensor_map_type(int dt) {
  switch (dt) {
    case 0: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    case 1: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    case 2: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    default: return CU_TENSOR_MAP_DATA_TYPE_UINT8;
  }
}

// 3-D view (d, N, B*H) of a dense [B, H, N, d] tensor; the box is one
// 128-byte swizzle row wide and box_rows high.  Rows past N inside a head
// read as zeros (out-of-bounds fill), so a ragged last tile never sees the
// next head.
template <int DT, int D>
inline bool encode_map(const LaunchArgs& a, const void* ptr, int box_rows, CUtensorMap* map) {
  using C = Cfg<DT, D>;
  const cuuint64_t es = static_cast<cuuint64_t>(C::kEsize);
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(a.N),
                        static_cast<cuuint64_t>(a.B) * static_cast<cuuint64_t>(a.H)};
  cuuint64_t strides[2] = {D * es, static_cast<cuuint64_t>(a.N) * D * es};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(C::kBoxInner), static_cast<cuuint32_t>(box_rows), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = a.encode(map, tensor_map_type(DT), 3, const_cast<void*>(ptr), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The output as the same 3-D view, in its own type (fp16 for fp16 inputs,
// bf16 otherwise), with boxes of 128 rows x 64 columns: the stores of the
// epilogue.  Rows past N are never written.
template <int DT, int D>
inline bool encode_out_map(const LaunchArgs& a, CUtensorMap* map) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(a.N),
                        static_cast<cuuint64_t>(a.B) * static_cast<cuuint64_t>(a.H)};
  cuuint64_t strides[2] = {D * 2ull, static_cast<cuuint64_t>(a.N) * D * 2ull};
  cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(kBlock), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = a.encode(map, DT == 1 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        3, a.o, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int DT, int D, bool CAUSAL>
int launch_instance(const LaunchArgs& a) {
  using C = Cfg<DT, D>;
  auto kern = attn_fwd_kernel<DT, D, CAUSAL>;
  // Per device, once: opt in to the shared memory size, and refuse to run
  // unless the kernel is launched with exactly 128 registers per thread
  // (the warpgroups' setmaxnreg split, 88 + 168 + 168 + 80, draws on that
  // pool and could never be satisfied by a smaller one) and one CTA fits
  // on an SM.
  static std::atomic<int> ready[kMaxDevices];
  if (a.device < 0 || a.device >= kMaxDevices) return kErrDevice;
  int st = ready[a.device].load(std::memory_order_acquire);
  if (st == 0) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) {
      cudaGetLastError();
      return kErrCuda;
    }
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess) {
      cudaGetLastError();
      return kErrCuda;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, C::kSmemBytes) !=
        cudaSuccess) {
      cudaGetLastError();
      return kErrCuda;
    }
    st = (fa.numRegs == 128 && fa.maxThreadsPerBlock >= kThreads && per_sm >= 1) ? 1 : 2;
    ready[a.device].store(st, std::memory_order_release);
  }
  if (st != 1) return kErrUnsupported;

  CUtensorMap mq, mk, mv, mo;
  if (!encode_map<DT, D>(a, a.q, kBlock, &mq) || !encode_map<DT, D>(a, a.k, kBlock, &mk) ||
      !encode_map<DT, D>(a, a.v, kBlock, &mv) || !encode_out_map<DT, D>(a, &mo))
    return kErrCuda;

  AttnParams p;
  p.o = a.o;
  p.lse = a.lse;
  p.N = a.N;
  p.BH = a.B * a.H;
  p.n_qt = (a.N + kBlock - 1) / kBlock;
  p.nkv = p.n_qt;
  p.n_pairs = (p.n_qt + C::kNQT - 1) / C::kNQT;
  p.n_items = p.BH * p.n_pairs;
  p.scale_log2 = a.scale_log2;
  p.out_scale = a.out_scale;
  p.q_block_scale = a.q_block_scale;
  p.k_block_scale = a.k_block_scale;
  p.timeout_ns = a.timeout_ns;
  p.status = a.status;
  p.where = a.where;
  // persistent grid: one CTA per SM (the shared-memory budget allows no
  // second), never more CTAs than work items
  const int grid = p.n_items < a.num_sms ? p.n_items : a.num_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = a.stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  if (cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mo, p) != cudaSuccess) {
    cudaGetLastError();
    return kErrCuda;
  }
  return kOk;
}

template <int DT, int D>
int launch_mask(const LaunchArgs& a) {
  return a.causal ? launch_instance<DT, D, true>(a) : launch_instance<DT, D, false>(a);
}

}  // namespace wsattn

// attn_instance.cuh - host launch of one kernel instance (element type,
// head dim, mask); included by the inst_*.cu units only.
#pragma once

#include <atomic>

#include "attn_fwd_kernel.cuh"
#include "attn_fwd_tail.cuh"
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

// Per device, once: opt in to the kernel's shared memory size, and refuse
// to run unless it is launched with exactly 128 registers per thread (the
// warpgroups' setmaxnreg split draws on that pool and could never be
// satisfied by a smaller one) and one CTA fits on an SM.  Returns a status.
template <typename K>
inline int prepare_fwd_kernel(K kern, int smem_bytes, int device, std::atomic<int>* ready) {
  int st = ready[device].load(std::memory_order_acquire);
  if (st == 0) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) {
      cudaGetLastError();
      return kErrCuda;
    }
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
        cudaSuccess) {
      cudaGetLastError();
      return kErrCuda;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem_bytes) !=
        cudaSuccess) {
      cudaGetLastError();
      return kErrCuda;
    }
    st = (fa.numRegs == 128 && fa.maxThreadsPerBlock >= kThreads && per_sm >= 1) ? 1 : 2;
    ready[device].store(st, std::memory_order_release);
  }
  return st == 1 ? kOk : kErrUnsupported;
}

template <int DT, int D, bool CAUSAL, int XF = 0>
int launch_instance(const LaunchArgs& a) {
  using C = Cfg<DT, D>;
  auto kern = attn_fwd_kernel<DT, D, CAUSAL, XF>;
  // the split tail runs the default (MUFU) exponentials only
  constexpr bool kTail = !C::kQTmem && XF == 0;
  static std::atomic<int> ready[kMaxDevices], ready_tail[kMaxDevices];
  if (a.device < 0 || a.device >= kMaxDevices) return kErrDevice;
  int rc = prepare_fwd_kernel(kern, C::kSmemBytes, a.device, ready);
  if (rc != kOk) return rc;

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
  p.tail_start = p.n_items;
  p.tail_items = 0;
  p.tail_ramp = 0;
  p.tail_units = 0;
  p.flags = nullptr;
  p.part = nullptr;

  // With a workspace, the main kernel runs whole rounds of num_sms items
  // and the tail launch the rest; without one, one launch runs all items.
  // (d = 256 keeps its Q in Tensor Memory, a layout the tail kernel does not
  // have: it always runs whole items.)
  const TailPlan plan =
      (a.workspace && kTail)
          ? plan_tail(p.BH, p.n_pairs, p.nkv, C::kNQT, CAUSAL, a.num_sms,
                      tail_max_pieces(D, C::kEsize))
          : TailPlan{};
  const int tail = plan.items;
  const int tail_grid = plan.grid;
  if constexpr (kTail) {
  if (tail > 0) {
    rc = prepare_fwd_kernel(attn_fwd_tail_kernel<DT, D, CAUSAL>, TailCfg<DT, D>::kSmemBytes,
                            a.device, ready_tail);
    if (rc != kOk) return rc;
    if (a.workspace_bytes < fwd_workspace_bytes(a.num_sms, D, C::kNQT)) return kErrInvalidArg;
    p.tail_start = plan.start;
    p.tail_items = tail;
    p.tail_units = static_cast<int>(plan.units);
    p.tail_ramp = tail_ramp(plan, plan.start > 0);
    p.flags = static_cast<unsigned int*>(a.workspace);
    p.part = reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) +
                                      fwd_flags_bytes(a.num_sms));
    p.n_items = p.tail_start;
    // the main launch clears the flags itself; without one, a memset does
    if (p.n_items == 0 &&
        cudaMemsetAsync(p.flags, 0, static_cast<size_t>(tail) * 2 * sizeof(unsigned int),
                        a.stream) != cudaSuccess) {
      cudaGetLastError();
      return kErrCuda;
    }
  }
  }
  // persistent grid: one CTA per SM (the shared-memory budget allows no
  // second), never more CTAs than work items
  if (p.n_items > 0) {
    const int grid = p.n_items < a.num_sms ? p.n_items : a.num_sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = a.stream;
    if (cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mo, p) != cudaSuccess) {
      cudaGetLastError();
      return kErrCuda;
    }
  }
  if constexpr (kTail) {
  if (tail > 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tail_grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = TailCfg<DT, D>::kSmemBytes;
    cfg.stream = a.stream;
    // behind a main launch, the tail CTAs take the SMs its CTAs leave
    // without waiting for the last of them (programmatic dependent launch;
    // the tail kernel waits for the main grid before it reads the flags)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (p.n_items > 0) {
      cfg.attrs = attr;
      cfg.numAttrs = 1;
    }
    if (cudaLaunchKernelEx(&cfg, attn_fwd_tail_kernel<DT, D, CAUSAL>, mq, mk, mv, mo, p) !=
        cudaSuccess) {
      cudaGetLastError();
      return kErrCuda;
    }
  }
  }
  (void)tail_grid;
  return kOk;
}

template <int DT, int D>
int launch_mask(const LaunchArgs& a) {
  return a.causal ? launch_instance<DT, D, true>(a) : launch_instance<DT, D, false>(a);
}

// The instances of ATTN_OPT_EXP2_FMA: 4 exponentials of every 32 on the FMA
// pipe.
template <int DT, int D>
int launch_mask_xf(const LaunchArgs& a) {
  return a.causal ? launch_instance<DT, D, true, 4>(a) : launch_instance<DT, D, false, 4>(a);
}

}  // namespace wsattn

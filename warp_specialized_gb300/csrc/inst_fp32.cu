// fp32 instances: d = 64, 128, on the FP32 CUDA-core kernel
#include "attn_fwd_fp32.cuh"
#include "attn_launch.h"

namespace wsattn {
namespace {

template <int D, bool CAUSAL>
int launch_fp32_instance(const LaunchArgs& a) {
  const long long rows = static_cast<long long>(a.B) * a.H * a.N;
  const long long blocks = (rows + kFp32WarpsPerBlock - 1) / kFp32WarpsPerBlock;
  attn_fwd_fp32_kernel<D, CAUSAL><<<static_cast<unsigned>(blocks), kFp32WarpsPerBlock * 32, 0,
                                    a.stream>>>(
      static_cast<const float*>(a.q), static_cast<const float*>(a.k),
      static_cast<const float*>(a.v), static_cast<float*>(a.o), a.lse, a.N, rows, a.scale_log2);
  return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

template <int D>
int launch_fp32_mask(const LaunchArgs& a) {
  return a.causal ? launch_fp32_instance<D, true>(a) : launch_fp32_instance<D, false>(a);
}

}  // namespace

int launch_fp32(const LaunchArgs& a) {
  switch (a.d) {
    case 64: return launch_fp32_mask<64>(a);
    case 128: return launch_fp32_mask<128>(a);
    default: return kErrUnsupported;
  }
}

}  // namespace wsattn

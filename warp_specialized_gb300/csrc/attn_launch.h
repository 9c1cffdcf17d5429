// attn_launch.h - host-side glue between the C ABI (attn_api.cu) and the
// per-dtype kernel instantiation units (inst_*.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace wsattn {

// cuTensorMapEncodeTiled, resolved at run time through the runtime's
// driver entry-point query so that the library does not link libcuda.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct LaunchArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, H, N, d;
  int causal;
  float scale_log2;   // softmax scale (with q/k descales) times log2(e)
  float out_scale;    // v descale
  const float* q_block_scale;  // e4m3 block scales (null: per-tensor)
  const float* k_block_scale;
  cudaStream_t stream;
  int device;
  int num_sms;
  unsigned long long timeout_ns;
  unsigned int* status;  // device watchdog words
  unsigned int* where;
  EncodeTiledFn encode;
};

// status codes (identical to attn.h)
enum : int {
  kOk = 0,
  kErrInvalidArg = 1,
  kErrUnsupported = 2,
  kErrMisaligned = 3,
  kErrDevice = 4,
  kErrCuda = 5,
  kErrTimeout = 6,
};

constexpr int kMaxDevices = 64;

// True when p lies in device memory of device `dev`.  Every pointer the
// kernels read or write through (TMA tensor maps included) must: host
// memory, managed memory and another GPU's memory are refused.
inline bool on_device(const void* p, int dev) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice && at.device == dev;
}

struct BwdLaunchArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  void* workspace;
  int B, H, N, d;
  int causal;
  int dtype;
  float scale;
  cudaStream_t stream;
  int device;
  int num_sms;
  unsigned long long timeout_ns;
  unsigned int* status;
  unsigned int* where;
  EncodeTiledFn encode;
};

// Workspace of the backward pass: (LSE * log2 e, dO . O) per row, rows
// padded to whole 128-row tiles per head.
inline unsigned long long bwd_workspace_bytes(int B, int H, int N) {
  const unsigned long long np = (static_cast<unsigned long long>(N) + 127ull) / 128ull * 128ull;
  return static_cast<unsigned long long>(B) * static_cast<unsigned long long>(H) * np * 8ull;
}

// Backward pass (fp16 / bf16, d = 64 or 128); returns a status code.
int launch_bwd(const BwdLaunchArgs& a);

// One entry per element type; each returns a status code.
int launch_fp32(const LaunchArgs& a);
int launch_fp16(const LaunchArgs& a);
int launch_bf16(const LaunchArgs& a);
int launch_fp8(const LaunchArgs& a);

}  // namespace wsattn

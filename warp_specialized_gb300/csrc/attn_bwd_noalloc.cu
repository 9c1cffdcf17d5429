// attn_bwd_noalloc.cu - the backward pass for callers that cannot allocate
// device memory.
//
// attn_bwd needs a small device workspace (8 bytes per query row).  Some
// callers cannot provide one at call time: a host program that has handed
// all device memory to its own pool and has no cudaMalloc left to make, a
// plugin whose host framework owns every allocation, or a training step that
// must not risk an allocation's latency or failure halfway through.  This
// entry point uses a workspace that lives inside the library instead: one
// fixed-size array in device global memory, created when the library is
// loaded on a device and held until the process exits.  It allocates
// nothing and frees nothing.
#include <cuda_runtime.h>

#include <mutex>

#include "attn.h"
#include "attn_launch.h"

namespace {

// Largest workspace the array can serve: 8 MiB, i.e. up to 1,048,576 query
// rows after each head is rounded up to whole 128-row tiles
// (B * H * ceil(N / 128) * 128 <= 2^20).
constexpr unsigned long long kScratchBytes = 8ull << 20;

// The library-owned workspace.  In host code this name is only a stand-in
// for the device array, never a device address: the address is looked up
// with cudaGetSymbolAddress for each device (below) and only that is passed
// to the kernels.
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[wsattn::kMaxDevices] = {};

// Device address of the array on the current device, looked up on the first
// call for that device (with that device current) and cached.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_DEVICE;
  }
  if (dev < 0 || dev >= wsattn::kMaxDevices) return ATTN_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                int B, int H, int N, int d, float scale, int causal, int dtype,
                                struct CUstream_st* stream) {
  if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
  if (wsattn::bwd_workspace_bytes(B, H, N) > kScratchBytes) return ATTN_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != ATTN_OK) return rc;
  // The first kernel of attn_bwd rewrites every workspace entry the later
  // kernels read, so whatever an earlier call left in the array is harmless.
  return attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, scratch, kScratchBytes, B, H, N, d, scale,
                  causal, dtype, stream);
}

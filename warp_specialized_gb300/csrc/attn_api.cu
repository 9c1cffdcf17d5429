// attn_api.cu - the C ABI declared in include/attn.h: argument checks,
// device checks, dispatch to the kernel instances, and the watchdog word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <initializer_list>

#include "attn.h"
#include "attn_fwd_kernel.cuh"
#include "attn_launch.h"

namespace wsattn {
namespace {

// The watchdog words of the current device: the first error any kernel of
// this library recorded, and which wait it was.
__device__ unsigned int g_status;
__device__ unsigned int g_where;

constexpr unsigned long long kTimeoutNs = 2000000000ull;  // 2 s per wait

struct DeviceInfo {
  std::atomic<int> state{0};  // 0 unknown, 1 usable, 2 not sm_103 / error
  int num_sms = 0;
  unsigned int* status = nullptr;
  unsigned int* where = nullptr;
};
DeviceInfo g_dev[kMaxDevices];

EncodeTiledFn g_encode = nullptr;
std::atomic<int> g_encode_state{0};

bool resolve_encode() {
  int st = g_encode_state.load(std::memory_order_acquire);
  if (st == 0) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e == cudaSuccess && q == cudaDriverEntryPointSuccess && fn) {
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
      st = 1;
    } else {
      cudaGetLastError();
      st = 2;
    }
    g_encode_state.store(st, std::memory_order_release);
  }
  return st == 1;
}

// Current device, checked once: compute capability 10.3, SM count, and the
// device addresses of the watchdog words.  Returns a status code.
int current_device(int* dev_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return kErrDevice;
  }
  if (dev < 0 || dev >= kMaxDevices) return kErrDevice;
  DeviceInfo& di = g_dev[dev];
  int st = di.state.load(std::memory_order_acquire);
  if (st == 0) {
    int major = 0, minor = 0, sms = 0;
    bool ok = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
              cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
              cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
    ok = ok && major == 10 && minor == 3 && sms > 0;
    void* ps = nullptr;
    void* pw = nullptr;
    if (ok)
      ok = cudaGetSymbolAddress(&ps, g_status) == cudaSuccess &&
           cudaGetSymbolAddress(&pw, g_where) == cudaSuccess;
    if (!ok) cudaGetLastError();
    di.num_sms = sms;
    di.status = static_cast<unsigned int*>(ps);
    di.where = static_cast<unsigned int*>(pw);
    st = ok ? 1 : 2;
    di.state.store(st, std::memory_order_release);
  }
  if (st != 1) return kErrDevice;
  *dev_out = dev;
  return kOk;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool finite_positive(float x) { return std::isfinite(x) && x > 0.0f; }

int check_args(const void* q, const void* k, const void* v, const void* o, const float* lse,
               int B, int H, int N, int d, float scale, int causal, int dtype) {
  if (!q || !k || !v || !o || !lse) return kErrInvalidArg;
  if (B < 1 || H < 1 || N < 1 || d < 1) return kErrInvalidArg;
  const long long bh = static_cast<long long>(B) * H;
  if (bh > (1LL << 24) || N > (1 << 24) || bh * N > INT_MAX) return kErrInvalidArg;
  if (!finite_positive(scale)) return kErrInvalidArg;
  if (causal != 0 && causal != 1) return kErrInvalidArg;
  if (dtype < ATTN_FP32 || dtype > ATTN_FP8_E4M3) return kErrInvalidArg;
  bool d_ok = false;
  switch (dtype) {
    case ATTN_FP32: d_ok = (d == 64 || d == 128); break;
    case ATTN_FP16:
    case ATTN_BF16: d_ok = (d == 64 || d == 128 || d == 256); break;
    case ATTN_FP8_E4M3: d_ok = (d == 128); break;
  }
  if (!d_ok) return kErrUnsupported;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return kErrMisaligned;
  return kOk;
}

// Workspace bytes of the forward's tail launch for (d, dtype) on a device
// with num_sms SMs; 0 where no tail launch exists (exact fp32 path).
unsigned long long fwd_workspace_size(int num_sms, int d, int dtype) {
  if (dtype != ATTN_FP16 && dtype != ATTN_BF16 && dtype != ATTN_FP8_E4M3) return 0ull;
  if (d == 256) return 0ull;  // the d = 256 kernel runs whole items only
  return fwd_workspace_bytes(num_sms, d, fwd_nqt(d, dtype == ATTN_FP8_E4M3 ? 1 : 2));
}

int run(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
        int d, float scale, int causal, int dtype, float q_descale, float k_descale,
        float v_descale, cudaStream_t stream, const float* q_block_scale = nullptr,
        const float* k_block_scale = nullptr, void* workspace = nullptr,
        unsigned long long workspace_bytes = 0ull, unsigned int opts = 0u) {
  int rc = check_args(q, k, v, o, lse, B, H, N, d, scale, causal, dtype);
  if (rc != kOk) return rc;
  if (opts & ~static_cast<unsigned int>(ATTN_OPT_EXP2_FMA)) return kErrInvalidArg;
  if (workspace && !aligned(workspace, 256)) return kErrMisaligned;
  if (!finite_positive(q_descale) || !finite_positive(k_descale) || !finite_positive(v_descale))
    return kErrInvalidArg;
  const double sl2 = static_cast<double>(scale) * q_descale * k_descale * 1.4426950408889634;
  if (!std::isfinite(sl2) || !(sl2 > 0.0) || sl2 > 3.0e38) return kErrInvalidArg;
  int dev = -1;
  rc = current_device(&dev);
  if (rc != kOk) return rc;
  if (!on_device(q, dev) || !on_device(k, dev) || !on_device(v, dev) || !on_device(o, dev) ||
      !on_device(lse, dev))
    return kErrInvalidArg;
  if (q_block_scale && (!on_device(q_block_scale, dev) || !on_device(k_block_scale, dev)))
    return kErrInvalidArg;
  if (workspace && (!on_device(workspace, dev) ||
                    workspace_bytes < fwd_workspace_size(g_dev[dev].num_sms, d, dtype)))
    return kErrInvalidArg;
  if (!resolve_encode()) return kErrCuda;

  LaunchArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.N = N;
  a.d = d;
  a.causal = causal;
  a.scale_log2 = static_cast<float>(sl2);
  a.out_scale = v_descale;
  a.q_block_scale = q_block_scale;
  a.k_block_scale = k_block_scale;
  a.stream = stream;
  a.device = dev;
  a.num_sms = g_dev[dev].num_sms;
  a.timeout_ns = kTimeoutNs;
  a.status = g_dev[dev].status;
  a.where = g_dev[dev].where;
  a.encode = g_encode;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  if (opts & ATTN_OPT_EXP2_FMA) return workspace ? kErrInvalidArg : launch_exp2_fma(a, dtype);
  switch (dtype) {
    case ATTN_FP32: return launch_fp32(a);
    case ATTN_FP16: return launch_fp16(a);
    case ATTN_BF16: return launch_bf16(a);
    default: return launch_fp8(a);
  }
}

int run_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
            const float* lse, void* dq, void* dk, void* dv, void* workspace,
            unsigned long long workspace_bytes, int B, int H, int N, int d, float scale,
            int causal, int dtype, cudaStream_t stream) {
  if (!o || !dout || !dq || !dk || !dv || !workspace) return kErrInvalidArg;
  if (dtype != ATTN_FP16 && dtype != ATTN_BF16) {
    if (dtype < ATTN_FP32 || dtype > ATTN_FP8_E4M3) return kErrInvalidArg;
    return kErrUnsupported;
  }
  // the forward's checks cover q, k, v, lse, sizes, scale, causal, dtype
  int rc = check_args(q, k, v, dq, lse, B, H, N, d, scale, causal, dtype);
  if (rc != kOk) return rc;
  if (d != 64 && d != 128) return kErrUnsupported;
  if (!aligned(o, 16) || !aligned(dout, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(workspace, 16))
    return kErrMisaligned;
  if (workspace_bytes < bwd_workspace_bytes(B, H, N)) return kErrInvalidArg;
  int dev = -1;
  rc = current_device(&dev);
  if (rc != kOk) return rc;
  for (const void* ptr : {q, k, v, o, dout, static_cast<const void*>(lse),
                          static_cast<const void*>(dq), static_cast<const void*>(dk),
                          static_cast<const void*>(dv), static_cast<const void*>(workspace)})
    if (!on_device(ptr, dev)) return kErrInvalidArg;
  if (!resolve_encode()) return kErrCuda;
  BwdLaunchArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.workspace = workspace;
  a.B = B;
  a.H = H;
  a.N = N;
  a.d = d;
  a.causal = causal;
  a.dtype = dtype;
  a.scale = scale;
  a.stream = stream;
  a.device = dev;
  a.num_sms = g_dev[dev].num_sms;
  a.timeout_ns = kTimeoutNs;
  a.status = g_dev[dev].status;
  a.where = g_dev[dev].where;
  a.encode = g_encode;
  return launch_bwd(a);
}

// Waits on an mbarrier that nobody arrives on, so the bounded wait runs out.
__global__ void watchdog_selftest_kernel(unsigned long long limit_ns, unsigned int* status,
                                         unsigned int* where) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtx wc{&abort_flag, limit_ns, status, where};
    wait_bar(smem_u32(&bar), 0u, wc, 0x7f);
  }
}

int read_and_clear_status(int dev) {
  unsigned int h = 0, zero = 0;
  if (cudaMemcpy(&h, g_dev[dev].status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(g_dev[dev].status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(g_dev[dev].where, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return kErrCuda;
  }
  return h == 0 ? kOk : static_cast<int>(h);
}

}  // namespace
}  // namespace wsattn

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
             int d, float scale, int causal, int dtype, struct CUstream_st* stream) {
  return wsattn::run(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, 1.0f, 1.0f, 1.0f,
                     reinterpret_cast<cudaStream_t>(stream));
}

int attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, float q_descale, float k_descale,
                 float v_descale, struct CUstream_st* stream) {
  return wsattn::run(q, k, v, o, lse, B, H, N, d, scale, causal, ATTN_FP8_E4M3, q_descale,
                     k_descale, v_descale, reinterpret_cast<cudaStream_t>(stream));
}

int attn_fwd_opt(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, int dtype, unsigned int opts,
                 struct CUstream_st* stream) {
  return wsattn::run(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, 1.0f, 1.0f, 1.0f,
                     reinterpret_cast<cudaStream_t>(stream), nullptr, nullptr, nullptr, 0ull,
                     opts);
}

int attn_fwd_fp8_opt(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int N, int d, float scale, int causal, float q_descale,
                     float k_descale, float v_descale, unsigned int opts,
                     struct CUstream_st* stream) {
  return wsattn::run(q, k, v, o, lse, B, H, N, d, scale, causal, ATTN_FP8_E4M3, q_descale,
                     k_descale, v_descale, reinterpret_cast<cudaStream_t>(stream), nullptr,
                     nullptr, nullptr, 0ull, opts);
}

unsigned long long attn_fwd_workspace_size(int d, int dtype) {
  int dev = -1;
  if (wsattn::current_device(&dev) != wsattn::kOk) return 0ull;
  if (d != 64 && d != 128 && d != 256) return 0ull;
  return wsattn::fwd_workspace_size(wsattn::g_dev[dev].num_sms, d, dtype);
}

int attn_fwd_split_advised(int B, int H, int N, int d, int causal, int dtype) {
  if (B < 1 || H < 1 || N < 1 || (causal != 0 && causal != 1)) return 0;
  if (dtype != ATTN_FP16 && dtype != ATTN_BF16 && dtype != ATTN_FP8_E4M3) return 0;
  if (d != 64 && d != 128) return 0;  // d = 256 runs whole items only
  const long long bh = static_cast<long long>(B) * H;
  if (bh > (1LL << 24) || N > (1 << 24) || bh * N > INT_MAX) return 0;
  int dev = -1;
  if (wsattn::current_device(&dev) != wsattn::kOk) return 0;
  const int esize = dtype == ATTN_FP8_E4M3 ? 1 : 2;
  const int nqt = wsattn::fwd_nqt(d, esize);
  const int n_qt = (N + 127) / 128;
  const int n_pairs = (n_qt + nqt - 1) / nqt;
  const wsattn::TailPlan t =
      wsattn::plan_tail(static_cast<int>(bh), n_pairs, n_qt, nqt, causal != 0,
                        wsattn::g_dev[dev].num_sms, wsattn::tail_max_pieces(d, esize));
  return wsattn::tail_split_pays(t) ? 1 : 0;
}

int attn_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int N, int d, float scale, int causal, int dtype, void* workspace,
                unsigned long long workspace_bytes, struct CUstream_st* stream) {
  if (!workspace) return wsattn::kErrInvalidArg;
  return wsattn::run(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, 1.0f, 1.0f, 1.0f,
                     reinterpret_cast<cudaStream_t>(stream), nullptr, nullptr, workspace,
                     workspace_bytes);
}

int attn_fwd_fp8_ws(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                    int H, int N, int d, float scale, int causal, float q_descale,
                    float k_descale, float v_descale, void* workspace,
                    unsigned long long workspace_bytes, struct CUstream_st* stream) {
  if (!workspace) return wsattn::kErrInvalidArg;
  return wsattn::run(q, k, v, o, lse, B, H, N, d, scale, causal, ATTN_FP8_E4M3, q_descale,
                     k_descale, v_descale, reinterpret_cast<cudaStream_t>(stream), nullptr,
                     nullptr, workspace, workspace_bytes);
}

unsigned long long attn_bwd_workspace_size(int B, int H, int N) {
  if (B < 1 || H < 1 || N < 1) return 0ull;
  return wsattn::bwd_workspace_bytes(B, H, N);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, void* workspace,
             unsigned long long workspace_bytes, int B, int H, int N, int d, float scale,
             int causal, int dtype, struct CUstream_st* stream) {
  return wsattn::run_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N,
                         d, scale, causal, dtype, reinterpret_cast<cudaStream_t>(stream));
}

int attn_fwd_fp8_blockscaled(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int H, int N, int d, float scale, int causal,
                             const float* q_scales, const float* k_scales, float v_descale,
                             struct CUstream_st* stream) {
  if (!q_scales || !k_scales) return wsattn::kErrInvalidArg;
  if (reinterpret_cast<uintptr_t>(q_scales) % 4 || reinterpret_cast<uintptr_t>(k_scales) % 4)
    return wsattn::kErrMisaligned;
  return wsattn::run(q, k, v, o, lse, B, H, N, d, scale, causal, ATTN_FP8_E4M3, 1.0f, 1.0f,
                     v_descale, reinterpret_cast<cudaStream_t>(stream), q_scales, k_scales);
}

int attn_fwd_status(struct CUstream_st* stream) {
  int dev = -1;
  int rc = wsattn::current_device(&dev);
  if (rc != wsattn::kOk) return rc;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return wsattn::kErrCuda;
  }
  return wsattn::read_and_clear_status(dev);
}

int attn_watchdog_selftest(unsigned int timeout_us, struct CUstream_st* stream) {
  if (timeout_us < 1u || timeout_us > 10000000u) return wsattn::kErrInvalidArg;
  int dev = -1;
  int rc = wsattn::current_device(&dev);
  if (rc != wsattn::kOk) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  wsattn::watchdog_selftest_kernel<<<1, 32, 0, s>>>(
      static_cast<unsigned long long>(timeout_us) * 1000ull, wsattn::g_dev[dev].status,
      wsattn::g_dev[dev].where);
  if (cudaGetLastError() != cudaSuccess) return wsattn::kErrCuda;
  return attn_fwd_status(stream);
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED";
    case ATTN_ERR_DEVICE: return "ATTN_ERR_DEVICE";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    default: return "ATTN_ERR_UNKNOWN";
  }
}

}  // extern "C"

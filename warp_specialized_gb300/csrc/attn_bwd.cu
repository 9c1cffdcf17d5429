// Backward-pass launches: preprocess, dQ kernel, dK/dV kernel for fp16 and
// bf16, d = 64 and 128.
#include "attn_bwd_kernel.cuh"
#include "attn_instance.cuh"

namespace wsattn {
namespace {

template <typename K>
int prepare_kernel(K kern, int smem_bytes, int device, std::atomic<int>* ready) {
  int st = ready[device].load(std::memory_order_acquire);
  if (st == 0) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
            cudaSuccess) {
      cudaGetLastError();
      return kErrCuda;
    }
    // the warpgroups' setmaxnreg split draws on exactly this many registers
    st = (fa.maxThreadsPerBlock >= kBwdThreads && fa.numRegs == kBwdLaunchRegs) ? 1 : 2;
    ready[device].store(st, std::memory_order_release);
  }
  return st == 1 ? kOk : kErrUnsupported;
}

template <int DT, int D, bool CAUSAL>
int launch_bwd_instance(const BwdLaunchArgs& a) {
  using BC = BwdCfg<DT, D>;
  if (a.device < 0 || a.device >= kMaxDevices) return kErrDevice;
  static std::atomic<int> ready_dq[kMaxDevices], ready_dkv[kMaxDevices];
  auto kdq = attn_bwd_dq_kernel<DT, D, CAUSAL>;
  auto kdkv = attn_bwd_dkv_kernel<DT, D, CAUSAL>;
  int rc = prepare_kernel(kdq, BC::kSmemDq, a.device, ready_dq);
  if (rc == kOk) rc = prepare_kernel(kdkv, BC::kSmemDkv, a.device, ready_dkv);
  if (rc != kOk) return rc;

  LaunchArgs la{};
  la.B = a.B;
  la.H = a.H;
  la.N = a.N;
  la.d = D;
  la.encode = a.encode;
  CUtensorMap mq, mk, mv, mdo;
  CUtensorMap mq64, mdo64;  // the dK/dV kernel streams Q and dO in 64-row halves
  if (!encode_map<DT, D>(la, a.q, kBlock, &mq) || !encode_map<DT, D>(la, a.k, kBlock, &mk) ||
      !encode_map<DT, D>(la, a.v, kBlock, &mv) || !encode_map<DT, D>(la, a.dout, kBlock, &mdo) ||
      !encode_map<DT, D>(la, a.q, 64, &mq64) || !encode_map<DT, D>(la, a.dout, 64, &mdo64))
    return kErrCuda;

  BwdParams p;
  p.o = a.o;
  p.dout = a.dout;
  p.lse = a.lse;
  p.ws = static_cast<float*>(a.workspace);
  p.dq = a.dq;
  p.dk = a.dk;
  p.dv = a.dv;
  p.N = a.N;
  p.nt = (a.N + kBlock - 1) / kBlock;
  p.Np = p.nt * kBlock;
  p.BH = a.B * a.H;
  p.n_items = p.BH * p.nt;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.timeout_ns = a.timeout_ns;
  p.status = a.status;
  p.where = a.where;

  const long long rows = static_cast<long long>(p.BH) * p.Np;
  constexpr int kPreRows = PreprocessShape<D>::kRowsPerBlock;
  const long long pre_blocks = (rows + kPreRows - 1) / kPreRows;
  const long long pre_cap = 8LL * a.num_sms;  // eight 256-thread blocks fill an SM
  attn_bwd_preprocess_kernel<DT, D>
      <<<static_cast<unsigned>(pre_blocks < pre_cap ? pre_blocks : pre_cap), 256, 0, a.stream>>>(p);
  const int grid = p.n_items < a.num_sms ? p.n_items : a.num_sms;
  kdq<<<grid, kBwdThreads, BC::kSmemDq, a.stream>>>(mq, mk, mv, mdo, p);
  if (cudaGetLastError() != cudaSuccess) return kErrCuda;
  // The dK/dV kernel reads only what the preprocess kernel (complete before
  // the dQ kernel started) and the caller wrote, so its CTAs may take the
  // SMs the dQ kernel's CTAs leave, over the dQ kernel's last round
  // (programmatic dependent launch); it waits for the dQ grid before it
  // exits, so that its completion still implies the dQ kernel's.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kBwdThreads, 1, 1);
  cfg.dynamicSmemBytes = BC::kSmemDkv;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kdkv, mq64, mk, mv, mdo64, p) != cudaSuccess) {
    cudaGetLastError();
    return kErrCuda;
  }
  return kOk;
}

template <int DT, int D>
int launch_bwd_mask(const BwdLaunchArgs& a) {
  return a.causal ? launch_bwd_instance<DT, D, true>(a) : launch_bwd_instance<DT, D, false>(a);
}

}  // namespace

int launch_bwd(const BwdLaunchArgs& a) {
  if (a.dtype == 2) {
    if (a.d == 64) return launch_bwd_mask<2, 64>(a);
    if (a.d == 128) return launch_bwd_mask<2, 128>(a);
  } else if (a.dtype == 1) {
    if (a.d == 64) return launch_bwd_mask<1, 64>(a);
    if (a.d == 128) return launch_bwd_mask<1, 128>(a);
  }
  return kErrUnsupported;
}

}  // namespace wsattn

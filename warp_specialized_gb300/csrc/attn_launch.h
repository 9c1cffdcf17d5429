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
  // caller workspace for the tail launch (null: whole rounds only)
  void* workspace;
  unsigned long long workspace_bytes;
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

// Workspace the forward tail launch needs on a device with num_sms SMs:
// the pieces' flags (two words per tail item, at most num_sms items), then
// two (O, m, l) slots per CTA and query tile, 128 * (d + 2) floats each.
inline unsigned long long fwd_flags_bytes(int num_sms) {
  return (static_cast<unsigned long long>(num_sms) * 2ull * 4ull + 255ull) / 256ull * 256ull;
}
inline unsigned long long fwd_workspace_bytes(int num_sms, int d, int nqt) {
  return fwd_flags_bytes(num_sms) +
         static_cast<unsigned long long>(num_sms) * 2ull * nqt * 128ull * (d + 2ull) * 4ull;
}

// The split of the work left after whole rounds (one item per SM per
// round) for the tail launch: items [start, n_items), their key blocks
// (units) in all, and the tail grid (at least kTailMinBlocks units per CTA:
// shorter runs cost more in start-up and merging than they save).
constexpr int kTailMinBlocks = 8;
// Key blocks the split costs beyond a CTA's share: the second launch's
// start, the pieces' partial writes and merges, and the stall of a CTA's
// next segment behind the hand-over of its first.  (Measured on GB300 for
// d = 128: 32 or 64 items of 64 blocks finish 15 to 18 % sooner split over
// the SMs; 128 items, 54 blocks a CTA, 13 to 16 % later.)
constexpr int kTailCostBlocks = 20;
// Behind a main launch the tail CTAs start as the main CTAs finish, over
// about this many key blocks' time; the first CTA gets half of it extra and
// the last half of it less (see tail_range_start).
constexpr int kTailRampBlocks = 8;
// Shared memory a merging piece may stage the other pieces' (O, m, l) rows
// in after its CTA's last MMA: the Q tiles and the K/V ring, in the forward
// kernel's layout (restated here for the host; the tail kernel asserts that
// the two agree).
constexpr int kFwdSmemLimit = 232448;
constexpr int kFwdMiscBytes = 1024 + 512 + 2 * 128 * 4 + 2 * 2 * 128 * 4;
constexpr int kFwdStageBytes = 128 * 128;
constexpr int fwd_tile_bytes(int d, int esize) { return d * esize * 128; }
constexpr int fwd_nqt(int d, int esize) {
  return (d <= 128 && fwd_tile_bytes(d, esize) <= 32768) ? 2 : 1;
}
constexpr int fwd_region_bytes(int d, int esize) {
  return (fwd_nqt(d, esize) +
          ((kFwdSmemLimit - kFwdMiscBytes - kFwdStageBytes * (esize == 1 ? 2 : 1) -
            fwd_nqt(d, esize) * fwd_tile_bytes(d, esize)) / fwd_tile_bytes(d, esize) > 8
               ? 8
               : (kFwdSmemLimit - kFwdMiscBytes - kFwdStageBytes * (esize == 1 ? 2 : 1) -
                  fwd_nqt(d, esize) * fwd_tile_bytes(d, esize)) / fwd_tile_bytes(d, esize))) *
         fwd_tile_bytes(d, esize);
}
// pieces per tile whose merge fits the staging (this piece and the others)
constexpr int tail_max_pieces(int d, int esize) {
  return 1 + fwd_region_bytes(d, esize) / ((d + 2) * 128 * 4);
}
struct TailPlan {
  int start = 0, items = 0, grid = 0, max_walk = 0;
  long long units = 0;
  bool causal = false;
};
// ramp of the tail ranges: none without a main launch, never more than a
// quarter of a CTA's share (so that every range holds work)
inline int tail_ramp(const TailPlan& t, bool after_main) {
  if (!after_main || t.grid == 0) return 0;
  const long long quarter = t.units / t.grid / 4;
  return static_cast<int>(quarter < kTailRampBlocks / 2 ? quarter : kTailRampBlocks / 2);
}
// The leftover items and the tail grid: as many CTAs as keep every CTA's
// share at kTailMinBlocks or more and at (longest item - 1) / (max_pieces -
// 1) or more (plus a margin for the ramp), so that an item falls to at most
// max_pieces CTAs and its merge can be staged.
inline TailPlan plan_tail(int BH, int n_pairs, int nkv, int nqt, bool causal, int num_sms,
                          int max_pieces) {
  TailPlan t;
  t.causal = causal;
  const int n_items = BH * n_pairs;
  t.items = n_items % num_sms;
  t.start = n_items - t.items;
  for (int it = t.start; it < n_items; ++it) {
    int walk = nkv;
    if (causal) {  // causal items run longest first, level by level
      const int pair = n_pairs - 1 - it / BH;
      walk = pair * nqt + nqt < nkv ? pair * nqt + nqt : nkv;
    }
    t.units += walk;
    if (walk > t.max_walk) t.max_walk = walk;
  }
  long long share = kTailMinBlocks;
  if (max_pieces >= 2) {
    const long long s = (t.max_walk - 1 + max_pieces - 2) / (max_pieces - 1) + 2;
    if (s > share) share = s;
  } else {
    share = t.max_walk;
  }
  long long g = t.units / share;
  if (g < 1) g = 1;
  t.grid = static_cast<int>(g < num_sms ? g : num_sms);
  if (t.items == 0) t.grid = 0;
  return t;
}
// Whether splitting pays: only where the whole problem is one partial round
// (fewer items than SMs), whose static cost is the longest item, against a
// CTA's share plus the split's own cost.  Behind whole rounds the measured
// gain is 2 % at best and often a loss (the causal schedule, largest items
// first in snake order, already evens the rounds out), so it is not advised
// there; attn_fwd_ws still splits when called.
inline bool tail_split_pays(const TailPlan& t) {
  if (t.items == 0 || t.grid == 0 || t.start > 0) return false;
  const long long share = (t.units + t.grid - 1) / t.grid;
  return t.max_walk > share + kTailCostBlocks;
}

// Backward pass (fp16 / bf16, d = 64 or 128); returns a status code.
int launch_bwd(const BwdLaunchArgs& a);

// One entry per element type; each returns a status code.
int launch_fp32(const LaunchArgs& a);
int launch_fp16(const LaunchArgs& a);
int launch_bf16(const LaunchArgs& a);
int launch_fp8(const LaunchArgs& a);
// ATTN_OPT_EXP2_FMA (bf16 d = 64 / 128, e4m3 d = 128; else kErrUnsupported)
int launch_exp2_fma(const LaunchArgs& a, int dtype);

}  // namespace wsattn

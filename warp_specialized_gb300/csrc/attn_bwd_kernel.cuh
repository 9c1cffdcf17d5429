// attn_bwd_kernel.cuh - backward pass of the fused attention for sm_103a:
// dQ, dK, dV from Q, K, V, O, dO and the forward's per-row logsumexp.
//
// The gradients of O = softmax(scale Q K^T [+ mask]) V for an output
// gradient dO, per (b, h):
//   P_ij  = exp(scale q_i.k_j - LSE_i)      (0 where masked)
//   D_i   = dO_i . O_i                      (= sum_j P_ij dP_ij)
//   dP_ij = dO_i . v_j
//   dS_ij = P_ij (dP_ij - D_i)
//   dV_j  = sum_i P_ij dO_i
//   dQ_i  = scale sum_j dS_ij k_j
//   dK_j  = scale sum_i dS_ij q_i
// The forward's LSE output ("Warp specialization" concept card, section
// "Implementation sketch": the consumer returns row_max + log(row_sum))
// lets every block recompute its probabilities directly, without a running
// max.
//
// Three kernels, all on the tensor cores where the work is a contraction:
//   preprocess   D_i and LSE_i * log2(e) per row into a workspace padded to
//                whole 128-row tiles (padding rows: LSE = +inf, D = 0, so
//                their probabilities are exactly 0);
//   dQ kernel    one 128-row query tile per work item, K_j and V_j streamed
//                through TMA rings of their own: S = Q K_j^T and dP = dO V_j^T into
//                Tensor Memory, dS written back to its own TMEM columns,
//                dQ += dS K_j accumulated in TMEM;
//   dK/dV kernel one 128-key tile per work item, Q_i / dO_i (and the
//                workspace rows of tile i) streamed: S^T = K Q_i^T and
//                dP^T = V dO_i^T, P^T and dS^T written over them in TMEM,
//                dV += P^T dO_i and dK += dS^T Q_i accumulated in TMEM.
// Neither kernel needs atomics; each output element is written once.
// Roles per CTA (384 threads): warp 0 lane 0 TMA producer, warp 1 lane 0
// MMA issuer, warps 4-7 and 8-11 two elementwise warpgroups that split the
// 128 columns of every block (columns 0-63 and 64-127; a thread is one row
// / TMEM lane of its half) and also write the outputs.  The MMA thread
// starts the products over the first half of the columns as soon as that
// half is ready.  Every wait is bounded.
#pragma once

#include <type_traits>

#include "attn_fwd_kernel.cuh"

namespace wsattn {

constexpr int kBwdThreads = 384;
// Registers per thread after setmaxnreg: the producer / MMA warpgroup gives
// up registers so that each elementwise thread can hold its half-row of S
// and dP (128 values) at once.  80 + 2 * 208 = 496 of the 3 * 168 the block
// is launched with (the host refuses to launch any other count).
constexpr int kBwdLaunchRegs = 168;
constexpr int kBwdRegsControl = 80;
constexpr int kBwdRegsElem = 208;
static_assert(kBwdRegsControl + 2 * kBwdRegsElem <= 3 * kBwdLaunchRegs, "register split");


// The same bounded wait executed by a whole warp, its result made
// warp-uniform (false for every lane if any lane gave up), for warps that
// go on to warp-synchronous TMEM loads and stores.
__device__ __forceinline__ bool wait_bar_all(uint32_t bar, uint32_t parity, const WaitCtx& wc,
                                            unsigned where) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, wc, where)) != 0;
}

template <int DT, int D>
struct BwdCfg {
  using C = Cfg<DT, D>;
  static constexpr int kTileBytes = C::kTileBytes;
  static constexpr int kVecBytes = 2 * kBlock * 4;  // (lse2, D) of one 128-row tile
  // dQ kernel: Q + dO resident, K/V ring
  static constexpr int kMiscDq = 1024 + 512;
  static constexpr int kSlotsDqFit = (kSmemLimit - kMiscDq - 2 * kTileBytes) / kTileBytes;
  static constexpr int kSlotsDq = kSlotsDqFit > kMaxSlots ? kMaxSlots : kSlotsDqFit;
  static constexpr int kSmemDq = kMiscDq + (2 + kSlotsDq) * kTileBytes;
  // dK/dV kernel: K + V resident, ring of (Q_i, dO_i, vec_i)
  static constexpr int kStageBytes = 2 * kTileBytes + kVecBytes;
  static constexpr int kMiscDkv = 1024 + 512;
  // the epilogue's per-warp staging: 8 elementwise warps x 32 rows x 64 bytes
  static constexpr int kEpiBytes = 8 * 32 * 64;
  static constexpr int kStagesFit =
      (kSmemLimit - kMiscDkv - kEpiBytes - 2 * kTileBytes) / kStageBytes;
  static constexpr int kStages = kStagesFit > 4 ? 4 : kStagesFit;
  static constexpr int kSmemDkv = kMiscDkv + 2 * kTileBytes + kStages * kStageBytes + kEpiBytes;
  static_assert(kSlotsDq >= 2 && kStages >= 2, "backward shared-memory budget");
  static_assert(kSmemDq <= kSmemLimit && kSmemDkv <= kSmemLimit, "shared memory budget");

  // instruction descriptors: K-major x K-major (S, dP, S^T, dP^T) and
  // TMEM A x MN-major B (dQ, dV, dK)
  static constexpr uint32_t kIdescSS = make_idesc(C::T::kFmt, C::T::kFmt, false, kBlock, kBlock);
  // the same with N = 64: one half of the streamed tile's rows as B
  static constexpr uint32_t kIdescSSHalf = make_idesc(C::T::kFmt, C::T::kFmt, false, 64, kBlock);
  static constexpr uint32_t kIdescTS = make_idesc(C::T::kFmt, C::T::kFmt, true, D, kBlock);
  // TMEM columns, dQ kernel: S | dP | dS (16-bit, 64 columns) | dQ | Q
  // (16-bit, the A operand of S = Q K^T, copied in once per query tile)
  static constexpr uint32_t kDqS = 0, kDqDP = 128, kDqDS = 256, kDqAcc = 320;
  static constexpr uint32_t kDqQ = kDqAcc + D;
  // TMEM columns, dK/dV kernel: S^T (P^T over it) | dP^T (dS^T over it) | dV | dK
  static constexpr uint32_t kKvS = 0, kKvDP = 128, kKvDV = 256, kKvDK = 256 + D;
  static_assert(kDqQ + D / 2 <= 512 && kKvDK + D <= 512, "Tensor Memory budget");
};

struct BwdParams {
  const void* o;       // forward output [B, H, N, d]
  const void* dout;    // output gradient [B, H, N, d]
  const float* lse;    // [B, H, N]
  float* ws;           // [B*H, Np, 2] (lse2, D), Np = N rounded up to 128
  void* dq;
  void* dk;
  void* dv;
  int N;
  int Np;
  int BH;
  int nt;              // 128-row tiles per head
  int n_items;         // BH * nt
  float scale;         // softmax scale (applied to dQ, dK)
  float scale_log2;    // scale * log2(e)
  unsigned long long timeout_ns;
  unsigned int* status;
  unsigned int* where;
};

// ---------------------------------------------------------------------------
// preprocess: D / 8 lanes per (padded) row, each reading 16 bytes of O and
// of dO (a warp holds 256 / D rows), so that every load is a whole 16-byte
// vector and a warp's loads cover whole rows

template <int D>
struct PreprocessShape {
  static constexpr int kLanesPerRow = D / 8;
  static constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  static constexpr int kRowsPerBlock = 8 * kRowsPerWarp;  // 256 threads
  static_assert(128 % kRowsPerBlock == 0, "blocks hold whole 128-row tiles");
};

// One (padded) row: D = dO . O and LSE * log2(e) into the workspace.
template <int DT, int D>
__device__ __forceinline__ void preprocess_row(const BwdParams& p, long long row, int sub) {
  using S = PreprocessShape<D>;
  const long long bh = row / p.Np;
  const int i = static_cast<int>(row - bh * p.Np);
  const bool real = i < p.N;  // padding rows: LSE = +inf, D = 0
  uint4 ov = make_uint4(0u, 0u, 0u, 0u), dv = ov;
  float lse = INFINITY;
  if (real) {  // all three loads in flight together
    const long long g = (bh * p.N + i) * D + sub * 8;
    ov = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.o) + g));
    dv = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.dout) + g));
    if (sub == 0) lse = __ldg(p.lse + bh * p.N + i) * 1.4426950408889634f;
  }
  const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, dw[4] = {dv.x, dv.y, dv.z, dv.w};
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float2 of, df;
    if constexpr (DT == 1) {
      of = __half22float2(*reinterpret_cast<const __half2*>(&ow[k]));
      df = __half22float2(*reinterpret_cast<const __half2*>(&dw[k]));
    } else {
      of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[k]));
      df = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dw[k]));
    }
    acc = fmaf(of.x, df.x, acc);
    acc = fmaf(of.y, df.y, acc);
  }
  // the lanes of a row are consecutive and aligned to kLanesPerRow
#pragma unroll
  for (int off = S::kLanesPerRow / 2; off > 0; off >>= 1)
    acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (sub == 0) reinterpret_cast<float2*>(p.ws)[row] = make_float2(lse, acc);
}

// A grid of a few blocks per SM strides over the rows, one row group per
// warp at a time; the padded row count is a multiple of 128, so every warp
// step covers whole rows and its shuffles see all 32 lanes.
template <int DT, int D>
__global__ void __launch_bounds__(256) attn_bwd_preprocess_kernel(const BwdParams p) {
  using S = PreprocessShape<D>;
  const int lane = threadIdx.x & 31;
  const int sub = lane % S::kLanesPerRow;  // 16-byte column group of the row
  const long long rows = static_cast<long long>(p.BH) * p.Np;
  const long long stride = static_cast<long long>(gridDim.x) * S::kRowsPerBlock;
#pragma unroll 4
  for (long long row = static_cast<long long>(blockIdx.x) * S::kRowsPerBlock +
                       (threadIdx.x >> 5) * S::kRowsPerWarp + lane / S::kLanesPerRow;
       row < rows; row += stride)
    preprocess_row<DT, D>(p, row, sub);
}

// ---------------------------------------------------------------------------
// shared helpers

struct BwdItem {
  int bh;
  int tile;  // query tile (dQ kernel) or key tile (dK/dV kernel)
  int n;     // number of streamed tiles
  int first; // first streamed tile
};

// dQ kernel item: query tile qi streams key tiles 0 .. n-1 (causal: qi+1
// of them), most work first when causal.
template <bool CAUSAL>
__device__ __forceinline__ BwdItem dq_item(int it, const BwdParams& p) {
  BwdItem w;
  if (CAUSAL) {
    w.tile = p.nt - 1 - it / p.BH;
    w.bh = it % p.BH;
    w.n = w.tile + 1;
  } else {
    w.bh = it / p.nt;
    w.tile = it % p.nt;
    w.n = p.nt;
  }
  w.first = 0;
  return w;
}

// dK/dV kernel item: key tile kj streams query tiles first .. nt-1
// (causal: from kj on), most work first when causal.
template <bool CAUSAL>
__device__ __forceinline__ BwdItem dkv_item(int it, const BwdParams& p) {
  BwdItem w;
  if (CAUSAL) {
    w.tile = it / p.BH;
    w.bh = it % p.BH;
    w.first = w.tile;
  } else {
    w.bh = it / p.nt;
    w.tile = it % p.nt;
    w.first = 0;
  }
  w.n = p.nt - w.first;
  return w;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

template <int DT, int D>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* map, int row0, int bh,
                                          uint32_t bar) {
  using C = Cfg<DT, D>;
#pragma unroll
  for (int b = 0; b < C::kNumBox; ++b)
    tma_load_3d(dst + b * C::kBoxBytes, map, b * C::kBoxInner, row0, bh, bar);
}

// A x B^T with both operands K-major in shared memory (S = Q K^T etc.)
template <int DT, int D>
__device__ __forceinline__ void mma_kk(uint32_t d_tmem, uint32_t sa, uint32_t sb, uint32_t idesc) {
  using C = Cfg<DT, D>;
  const uint64_t a0 = make_sdesc_sw128(sa, 16, 1024);
  const uint64_t b0 = make_sdesc_sw128(sb, 16, 1024);
#pragma unroll
  for (int k = 0; k < C::kNumQKMma; ++k) {
    const uint32_t off = ((k >> 2) * C::kBoxBytes + (k & 3) * 32) >> 4;
    mma_ss<C::T::kKind>(d_tmem, a0 + off, b0 + off, idesc, k > 0 ? 1u : 0u);
  }
}


// mma_tk over half of B's 128 rows (HALF 0: rows 0-63, HALF 1: 64-127), N = 64
template <int DT, int D, int HALF>
__device__ __forceinline__ void mma_tk_half(uint32_t d_tmem, uint32_t a_tmem, uint32_t sb,
                                            uint32_t idesc) {
  using C = Cfg<DT, D>;
  const uint64_t b0 = make_sdesc_sw128(sb + HALF * 64 * 128, 16, 1024);
#pragma unroll
  for (int k = 0; k < C::kNumQKMma; ++k) {
    const uint32_t off = ((k >> 2) * C::kBoxBytes + (k & 3) * 32) >> 4;
    mma_ts<C::T::kKind>(d_tmem, a_tmem + k * 8, b0 + off, idesc, k > 0 ? 1u : 0u);
  }
}

// D (+)= A B with A (128 x 128, 16-bit) in TMEM and B = a [128 rows x d]
// tile (d contiguous) as the MN-major B operand
template <int DT, int D>
__device__ __forceinline__ void mma_tmn(uint32_t d_tmem, uint32_t a_tmem, uint32_t sb,
                                        uint32_t idesc, bool accumulate) {
  using C = Cfg<DT, D>;
  const uint64_t b0 = make_sdesc_sw128(sb, C::kBoxBytes, 1024);
#pragma unroll
  for (int k = 0; k < C::kNumPVMma; ++k) {
    const uint32_t off = (k * C::kKPerMma * 128) >> 4;
    mma_ts<C::T::kKind>(d_tmem, a_tmem + k * 8, b0 + off, idesc, (accumulate || k > 0) ? 1u : 0u);
  }
}

// The same over half of the contraction (HALF 0: rows 0-63 of B and TMEM
// columns 0-31 of A; HALF 1: rows 64-127, columns 32-63)
template <int DT, int D, int HALF>
__device__ __forceinline__ void mma_tmn_half(uint32_t d_tmem, uint32_t a_tmem, uint32_t sb,
                                             uint32_t idesc, bool accumulate) {
  using C = Cfg<DT, D>;
  constexpr int kHalf = C::kNumPVMma / 2;
  const uint64_t b0 = make_sdesc_sw128(sb, C::kBoxBytes, 1024);
#pragma unroll
  for (int k = HALF * kHalf; k < (HALF + 1) * kHalf; ++k) {
    const uint32_t off = (k * C::kKPerMma * 128) >> 4;
    mma_ts<C::T::kKind>(d_tmem, a_tmem + k * 8, b0 + off, idesc, (accumulate || k > 0) ? 1u : 0u);
  }
}

// A x B^T over half of B's 128 rows (HALF 0: rows 0-63, HALF 1: 64-127;
// each is 8 whole 128-byte swizzle atoms per box), N = 64, into d_tmem.
template <int DT, int D, int HALF>
__device__ __forceinline__ void mma_kk_half(uint32_t d_tmem, uint32_t sa, uint32_t sb,
                                            uint32_t idesc) {
  using C = Cfg<DT, D>;
  const uint64_t a0 = make_sdesc_sw128(sa, 16, 1024);
  const uint64_t b0 = make_sdesc_sw128(sb + HALF * 64 * 128, 16, 1024);
#pragma unroll
  for (int k = 0; k < C::kNumQKMma; ++k) {
    const uint32_t off = ((k >> 2) * C::kBoxBytes + (k & 3) * 32) >> 4;
    mma_ss<C::T::kKind>(d_tmem, a0 + off, b0 + off, idesc, k > 0 ? 1u : 0u);
  }
}

// D (+)= A B over one half of the contraction, with that half of A packed
// in its own 32 TMEM columns from a_half (B rows 64 HALF .. 64 HALF + 63).
template <int DT, int D, int HALF>
__device__ __forceinline__ void mma_tmn_part(uint32_t d_tmem, uint32_t a_half, uint32_t sb,
                                             uint32_t idesc, bool accumulate) {
  using C = Cfg<DT, D>;
  constexpr int kHalf = C::kNumPVMma / 2;
  const uint64_t b0 = make_sdesc_sw128(sb, C::kBoxBytes, 1024);
#pragma unroll
  for (int k = HALF * kHalf; k < (HALF + 1) * kHalf; ++k) {
    const uint32_t off = (k * C::kKPerMma * 128) >> 4;
    mma_ts<C::T::kKind>(d_tmem, a_half + (k - HALF * kHalf) * 8, b0 + off, idesc,
                        (accumulate || k > 0) ? 1u : 0u);
  }
}

// 32 fp32 values of a row times `f` -> output type, 64 (16-bit) bytes
template <int DT>
__device__ __forceinline__ void store_row_chunk(void* dst, const uint32_t (&v)[32], float f) {
  float x[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(v[i]) * f;
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] = pack8_out<DT>(x + 8 * i);
}

// 32 fp32 values of each of a warp's 32 consecutive rows (lane l: row l),
// times `f`, to the output type, through a 2 KiB shared-memory area of the
// warp: written one row per lane, read back so that each global store
// instruction covers 8 rows x 64 contiguous bytes (whole 32-byte sectors)
// instead of 32 rows x 16 bytes.  Chunk c of row r sits at chunk
// c ^ ((r >> 1) & 3) of its 64-byte row, which keeps both the row-per-lane
// writes and the row-group reads free of bank conflicts.  out: this warp's
// row 0 at the chunk's first column; pitch: bytes per row; n_valid: rows
// that exist (the others are not stored).
template <int DT>
__device__ __forceinline__ void store_rows_staged(uint8_t* out, size_t pitch, int n_valid,
                                                  const uint32_t (&v)[32], float f,
                                                  uint32_t stage, uint32_t lane) {
  float x[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(v[i]) * f;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    st_shared_v4(stage + lane * 64u + ((static_cast<uint32_t>(c) ^ ((lane >> 1) & 3u)) << 4),
                 pack8_out<DT>(x + 8 * c));
  __syncwarp();
  const uint32_t ch = lane & 3u;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t rr = 8u * k + (lane >> 2);
    const uint4 w = ld_shared_v4(stage + rr * 64u + ((ch ^ ((rr >> 1) & 3u)) << 4));
    if (static_cast<int>(rr) < n_valid)
      *reinterpret_cast<uint4*>(out + rr * pitch + ch * 16u) = w;
  }
  __syncwarp();  // the area is rewritten by the next call
}

// ---------------------------------------------------------------------------
// dQ kernel

// K and V stream through rings of their own: V_j is free as soon as dP(j)
// is done, K_j only after dQ += dS(j) K_j, and one shared ring would hold
// each V load back behind a K slot.
template <int NK, int NV>
struct DqCtrl {
  uint64_t qd_full, qd_empty;
  uint64_t k_full[NK], k_empty[NK];
  uint64_t v_full[NV], v_empty[NV];
  uint64_t s_full[2];    // S(j), dP(j), keys 0-63 / 64-127, in TMEM (commit)
  uint64_t sdp_free[2];  // elementwise read them (the 4 warps of that key half)
  uint64_t ds_full[2];  // dS(j), keys 0-63 / 64-127, in TMEM (4 warps each)
  uint64_t ds_free;   // dQ += dS(j) K_j done            (commit)
  uint64_t dq_full;   // last dQ MMA of the item done    (commit)
  uint64_t dq_empty;  // epilogue read dQ                (8 warps)
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort;
};

template <int DT, int D, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const BwdParams p) {
  using C = Cfg<DT, D>;
  using BC = BwdCfg<DT, D>;
  constexpr int NS = BC::kSlotsDq;
  constexpr int NV = NS / 2, NK = NS - NV;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* sbase = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sQ = smem_u32(sbase), sdO = sQ + C::kTileBytes, sK = sdO + C::kTileBytes,
                 sV = sK + NK * C::kTileBytes;
  DqCtrl<NK, NV>* c = reinterpret_cast<DqCtrl<NK, NV>*>(sbase + (2 + NS) * C::kTileBytes);
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&c->qd_full), 1);
    mbar_init(smem_u32(&c->qd_empty), 1);
    for (int s = 0; s < NK; ++s) {
      mbar_init(smem_u32(&c->k_full[s]), 1);
      mbar_init(smem_u32(&c->k_empty[s]), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(smem_u32(&c->v_full[s]), 1);
      mbar_init(smem_u32(&c->v_empty[s]), 1);
    }
    mbar_init(smem_u32(&c->s_full[0]), 1);
    mbar_init(smem_u32(&c->s_full[1]), 1);
    mbar_init(smem_u32(&c->sdp_free[0]), 4);
    mbar_init(smem_u32(&c->sdp_free[1]), 4);
    mbar_init(smem_u32(&c->ds_full[0]), 4);
    mbar_init(smem_u32(&c->ds_full[1]), 4);
    mbar_init(smem_u32(&c->ds_free), 1);
    mbar_init(smem_u32(&c->dq_full), 1);
    mbar_init(smem_u32(&c->dq_empty), 8);
    mbar_init(smem_u32(&c->drain), 1);
    c->abort = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&c->tmem_base), 512);
    tmem_relinquish();
  }
  // the dK/dV grid, which reads nothing this one writes, may take the SMs
  // this grid's CTAs leave (programmatic dependent launch)
  if (threadIdx.x == 0) griddep_launch_dependents();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = c->tmem_base;
  const WaitCtx wc{&c->abort, p.timeout_ns, p.status, p.where};

  if (warp < 4) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kBwdRegsControl));
  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    uint32_t qd_uses = 0, loads[2] = {0, 0}, round[2] = {0, 0};
    int slot[2] = {0, 0};
    bool ok = true;
    // the next tile of ring kv (0: K, 1: V) once its slot is free
    auto load_ring = [&](int kv, int j, int bh) -> bool {
      const int s = slot[kv];
      const uint32_t empty = smem_u32(kv == 0 ? &c->k_empty[s] : &c->v_empty[s]);
      const uint32_t full = smem_u32(kv == 0 ? &c->k_full[s] : &c->v_full[s]);
      if (!wait_bar(empty, (round[kv] & 1u) ^ 1u, wc, 0x42)) return false;
      mbar_arrive_expect_tx(full, C::kTileBytes);
      load_tile<DT, D>((kv == 0 ? sK : sV) + s * C::kTileBytes, kv == 0 ? &tmK : &tmV, j * kBlock,
                       bh, full);
      ++loads[kv];
      if (++slot[kv] == (kv == 0 ? NK : NV)) {
        slot[kv] = 0;
        ++round[kv];
      }
      return true;
    };
    for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < p.n_items && ok; ++rnd) {
      const int it = round_item(rnd, p.n_items);
      if (it < 0) continue;
      const BwdItem w = dq_item<CAUSAL>(it, p);
      if (!wait_bar(smem_u32(&c->qd_empty), (qd_uses & 1u) ^ 1u, wc, 0x41)) break;
      mbar_arrive_expect_tx(smem_u32(&c->qd_full), 2 * C::kTileBytes);
      load_tile<DT, D>(sQ, &tmQ, w.tile * kBlock, w.bh, smem_u32(&c->qd_full));
      load_tile<DT, D>(sdO, &tmdO, w.tile * kBlock, w.bh, smem_u32(&c->qd_full));
      ++qd_uses;
      for (int j = 0; j < w.n && ok; ++j) ok = load_ring(0, j, w.bh) && load_ring(1, j, w.bh);
    }
    volatile uint32_t never = 0;
    const WaitCtx wn{&never, p.timeout_ns, p.status, p.where};
    for (int s = 0; s < NK; ++s) {
      const uint32_t uses = loads[0] / NK + (static_cast<uint32_t>(s) < loads[0] % NK ? 1u : 0u);
      if (uses) wait_bar(smem_u32(&c->k_full[s]), (uses - 1u) & 1u, wn, 0x43);
    }
    for (int s = 0; s < NV; ++s) {
      const uint32_t uses = loads[1] / NV + (static_cast<uint32_t>(s) < loads[1] % NV ? 1u : 0u);
      if (uses) wait_bar(smem_u32(&c->v_full[s]), (uses - 1u) & 1u, wn, 0x43);
    }
    if (qd_uses) wait_bar(smem_u32(&c->qd_full), (qd_uses - 1u) & 1u, wn, 0x44);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA
    uint32_t qd_w = 0, sf_w = 0, ds_w = 0, dqe_w = 0;
    uint32_t round[2] = {0, 0};
    int slot[2] = {0, 0};
    auto next_slot = [&](int kv, int& s, uint32_t& par) {
      s = slot[kv];
      par = round[kv] & 1u;
      if (++slot[kv] == (kv == 0 ? NK : NV)) {
        slot[kv] = 0;
        ++round[kv];
      }
    };
    const uint32_t tS = tbase + BC::kDqS, tDP = tbase + BC::kDqDP, tDS = tbase + BC::kDqDS,
                   tDQ = tbase + BC::kDqAcc, tQ = tbase + BC::kDqQ;
    bool ok = true;
    for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < p.n_items && ok; ++rnd) {
      const int it = round_item(rnd, p.n_items);
      if (it < 0) continue;
      const BwdItem w = dq_item<CAUSAL>(it, p);
      int ks, vs;
      uint32_t kp, vp;
      next_slot(0, ks, kp);
      next_slot(1, vs, vp);
      ok = wait_bar(smem_u32(&c->qd_full), qd_w & 1u, wc, 0x51) &&
           wait_bar(smem_u32(&c->k_full[ks]), kp, wc, 0x52) &&
           wait_bar(smem_u32(&c->v_full[vs]), vp, wc, 0x52);
      ++qd_w;
      if (!ok) break;
      tc_fence_after_sync();
      // Q into Tensor Memory (the previous tile's last S was issued before,
      // and the tensor pipe runs this thread's operations in order), so
      // that S = Q K_j^T reads only K_j from shared memory
      copy_tile_to_tmem<DT, D>(tQ, sQ);
      // S and dP in two halves of the keys, each announced on its own, so
      // that each elementwise warpgroup starts as soon as its half is there
      // and frees it for the next block on its own
      auto issue_sdp = [&](int h, int kslot, int vslot) {
        const uint32_t sk = sK + kslot * C::kTileBytes, sv = sV + vslot * C::kTileBytes;
        if (h == 0) {
          mma_tk_half<DT, D, 0>(tS, tQ, sk, BC::kIdescSSHalf);
          mma_kk_half<DT, D, 0>(tDP, sdO, sv, BC::kIdescSSHalf);
        } else {
          mma_tk_half<DT, D, 1>(tS + 64, tQ, sk, BC::kIdescSSHalf);
          mma_kk_half<DT, D, 1>(tDP + 64, sdO, sv, BC::kIdescSSHalf);
        }
        mma_commit(smem_u32(&c->s_full[h]));
      };
      issue_sdp(0, ks, vs);
      issue_sdp(1, ks, vs);
      mma_commit(smem_u32(&c->v_empty[vs]));
      if (w.n == 1) mma_commit(smem_u32(&c->qd_empty));
      for (int j = 0; j < w.n && ok; ++j) {
        const int kcur = ks;
        if (j + 1 < w.n) {
          // S(j+1), dP(j+1) once the elementwise warps have read S(j), dP(j)
          next_slot(0, ks, kp);
          next_slot(1, vs, vp);
          ok = wait_bar(smem_u32(&c->k_full[ks]), kp, wc, 0x54) &&
               wait_bar(smem_u32(&c->v_full[vs]), vp, wc, 0x54) &&
               wait_bar(smem_u32(&c->sdp_free[0]), sf_w & 1u, wc, 0x53);
          if (!ok) break;
          tc_fence_after_sync();
          issue_sdp(0, ks, vs);
          if (!wait_bar(smem_u32(&c->sdp_free[1]), sf_w & 1u, wc, 0x53)) break;
          ++sf_w;
          tc_fence_after_sync();
          issue_sdp(1, ks, vs);
          mma_commit(smem_u32(&c->v_empty[vs]));
          if (j + 2 == w.n) mma_commit(smem_u32(&c->qd_empty));
        } else {
          // keep the sdp_free phases in step: the last read of the item
          ok = wait_bar(smem_u32(&c->sdp_free[0]), sf_w & 1u, wc, 0x53) &&
               wait_bar(smem_u32(&c->sdp_free[1]), sf_w & 1u, wc, 0x53);
          ++sf_w;
          if (!ok) break;
        }
        // dQ += dS(j) K_j, keys 0-63 as soon as their dS is there
        ok = wait_bar(smem_u32(&c->ds_full[0]), ds_w & 1u, wc, 0x55);
        if (ok && j == 0) {
          ok = wait_bar(smem_u32(&c->dq_empty), (dqe_w & 1u) ^ 1u, wc, 0x56);
          ++dqe_w;
        }
        if (!ok) break;
        tc_fence_after_sync();
        mma_tmn_half<DT, D, 0>(tDQ, tDS, sK + kcur * C::kTileBytes, BC::kIdescTS, j > 0);
        ok = wait_bar(smem_u32(&c->ds_full[1]), ds_w & 1u, wc, 0x58);
        ++ds_w;
        if (!ok) break;
        tc_fence_after_sync();
        mma_tmn_half<DT, D, 1>(tDQ, tDS, sK + kcur * C::kTileBytes, BC::kIdescTS, true);
        mma_commit(smem_u32(&c->ds_free));
        mma_commit(smem_u32(&c->k_empty[kcur]));
        if (j + 1 == w.n) mma_commit(smem_u32(&c->dq_full));
      }
    }
    mma_commit(smem_u32(&c->drain));
    volatile uint32_t never = 0;
    const WaitCtx wn{&never, p.timeout_ns, p.status, p.where};
    wait_bar(smem_u32(&c->drain), 0u, wn, 0x57);
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kBwdRegsElem));
    // ------------------------------------------------------------ elementwise
    // warpgroup `half` owns key columns [64 half, 64 half + 64) of S, dP
    // and dS, and dQ columns [d/2 half, d/2 half + d/2) in the epilogue
    const uint32_t wq = warp & 3u, half = (warp - 4u) >> 2;
    const int r = static_cast<int>(wq * 32u + lane);
    const uint32_t lane_off = (wq * 32u) << 16;
    const uint32_t tS = tbase + lane_off + BC::kDqS + 64 * half,
                   tDP = tbase + lane_off + BC::kDqDP + 64 * half,
                   tDS = tbase + lane_off + BC::kDqDS + 32 * half,
                   tDQ = tbase + lane_off + BC::kDqAcc + (D / 2) * half;
    const float sl2 = p.scale_log2;
    uint32_t sf_w = 0, dsf_w = 0, dqf_w = 0;
    bool first_ds = true;
    for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < p.n_items; ++rnd) {
      const int it = round_item(rnd, p.n_items);
      if (it < 0) continue;
      const BwdItem w = dq_item<CAUSAL>(it, p);
      const float2 lv = reinterpret_cast<const float2*>(p.ws)[static_cast<size_t>(w.bh) * p.Np +
                                                               w.tile * kBlock + r];
      const float lse2 = lv.x, Dr = lv.y;
      for (int j = 0; j < w.n; ++j) {
        if (!wait_bar_all(smem_u32(&c->s_full[half]), sf_w & 1u, wc, 0x61)) goto done;
        ++sf_w;
        tc_fence_after_sync();
        // keys >= N masked; causal: keys after the query on the diagonal
        int lim = p.N - j * kBlock - 64 * static_cast<int>(half);
        if (CAUSAL && j == w.tile) lim = min(lim, r + 1 - 64 * static_cast<int>(half));
        uint32_t dsp[32];
        {
          uint32_t v[128];  // S (this half's 64 keys), then dP
          tmem_ld_2x64_at(tS, tDP, v);
#pragma unroll
          for (int i = 0; i < 64; i += 2) {
            float p0 = ex2_approx(fmaf(__uint_as_float(v[i]), sl2, -lse2));
            float p1 = ex2_approx(fmaf(__uint_as_float(v[i + 1]), sl2, -lse2));
            if (i >= lim) p0 = 0.f;
            if (i + 1 >= lim) p1 = 0.f;
            const float ds0 = p0 * (__uint_as_float(v[64 + i]) - Dr);
            const float ds1 = p1 * (__uint_as_float(v[64 + i + 1]) - Dr);
            dsp[i / 2] = pack2<DT>(ds0, ds1);
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&c->sdp_free[half]));
        // dS(j-1) must have been consumed before its columns are rewritten
        if (!first_ds) {
          if (!wait_bar_all(smem_u32(&c->ds_free), dsf_w & 1u, wc, 0x62)) goto done;
          ++dsf_w;
          tc_fence_after_sync();
        }
        first_ds = false;
        tmem_st_x32(tDS, dsp);
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&c->ds_full[half]));
      }
      // epilogue: dQ * scale -> output rows (this half's columns)
      if (!wait_bar_all(smem_u32(&c->dq_full), dqf_w & 1u, wc, 0x63)) goto done;
      ++dqf_w;
      tc_fence_after_sync();
      {
        const int row = w.tile * kBlock + r;
        uint8_t* dst = static_cast<uint8_t*>(p.dq) +
                       ((static_cast<size_t>(w.bh) * p.N + row) * D + (D / 2) * half) *
                           C::T::kOutEsize;
#pragma unroll 1
        for (int cc = 0; cc < D / 2; cc += 32) {
          uint32_t v[32];
          tmem_ld_x32(tDQ + cc, v);
          if (row < p.N) store_row_chunk<DT>(dst + cc * C::T::kOutEsize, v, p.scale);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&c->dq_empty));
    }
  }
done:
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, 512);
  }
}

// ---------------------------------------------------------------------------
// dK / dV kernel

template <int NST>
struct DkvCtrl {
  uint64_t kv_full, kv_empty;
  uint64_t st_full[NST][2], st_empty[NST][2];  // stage i, query half h: Q_i, dO_i, (lse2, D)_i rows 64h .. 64h + 63
  uint64_t s_full[2];  // S^T(i), dP^T(i), queries 0-63 / 64-127, in TMEM (commit)
  uint64_t pds_full[2];  // P^T(i), dS^T(i), queries 0-63 / 64-127, in TMEM (4 warps each)
  uint64_t acc_full;   // last dV / dK MMA of the item done (commit)
  uint64_t acc_empty;  // epilogue read dV, dK             (8 warps)
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort;
};

template <int DT, int D, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dkv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                        const BwdParams p) {
  using C = Cfg<DT, D>;
  using BC = BwdCfg<DT, D>;
  constexpr int NST = BC::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* sbase = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sK = smem_u32(sbase), sV = sK + C::kTileBytes, sSt = sV + C::kTileBytes;
  uint8_t* st_base = sbase + 2 * C::kTileBytes;
  const uint32_t sEpi = sSt + NST * BC::kStageBytes;
  DkvCtrl<NST>* c = reinterpret_cast<DkvCtrl<NST>*>(sbase + 2 * C::kTileBytes +
                                                    NST * BC::kStageBytes + BC::kEpiBytes);
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&c->kv_full), 1);
    mbar_init(smem_u32(&c->kv_empty), 1);
    for (int s = 0; s < NST; ++s) {
      for (int h = 0; h < 2; ++h) {
        mbar_init(smem_u32(&c->st_full[s][h]), 1);
        mbar_init(smem_u32(&c->st_empty[s][h]), 1);
      }
    }
    mbar_init(smem_u32(&c->s_full[0]), 1);
    mbar_init(smem_u32(&c->s_full[1]), 1);
    mbar_init(smem_u32(&c->pds_full[0]), 4);
    mbar_init(smem_u32(&c->pds_full[1]), 4);
    mbar_init(smem_u32(&c->acc_full), 1);
    mbar_init(smem_u32(&c->acc_empty), 8);
    mbar_init(smem_u32(&c->drain), 1);
    c->abort = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&c->tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = c->tmem_base;
  const WaitCtx wc{&c->abort, p.timeout_ns, p.status, p.where};

  if (warp < 4) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kBwdRegsControl));
  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    uint32_t kv_uses = 0, loads = 0, round = 0;
    int st = 0;
    bool ok = true;
    for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < p.n_items && ok; ++rnd) {
      const int it = round_item(rnd, p.n_items);
      if (it < 0) continue;
      const BwdItem w = dkv_item<CAUSAL>(it, p);
      if (!wait_bar(smem_u32(&c->kv_empty), (kv_uses & 1u) ^ 1u, wc, 0x71)) break;
      mbar_arrive_expect_tx(smem_u32(&c->kv_full), 2 * C::kTileBytes);
      load_tile<DT, D>(sK, &tmK, w.tile * kBlock, w.bh, smem_u32(&c->kv_full));
      load_tile<DT, D>(sV, &tmV, w.tile * kBlock, w.bh, smem_u32(&c->kv_full));
      ++kv_uses;
      for (int i = 0; i < w.n; ++i) {
        const int qi = w.first + i;
        const uint32_t dst = sSt + st * BC::kStageBytes;
        for (int h = 0; h < 2 && ok; ++h) {
          if (!wait_bar(smem_u32(&c->st_empty[st][h]), (round & 1u) ^ 1u, wc, 0x72)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_u32(&c->st_full[st][h]);
          mbar_arrive_expect_tx(bar, BC::kStageBytes / 2);
          // rows 64h .. 64h + 63 of each 128-row box: the bottom half starts at
          // 8 KiB, a whole number of 1024-byte swizzle atoms, so the bytes are
          // those of the full box
#pragma unroll
          for (int b = 0; b < C::kNumBox; ++b) {
            tma_load_3d(dst + b * C::kBoxBytes + h * (C::kBoxBytes / 2), &tmQ, b * C::kBoxInner,
                        qi * kBlock + 64 * h, w.bh, bar);
            tma_load_3d(dst + C::kTileBytes + b * C::kBoxBytes + h * (C::kBoxBytes / 2), &tmdO,
                        b * C::kBoxInner, qi * kBlock + 64 * h, w.bh, bar);
          }
          bulk_load(dst + 2 * C::kTileBytes + h * (BC::kVecBytes / 2),
                    p.ws + (static_cast<size_t>(w.bh) * p.Np + qi * kBlock + 64 * h) * 2,
                    BC::kVecBytes / 2, bar);
        }
        if (!ok) break;
        ++loads;
        if (++st == NST) {
          st = 0;
          ++round;
        }
      }
    }
    volatile uint32_t never = 0;
    const WaitCtx wn{&never, p.timeout_ns, p.status, p.where};
    for (int s = 0; s < NST; ++s) {
      const uint32_t uses = loads / NST + (static_cast<uint32_t>(s) < loads % NST ? 1u : 0u);
      for (int h = 0; h < 2 && uses; ++h)
        wait_bar(smem_u32(&c->st_full[s][h]), (uses - 1u) & 1u, wn, 0x73);
    }
    if (kv_uses) wait_bar(smem_u32(&c->kv_full), (kv_uses - 1u) & 1u, wn, 0x74);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA
    uint32_t kv_w = 0, pds_w = 0, ae_w = 0, round = 0;
    int st = 0;
    const uint32_t tS = tbase + BC::kKvS, tDP = tbase + BC::kKvDP, tDV = tbase + BC::kKvDV,
                   tDK = tbase + BC::kKvDK;
    bool ok = true;
    for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < p.n_items && ok; ++rnd) {
      const int it = round_item(rnd, p.n_items);
      if (it < 0) continue;
      const BwdItem w = dkv_item<CAUSAL>(it, p);
      ok = wait_bar(smem_u32(&c->kv_full), kv_w & 1u, wc, 0x81) &&
           wait_bar(smem_u32(&c->st_full[st][0]), round & 1u, wc, 0x82);
      ++kv_w;
      if (!ok) break;
      tc_fence_after_sync();
      // S^T = K Q_i^T and dP^T = V dO_i^T in two halves of the queries
      // (columns 0-63 and 64-127).  Half h's P^T / dS^T are packed into the
      // first 32 columns of its own S^T / dP^T columns, so the next block's
      // half h may be issued right after this block's products of half h:
      // the two halves alternate on the tensor pipe while the other half's
      // elementwise warps work.
      auto issue_sdp = [&](int h, uint32_t sq) {
        if (h == 0) {
          mma_kk_half<DT, D, 0>(tS, sK, sq, BC::kIdescSSHalf);
          mma_kk_half<DT, D, 0>(tDP, sV, sq + C::kTileBytes, BC::kIdescSSHalf);
        } else {
          mma_kk_half<DT, D, 1>(tS + 64, sK, sq, BC::kIdescSSHalf);
          mma_kk_half<DT, D, 1>(tDP + 64, sV, sq + C::kTileBytes, BC::kIdescSSHalf);
        }
        mma_commit(smem_u32(&c->s_full[h]));
      };
      {
        const uint32_t sq = sSt + st * BC::kStageBytes;
        issue_sdp(0, sq);
        if (!wait_bar(smem_u32(&c->st_full[st][1]), round & 1u, wc, 0x82)) break;
        tc_fence_after_sync();
        issue_sdp(1, sq);
        // K and V serve only S^T and dP^T: free them for the next item's
        // tiles once the item's last S^T and dP^T are issued
        if (w.n == 1) mma_commit(smem_u32(&c->kv_empty));
      }
      for (int i = 0; i < w.n && ok; ++i) {
        const uint32_t sq = sSt + st * BC::kStageBytes;
        const bool have_next = i + 1 < w.n;
        const int nst = st + 1 == NST ? 0 : st + 1;
        const uint32_t nround = st + 1 == NST ? round + 1 : round;
        const uint32_t sn = sSt + nst * BC::kStageBytes;
        // queries 0-63: dV += P^T dO_i, dK += dS^T Q_i
        ok = wait_bar(smem_u32(&c->pds_full[0]), pds_w & 1u, wc, 0x83);
        if (ok && i == 0) {
          ok = wait_bar(smem_u32(&c->acc_empty), (ae_w & 1u) ^ 1u, wc, 0x84);
          ++ae_w;
        }
        if (!ok) break;
        tc_fence_after_sync();
        mma_tmn_part<DT, D, 0>(tDV, tS, sq + C::kTileBytes, BC::kIdescTS, i > 0);
        mma_tmn_part<DT, D, 0>(tDK, tDP, sq, BC::kIdescTS, i > 0);
        mma_commit(smem_u32(&c->st_empty[st][0]));
        if (have_next) {
          if (!wait_bar(smem_u32(&c->st_full[nst][0]), nround & 1u, wc, 0x82)) break;
          tc_fence_after_sync();
          issue_sdp(0, sn);
        }
        // queries 64-127
        ok = wait_bar(smem_u32(&c->pds_full[1]), pds_w & 1u, wc, 0x86);
        ++pds_w;
        if (!ok) break;
        tc_fence_after_sync();
        mma_tmn_part<DT, D, 1>(tDV, tS + 64, sq + C::kTileBytes, BC::kIdescTS, true);
        mma_tmn_part<DT, D, 1>(tDK, tDP + 64, sq, BC::kIdescTS, true);
        mma_commit(smem_u32(&c->st_empty[st][1]));
        st = nst;
        round = nround;
        if (have_next) {
          if (!wait_bar(smem_u32(&c->st_full[st][1]), round & 1u, wc, 0x82)) break;
          tc_fence_after_sync();
          issue_sdp(1, sn);
          if (i + 2 == w.n) mma_commit(smem_u32(&c->kv_empty));
        } else {
          mma_commit(smem_u32(&c->acc_full));
        }
      }
    }
    mma_commit(smem_u32(&c->drain));
    volatile uint32_t never = 0;
    const WaitCtx wn{&never, p.timeout_ns, p.status, p.where};
    wait_bar(smem_u32(&c->drain), 0u, wn, 0x85);
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kBwdRegsElem));
    // ------------------------------------------------------------ elementwise
    // warpgroup `half` owns query columns [64 half, 64 half + 64) of S^T and
    // dP^T; their P^T and dS^T go, packed, to the first 32 of those columns,
    // and dV / dK columns [d/2 half, d/2 half + d/2) are its share of the
    // epilogue.
    const uint32_t wq = warp & 3u, half = (warp - 4u) >> 2;
    const int r = static_cast<int>(wq * 32u + lane);  // key row within the tile
    const uint32_t lane_off = (wq * 32u) << 16;
    const uint32_t tS = tbase + lane_off + BC::kKvS, tDP = tbase + lane_off + BC::kKvDP,
                   tDV = tbase + lane_off + BC::kKvDV + (D / 2) * half,
                   tDK = tbase + lane_off + BC::kKvDK + (D / 2) * half;
    const float sl2 = p.scale_log2;
    uint32_t sf_w = 0, af_w = 0, round = 0;
    int st = 0;
    for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < p.n_items; ++rnd) {
      const int it = round_item(rnd, p.n_items);
      if (it < 0) continue;
      const BwdItem w = dkv_item<CAUSAL>(it, p);
      for (int i = 0; i < w.n; ++i) {
        const int qi = w.first + i;
        // S^T(i), dP^T(i) in TMEM, and the stage's (lse2, D) rows landed
        // (observed here, not only through the MMA thread)
        if (!wait_bar_all(smem_u32(&c->s_full[half]), sf_w & 1u, wc, 0x91) ||
            !wait_bar_all(smem_u32(&c->st_full[st][half]), round & 1u, wc, 0x93))
          goto done;
        ++sf_w;
        tc_fence_after_sync();
        const float2* vec =
            reinterpret_cast<const float2*>(st_base + st * BC::kStageBytes + 2 * C::kTileBytes);
        // causal: query column cq is visible to this key iff cq >= r on the
        // diagonal tile
        const int qlim = (CAUSAL && qi == w.tile) ? r : 0;
        uint32_t pp[32], dd[32];
        {
          uint32_t v[128];  // S^T (this half's 64 queries), then dP^T
          tmem_ld_2x64_at(tS + 64 * half, tDP + 64 * half, v);
          const float4* vec4 = reinterpret_cast<const float4*>(vec) + 32 * half;
#pragma unroll
          for (int i2 = 0; i2 < 64; i2 += 2) {
            const int cq = 64 * static_cast<int>(half) + i2;
            const float4 lv = vec4[i2 / 2];  // (lse2, D) of query columns cq, cq + 1
            float p0 = ex2_approx(fmaf(__uint_as_float(v[i2]), sl2, -lv.x));
            float p1 = ex2_approx(fmaf(__uint_as_float(v[i2 + 1]), sl2, -lv.z));
            if (cq < qlim) p0 = 0.f;
            if (cq + 1 < qlim) p1 = 0.f;
            pp[i2 / 2] = pack2<DT>(p0, p1);
            dd[i2 / 2] = pack2<DT>(p0 * (__uint_as_float(v[64 + i2]) - lv.y),
                                   p1 * (__uint_as_float(v[64 + i2 + 1]) - lv.w));
          }
        }
        // P^T over this half's S^T columns (already read), dS^T over dP^T
        tmem_st_x32(tS + 64 * half, pp);
        tmem_st_x32(tDP + 64 * half, dd);
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&c->pds_full[half]));
        if (++st == NST) {
          st = 0;
          ++round;
        }
      }
      // epilogue: dV and dK * scale -> output rows (this half's columns)
      if (!wait_bar_all(smem_u32(&c->acc_full), af_w & 1u, wc, 0x92)) goto done;
      ++af_w;
      tc_fence_after_sync();
      {
        // this warp's 32 rows, coalesced through its staging area
        const int row0 = w.tile * kBlock + static_cast<int>(wq) * 32;
        const size_t off =
            ((static_cast<size_t>(w.bh) * p.N + row0) * D + (D / 2) * half) * C::T::kOutEsize;
        uint8_t* dv = static_cast<uint8_t*>(p.dv) + off;
        uint8_t* dk = static_cast<uint8_t*>(p.dk) + off;
        const int n_valid = p.N - row0;
        const size_t pitch = static_cast<size_t>(D) * C::T::kOutEsize;
        const uint32_t stage = sEpi + (warp - 4u) * 2048u;
#pragma unroll 1
        for (int cc = 0; cc < D / 2; cc += 32) {
          uint32_t v[32];
          tmem_ld_x32(tDV + cc, v);
          store_rows_staged<DT>(dv + cc * C::T::kOutEsize, pitch, n_valid, v, 1.0f, stage, lane);
          tmem_ld_x32(tDK + cc, v);
          store_rows_staged<DT>(dk + cc * C::T::kOutEsize, pitch, n_valid, v, p.scale, stage, lane);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&c->acc_empty));
    }
    (void)round;
  }
done:
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, 512);
  }
  // this grid completes only after the dQ grid before it (a no-op when it
  // was launched without programmatic serialization)
  if (threadIdx.x == 0) griddep_wait();
}

}  // namespace wsattn

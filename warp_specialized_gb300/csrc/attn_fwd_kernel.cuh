// attn_fwd_kernel.cuh - the warp-specialised fused attention forward kernel
// for sm_103a (GB300).
//
// What it computes, per (b, h) and query row i (natural-log LSE):
//   S = scale * Q K^T, masked (-inf) where key > query when causal and
//   where key >= N; O = softmax(S) V; LSE = log sum exp S.
// It walks the key/value blocks j with the online softmax of the
// "Warp specialization" concept card (wikillm), section "Implementation
// sketch": running row max m and row sum l, the old sum and output rescaled
// by exp(m_old - m_new) (the card's form, not the inverse factor it
// rejects), O / l and m + log l at the end.
//
// Schedule (GB300 form of the producer/consumer split of the card's
// "Variants" section and of the tekromancy page, sections 1-4):
//   warp 0        producer: one thread streams Q tiles and the K_j / V_j
//                 tiles into a shared-memory ring with TMA; every ring slot
//                 has a "full" mbarrier (TMA transaction bytes) and an
//                 "empty" mbarrier (released by the MMA commit).
//   warp 1        MMA issuer: one thread issues tcgen05.mma; S = Q K_j^T
//                 lands in Tensor Memory, O += P V_j accumulates there with
//                 P read from Tensor Memory.
//   warps 4-7     softmax of query tile A, one thread per row (lane) of the
//                 128-row tile: row max, exp2, row sum, P written back over
//                 S in Tensor Memory (no shuffles: a row lives in one
//                 thread, spheron page, section on Blackwell).
//   warps 8-11    softmax of query tile B.  The MMA thread alternates
//                 between the two tiles (S_A, S_B, PV_A, S_A', PV_B, S_B',
//                 ...), so the exponentials of one tile overlap the matrix
//                 products of the other: the two-consumer pingpong of the
//                 card's "Pingpong scheduling" variant, with the turn-taking
//                 done by the MMA issue order instead of named barriers.
//                 Each softmax hands its P over in two halves of 64 keys,
//                 and the MMA thread issues P V_j for the first half while
//                 the second half's exponentials are computed.
//   warps 12-15   correction and epilogue: rescales O in Tensor Memory by
//                 exp2(m_old - m_new) when a row max grew, and at the end
//                 writes O / l and lets the softmax warps write LSE.
// The grid is persistent (one CTA per SM); CTAs walk a static list of
// (head, pair of query tiles) work items.  With the causal mask blocks
// above the diagonal are never loaded or multiplied, and the list starts
// with the items that have the most blocks.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx_sm103.cuh"

namespace wsattn {

// status codes mirrored from attn.h (kept numerically identical)
constexpr unsigned kStatusTimeout = 6u;

// element types: 1 fp16, 2 bf16, 3 e4m3 (fp32 inputs use attn_fwd_fp32.cuh)
template <int DT>
struct DTypeTraits;
template <>
struct DTypeTraits<1> {
  static constexpr int kEsize = 2;
  static constexpr uint32_t kFmt = 0;  // f16
  static constexpr MmaKind kKind = MmaKind::kF16;
  static constexpr int kOutEsize = 2;
};
template <>
struct DTypeTraits<2> {
  static constexpr int kEsize = 2;
  static constexpr uint32_t kFmt = 1;  // bf16
  static constexpr MmaKind kKind = MmaKind::kF16;
  static constexpr int kOutEsize = 2;
};
template <>
struct DTypeTraits<3> {
  static constexpr int kEsize = 1;
  static constexpr uint32_t kFmt = 0;  // e4m3
  static constexpr MmaKind kKind = MmaKind::kF8F6F4;
  static constexpr int kOutEsize = 2;  // bf16 output
};

constexpr int kThreads = 512;
constexpr int kBlock = 128;            // query rows per tile = keys per block
constexpr int kSmemLimit = 232448;     // opt-in shared memory per block on sm_100/sm_103
constexpr int kMaxSlots = 8;

template <int DT, int D>
struct Cfg {
  using T = DTypeTraits<DT>;
  static constexpr int kEsize = T::kEsize;
  static constexpr int kRowBytes = D * kEsize;
  static constexpr int kBoxInner = 128 / kEsize;     // elements per 128-byte swizzled row
  static constexpr int kNumBox = kRowBytes / 128;    // TMA boxes per tile
  static constexpr int kBoxBytes = kBlock * 128;     // 16 KiB
  static constexpr int kTileBytes = kNumBox * kBoxBytes;
  // two query tiles per CTA when both S and O of both fit in Tensor Memory
  // (2 * (128 + D) <= 512 columns) and in shared memory
  static constexpr int kNQT = (D <= 128 && kTileBytes <= 32768) ? 2 : 1;
  // d = 256 (one query tile per CTA): Q is copied into Tensor Memory once per
  // item (tcgen05.cp) and taken from there as the A operand of S = Q K^T,
  // and the Q tile's shared memory joins the K/V ring, which then holds
  // three 64 KiB tiles instead of two, so that K_{j+1} loads while K_j and
  // V_j are in use.  (TMEM: S 128 + O 256 + Q 128 = 512 columns.)
  static constexpr bool kQTmem = D == 256;
  static constexpr int kQBufTiles = kQTmem ? 0 : kNQT;  // Q tiles in shared memory
  // issue the next work item's first S behind this item's last P V
  static constexpr bool kEarlyS0 = !kQTmem;
  // epilogue: read and pack a whole 64-column box of O before waiting for
  // the staging box (measured +3% with e4m3; at 16 bits the extra live
  // registers spill and it loses up to 1%)
  static constexpr bool kEpiPrefetch = DT == 3;
  static constexpr int kMiscBytes = 1024 /*alignment*/ + 512 /*barriers*/ +
                                    2 * kBlock * 4 /*alpha*/ + 2 * 2 * kBlock * 4 /*1/l*/;
  // staging box of the output: 128 rows x 128 bytes (64 columns of 16 bits)
  static constexpr int kStageBytes = kBlock * 128;
  // e4m3 has shared memory to spare for a second box, so that one box is
  // written while the store of the other still reads it (measured +0.7%,
  // causal +1.3%); at 16 bits a second box would cost a K/V ring slot
  static constexpr int kStageBufs = DT == 3 ? 2 : 1;
  static constexpr int kStageTotal = kStageBufs * kStageBytes;
  static constexpr int kSlotsFit =
      (kSmemLimit - kMiscBytes - kStageTotal - kQBufTiles * kTileBytes) / kTileBytes;
  static constexpr int kSlots = kSlotsFit > kMaxSlots ? kMaxSlots : kSlotsFit;
  static_assert(kSlots >= 2, "the K/V ring needs at least two slots");
  // Ring stages.  With four or more slots a stage is a pair of slots that
  // holds V_j and the K tile that follows it in the stream (K_{j+1}, or
  // K_0 of the next item), filled and released as one: the MMA thread
  // waits once and releases once per block.  With two slots (d = 256) every
  // tile is a stage of its own, so that K_{j+1} can load while V_j is used.
  static constexpr bool kPair = kSlots >= 4;
  static constexpr int kStages = kPair ? kSlots / 2 : kSlots;
  static __host__ __device__ constexpr int v_slot(int st) { return kPair ? 2 * st : st; }
  static __host__ __device__ constexpr int k_slot(int st) { return kPair ? 2 * st + 1 : st; }
  // S lookahead (defined below) keeps a second alpha array right after the
  // control block
  static constexpr int kAlphaOddBytes = (kNQT == 2 && 3 * kBlock + 2 * D <= 512) ? 2 * kBlock * 4 : 0;
  static constexpr int kSmemBytes =
      kMiscBytes + (kQBufTiles + kSlots) * kTileBytes + kStageTotal + kAlphaOddBytes;
  // a piece's (O, m, l) in the tail launch's workspace: O as [D / 4][128]
  // float4 (four columns of one row per 16 bytes, the 128 rows of a column
  // quad contiguous, so that a warp's 16-byte accesses are contiguous),
  // then m[128], l[128]
  static constexpr int kPartFloats = kBlock * (D + 2);
  static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
  static_assert(kNQT * kTileBytes % 1024 == 0 && kTileBytes % 1024 == 0, "tile alignment");
  static_assert(kRowBytes % 128 == 0, "head dim must fill whole 128-byte swizzle rows");

  // tensor-core shapes: M = 128 rows, K per instruction = 32 bytes
  static constexpr int kKPerMma = 32 / kEsize;
  static constexpr int kNumQKMma = kRowBytes / 32;
  static constexpr int kNumPVMma = kBlock / kKPerMma;
  static constexpr int kPCols = kBlock * kEsize / 4;  // TMEM columns holding P
  static constexpr uint32_t kIdescQK = make_idesc(T::kFmt, T::kFmt, false, kBlock, kBlock);
  static constexpr uint32_t kIdescPV = make_idesc(T::kFmt, T::kFmt, true, D, kBlock);

  // S lookahead (two query tiles with D <= 64): a third S buffer fits in
  // Tensor Memory (3 x 128 + 2 x D <= 512 columns), so the S buffers are
  // used in turn, in the order the S products are issued, and a tile's
  // S(j + 1) goes out before its P(j) V instead of after it: the softmax
  // then moves on to block j + 1 without waiting for P(j) V and S(j + 1) to
  // pass through the tensor pipe.  Barriers that could otherwise complete
  // a second phase before their waiter has seen the first (s_full, the
  // second half of p_full, and alpha's sc_full with alpha itself) are kept
  // in two sets used in turn.
  static constexpr bool kSLook = kNQT == 2 && 3 * kBlock + 2 * D <= 512;
  static constexpr int kSBufs = kSLook ? 3 : kNQT;
  static constexpr int kBarSets = kSLook ? 2 : 1;
  static_assert(kAlphaOddBytes == (kSLook ? 2 * kBlock * 4 : 0), "second alpha array");

  // Tensor Memory columns
  static constexpr uint32_t kTmemCols = 512;
  static __host__ __device__ constexpr uint32_t s_col(int t) { return t * kBlock; }
  static __host__ __device__ constexpr uint32_t s_buf_col(uint32_t b) { return b * kBlock; }
  static __host__ __device__ constexpr uint32_t o_col(int t) { return kSBufs * kBlock + t * D; }
  // Q in Tensor Memory (kQTmem): 16-bit pairs, D / 2 columns
  static __host__ __device__ constexpr uint32_t q_col() { return kNQT * (kBlock + D); }
  static_assert(!kQTmem || (kNQT == 1 && q_col() + D / 2 <= 512), "Tensor Memory budget (Q)");
  static_assert(kSBufs * kBlock + kNQT * D <= 512, "Tensor Memory budget");
};

struct AttnParams {
  void* o;
  float* lse;
  int N;
  int BH;
  int n_qt;       // query tiles per head
  int n_pairs;    // groups of kNQT query tiles per head (one work item each)
  int n_items;    // BH * n_pairs
  int nkv;        // key blocks per head
  float scale_log2;   // scale * (q, k descales) * log2(e)
  float out_scale;    // v descale (1 for non-fp8)
  // e4m3 with block scales: one fp32 scale per 128-row tile of Q and of K,
  // [B*H, n_qt] (null for per-tensor descales)
  const float* q_block_scale;
  const float* k_block_scale;
  unsigned long long timeout_ns;
  // library-owned device words: the first error seen by any kernel, and a
  // code saying which wait ran out (role * 16 + barrier kind)
  unsigned int* status;
  unsigned int* where;
  // the tail launch (attn_fwd_tail.cuh): items [tail_start, tail_start +
  // tail_items) with tail_units key blocks in all, shared out over the grid;
  // the pieces' flags ([tail_items][2], zeroed before the launch) and
  // results ([G][2][kNQT] of kPartFloats) in the caller's workspace
  int tail_start;
  int tail_items;
  int tail_ramp;   // extra units of the first tail CTA (see tail_range_start)
  int tail_units;
  unsigned int* flags;
  float* part;
};

// One work item: kNQT adjacent query tiles of one head, walked over the
// key/value blocks they need.
struct Item {
  int bh;
  int qt0;
  int n[2];    // key blocks of each query tile (0: no such tile)
  int nmax;
};

template <int NQT, bool CAUSAL>
__device__ __forceinline__ Item decode_item(int it, const AttnParams& p) {
  Item r;
  int pair;
  if (CAUSAL) {  // most blocks first
    pair = p.n_pairs - 1 - it / p.BH;
    r.bh = it % p.BH;
  } else {       // head-major, so that a head's K/V stay hot in L2
    r.bh = it / p.n_pairs;
    pair = it % p.n_pairs;
  }
  r.qt0 = pair * NQT;
  r.nmax = 0;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qt = r.qt0 + t;
    const int n = CAUSAL ? min(qt + 1, p.nkv) : p.nkv;
    r.n[t] = t < NQT ? n : 0;
    r.nmax = max(r.nmax, r.n[t]);
  }
  return r;
}

// Static persistent schedule: in round r, CTA c of G takes item r*G + c
// on even rounds and r*G + (G-1-c) on odd ones, so that causal items of
// decreasing size even out.
__device__ __forceinline__ int snake_item(int r, int g, int c, int n_items) {
  const int it = r * g + ((r & 1) ? g - 1 - c : c);
  return it < n_items ? it : -1;
}
__device__ __forceinline__ int round_item(int r, int n_items) {
  return snake_item(r, static_cast<int>(gridDim.x), static_cast<int>(blockIdx.x), n_items);
}

// The item this CTA takes after the one of round rnd, if any.
template <int NQT, bool CAUSAL>
__device__ __forceinline__ bool next_item(int rnd, const AttnParams& p, Item& wn) {
  for (int r2 = rnd + 1; r2 * static_cast<int>(gridDim.x) < p.n_items; ++r2) {
    const int i2 = round_item(r2, p.n_items);
    if (i2 < 0) continue;
    wn = decode_item<NQT, CAUSAL>(i2, p);
    return true;
  }
  return false;
}

// Position in the K/V ring: stage index and how many times it wrapped.
struct RingPos {
  int st = 0;
  uint32_t round = 0;
  template <int NST>
  __device__ __forceinline__ void next(int& s, uint32_t& parity) {
    s = st;
    parity = round & 1u;
    if (++st == NST) {
      st = 0;
      ++round;
    }
  }
};

// Shared-memory control block (after the tiles).
template <int NSLOT>
struct Ctrl {
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[NSLOT], kv_empty[NSLOT];
  uint64_t s_full[2][2];  // S_t(j) in TMEM, [tile][set]  (MMA commit)
  // [t][0]: P_t(j) keys 0-63 in TMEM and O_t rescaled for block j (4
  // softmax + 4 correction warps); [t][1 + set]: P_t(j) keys 64-127 in
  // TMEM (4 softmax warps)
  uint64_t p_full[2][3];
  uint64_t sc_full[2];   // alpha_t(j) in smem        (4 softmax warps)
  uint64_t o_full[2];    // P_t V of the item's last block done (MMA commit)
  uint64_t pv_done[2];   // S lookahead: P_t V of a block that is not the last (MMA commit)
  uint64_t drain;        // all MMAs done             (MMA commit)
  uint32_t tmem_base;
  uint32_t abort;        // set when a wait in this CTA ran out
  float alpha[2][kBlock];
  float inv_l[2][2][kBlock];  // [item parity][tile][row]
  // S lookahead: alpha of a tile's blocks of odd count goes to a second
  // array (alpha_odd, right after this block) under a barrier of its own,
  // so that the softmax never waits for the correction warps' read of the
  // previous alpha.  (Placed here, after the arrays: measured 4% faster at
  // d = 64 than beside the other barriers.)
  uint64_t sc_full_odd[2];
};

// The second alpha array of the S lookahead, [tile][row], right after the
// control block (counted in Cfg::kSmemBytes).
template <class CtrlT>
__device__ __forceinline__ float* alpha_odd(CtrlT* c) {
  return reinterpret_cast<float*>(c + 1);
}

// The alpha barrier of tile t's k-th block (from 0), and its phase parity:
// with the S lookahead two barriers used in turn, else one.
template <bool LOOK, class CtrlT>
__device__ __forceinline__ uint32_t sc_bar(CtrlT* c, int t, uint32_t k) {
  return smem_u32(LOOK && (k & 1u) ? &c->sc_full_odd[t] : &c->sc_full[t]);
}
template <bool LOOK>
__device__ __forceinline__ uint32_t sc_par(uint32_t k) {
  return LOOK ? ((k >> 1) & 1u) : (k & 1u);
}

// The k-th use (from 0) of a barrier kept in `sets` copies used in turn:
// which copy, and the parity of its phase.
__device__ __forceinline__ uint32_t bar_set(uint32_t k, int sets) {
  return sets == 2 ? (k & 1u) : 0u;
}
__device__ __forceinline__ uint32_t bar_par(uint32_t k, int sets) {
  return sets == 2 ? ((k >> 1) & 1u) : (k & 1u);
}

// Bounded wait: true when the phase with `parity` has completed; false when
// another thread of this CTA gave up or the limit ran out (then the status
// word records a timeout and `where`).
struct WaitCtx {
  volatile uint32_t* abort;
  unsigned long long limit_ns;
  unsigned int* status;
  unsigned int* where;
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const WaitCtx& wc,
                                        unsigned where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*wc.abort) return false;
    if (global_timer_ns() - t0 > wc.limit_ns) {
      *wc.abort = 1u;
      atomicCAS(wc.status, 0u, kStatusTimeout);
      atomicExch(wc.where, where);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// producer: Q tiles, then the K and V tiles through the ring

template <int DT, int D, bool CAUSAL>
__device__ void role_producer(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                              const CUtensorMap* tmV, uint8_t* sbase,
                              Ctrl<Cfg<DT, D>::kSlots>* c, const AttnParams& p) {
  using C = Cfg<DT, D>;
  const WaitCtx wc{&c->abort, p.timeout_ns, p.status, p.where};
  const uint8_t* sq = sbase;
  const uint32_t skv = smem_u32(sbase + C::kQBufTiles * C::kTileBytes);
  uint32_t q_uses[2] = {0, 0};
  RingPos ring;
  uint32_t stages = 0;  // ring stages filled
  bool ok = true;

  // One ring stage: V rows [vrow, vrow + 128) and / or K rows [krow, ...)
  // of heads vbh / kbh (a negative row: no such tile in this stage).
  auto fill = [&](int vrow, int vbh, int krow, int kbh) -> bool {
    int st;
    uint32_t par;
    ring.next<C::kStages>(st, par);
    if (!wait_bar(smem_u32(&c->kv_empty[st]), par ^ 1u, wc, 0x02)) return false;
    const uint32_t full = smem_u32(&c->kv_full[st]);
    mbar_arrive_expect_tx(full, ((vrow >= 0) + (krow >= 0)) * C::kTileBytes);
    if (vrow >= 0) {
      const uint32_t dst = skv + C::v_slot(st) * C::kTileBytes;
#pragma unroll
      for (int b = 0; b < C::kNumBox; ++b)
        tma_load_3d(dst + b * C::kBoxBytes, tmV, b * C::kBoxInner, vrow, vbh, full);
    }
    if (krow >= 0) {
      const uint32_t dst = skv + C::k_slot(st) * C::kTileBytes;
#pragma unroll
      for (int b = 0; b < C::kNumBox; ++b)
        tma_load_3d(dst + b * C::kBoxBytes, tmK, b * C::kBoxInner, krow, kbh, full);
    }
    ++stages;
    return true;
  };

  bool k0_loaded = false;  // this item's K_0 went out with the previous item's last V
  for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < p.n_items && ok; ++rnd) {
    const int it = round_item(rnd, p.n_items);
    if (it < 0) continue;
    const Item w = decode_item<C::kNQT, CAUSAL>(it, p);
    Item wn;
    const bool has_next = next_item<C::kNQT, CAUSAL>(rnd, p, wn);
    if constexpr (C::kQTmem) {
      // the item's Q tile through the ring, ahead of its first K
      int st;
      uint32_t par;
      ring.next<C::kStages>(st, par);
      if (!wait_bar(smem_u32(&c->kv_empty[st]), par ^ 1u, wc, 0x02)) break;
      const uint32_t full = smem_u32(&c->kv_full[st]);
      mbar_arrive_expect_tx(full, C::kTileBytes);
      const uint32_t dst = skv + C::k_slot(st) * C::kTileBytes;
#pragma unroll
      for (int b = 0; b < C::kNumBox; ++b)
        tma_load_3d(dst + b * C::kBoxBytes, tmQ, b * C::kBoxInner, w.qt0 * kBlock, w.bh, full);
      ++stages;
    }
#pragma unroll
    for (int t = 0; t < (C::kQTmem ? 0 : C::kNQT); ++t) {
      const uint32_t full = smem_u32(&c->q_full[t]);
      if (!wait_bar(smem_u32(&c->q_empty[t]), (q_uses[t] & 1u) ^ 1u, wc, 0x01)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(full, C::kTileBytes);
      const uint32_t dst = smem_u32(sq + t * C::kTileBytes);
#pragma unroll
      for (int b = 0; b < C::kNumBox; ++b)
        tma_load_3d(dst + b * C::kBoxBytes, tmQ, b * C::kBoxInner, (w.qt0 + t) * kBlock, w.bh, full);
      ++q_uses[t];
    }
    if constexpr (C::kPair) {
      // stages (V_j, next K): K_{j+1}, or K_0 of the next item
      if (ok && !k0_loaded) ok = fill(-1, 0, 0, w.bh);
      for (int j = 0; j < w.nmax && ok; ++j) {
        if (j + 1 < w.nmax)
          ok = fill(j * kBlock, w.bh, (j + 1) * kBlock, w.bh);
        else
          ok = fill(j * kBlock, w.bh, has_next ? 0 : -1, has_next ? wn.bh : 0);
      }
      k0_loaded = has_next;
    } else {
      // one tile per stage: K_j, then V_j
      for (int j = 0; j < w.nmax && ok; ++j) {
        ok = fill(-1, 0, j * kBlock, w.bh);
        if (ok) ok = fill(j * kBlock, w.bh, -1, 0);
      }
    }
  }
  // Never leave a copy in flight: wait until the last fill of every stage
  // and of every Q tile has landed (immediate on the normal path).
  for (int st = 0; st < C::kStages; ++st) {
    const uint32_t uses =
        stages / C::kStages + (static_cast<uint32_t>(st) < stages % C::kStages ? 1u : 0u);
    if (uses) {
      volatile uint32_t never = 0;
      const WaitCtx wc_never{&never, p.timeout_ns, p.status, p.where};
      wait_bar(smem_u32(&c->kv_full[st]), (uses - 1u) & 1u, wc_never, 0x03);
    }
  }
  for (int t = 0; t < C::kNQT; ++t) {
    if (q_uses[t]) {
      volatile uint32_t never = 0;
      const WaitCtx wc_never{&never, p.timeout_ns, p.status, p.where};
      wait_bar(smem_u32(&c->q_full[t]), (q_uses[t] - 1u) & 1u, wc_never, 0x04);
    }
  }
}

// ---------------------------------------------------------------------------
// MMA issuer (one thread)

// A shared-memory descriptor moved on by off16 (a byte offset / 16); the
// start-address field cannot carry into the upper word, since shared
// addresses stay below 2^18 bytes.
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t off16) {
  return (d & 0xFFFFFFFF00000000ull) | static_cast<uint32_t>(static_cast<uint32_t>(d) + off16);
}

// A 128-row, K-major tile (Q) from shared memory into Tensor Memory, in the
// layout a tcgen05.mma A operand takes there: row r in lane r, elements
// (2m, 2m + 1) in column m.  One 32-byte K slice per copy, the slices
// exactly those an SS MMA would read for each K step.
template <int DT, int D>
__device__ __forceinline__ void copy_tile_to_tmem(uint32_t t, uint32_t s) {
  using C = Cfg<DT, D>;
  const uint64_t a0 = make_sdesc_sw128(s, 16, 1024);
#pragma unroll
  for (int k = 0; k < C::kNumQKMma; ++k) {
    const uint32_t off = ((k >> 2) * C::kBoxBytes + (k & 3) * 32) >> 4;
    tmem_cp_128x256b(t + k * 8, a0 + off);
  }
}

// A x B^T with A (128 rows, K-major) in Tensor Memory and B K-major in
// shared memory (S = Q K^T with Q copied into TMEM)
template <int DT, int D>
__device__ __forceinline__ void mma_tk(uint32_t d_tmem, uint32_t a_tmem, uint32_t sb,
                                       uint32_t idesc) {
  using C = Cfg<DT, D>;
  const uint64_t b0 = make_sdesc_sw128(sb, 16, 1024);
#pragma unroll
  for (int k = 0; k < C::kNumQKMma; ++k) {
    const uint32_t off = ((k >> 2) * C::kBoxBytes + (k & 3) * 32) >> 4;
    mma_ts<C::T::kKind>(d_tmem, a_tmem + k * 8, b0 + off, idesc, k > 0 ? 1u : 0u);
  }
}

template <int DT, int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t sq, uint32_t sk) {
  using C = Cfg<DT, D>;
  const uint64_t a0 = make_sdesc_sw128(sq, 16, 1024);
  const uint64_t b0 = make_sdesc_sw128(sk, 16, 1024);
#pragma unroll
  for (int k = 0; k < C::kNumQKMma; ++k) {
    const uint32_t off = ((k >> 2) * C::kBoxBytes + (k & 3) * 32) >> 4;
    mma_ss<C::T::kKind>(d_tmem, desc_add(a0, off), desc_add(b0, off), C::kIdescQK,
                        k > 0 ? 1u : 0u);
  }
}

// O_t += P_t V_j over one half of the block's keys (HALF 0: keys 0-63, whose
// P the softmax hands over first; HALF 1: keys 64-127).
template <int DT, int D, int HALF>
__device__ __forceinline__ void issue_pv_half(uint32_t d_tmem, uint32_t p_tmem, uint32_t sv,
                                              bool accumulate) {
  using C = Cfg<DT, D>;
  constexpr int kHalf = C::kNumPVMma / 2;
  static_assert(C::kNumPVMma % 2 == 0, "PV splits into two key halves");
  // V is [keys, d] with d contiguous: an MN-major B operand.  Each 8-key
  // group is one 1024-byte swizzle atom (SBO); 128-byte column blocks of d
  // are one TMA box apart (LBO).
  const uint64_t b0 = make_sdesc_sw128(sv, C::kBoxBytes, 1024);
#pragma unroll
  for (int k = HALF * kHalf; k < (HALF + 1) * kHalf; ++k) {
    mma_ts<C::T::kKind>(d_tmem, p_tmem + k * 8, desc_add(b0, (k * C::kKPerMma * 128) >> 4),
                        C::kIdescPV, (accumulate || k > 0) ? 1u : 0u);
  }
}

template <int DT, int D, bool CAUSAL>
__device__ void role_mma(uint8_t* sbase, Ctrl<Cfg<DT, D>::kSlots>* c, uint32_t tbase,
                         const AttnParams& p) {
  using C = Cfg<DT, D>;
  constexpr int NQT = C::kNQT;
  const WaitCtx wc{&c->abort, p.timeout_ns, p.status, p.where};
  const uint32_t sq = smem_u32(sbase);
  const uint32_t skv = sq + C::kQBufTiles * C::kTileBytes;
  uint32_t q_waits[2] = {0, 0}, p_waits[2] = {0, 0};
  uint32_t s_cnt[2] = {0, 0};  // S products issued per tile
  uint32_t s_next = 0;         // S lookahead: the buffer the next S goes to
  // S buffer of each tile's S products not yet consumed by P V (at most
  // two a tile): two bits at bit 4 * t + 2 * (count & 1)
  uint32_t pbuf = 0x50u;
  RingPos ring;
  bool ok = true;

  // S_t = Q_t K^T with K in shared memory at sk, committed to s_full: Q_t
  // from shared memory, or (kQTmem) from Tensor Memory; into the tile's own
  // S buffer, or (S lookahead) the next one in turn
  auto issue_s = [&](int t, uint32_t sk) {
    const uint32_t b = C::kSLook ? s_next : static_cast<uint32_t>(t);
    const uint32_t d_tmem = tbase + C::s_buf_col(b);
    if constexpr (C::kQTmem)
      mma_tk<DT, D>(d_tmem, tbase + C::q_col(), sk, C::kIdescQK);
    else
      issue_qk<DT, D>(d_tmem, sq + t * C::kTileBytes, sk);
    if constexpr (C::kSLook) {
      const uint32_t sh = 4u * static_cast<uint32_t>(t) + 2u * (s_cnt[t] & 1u);
      pbuf = (pbuf & ~(3u << sh)) | (b << sh);
      mma_commit(smem_u32(&c->s_full[t][bar_set(s_cnt[t], C::kBarSets)]));
      ++s_cnt[t];
      s_next = s_next == 2u ? 0u : s_next + 1u;
    } else {
      mma_commit(smem_u32(&c->s_full[t][0]));
    }
  };
  // S_t(0) of item w with K_0 in stage ks; false when a wait gave up
  auto issue_s0 = [&](const Item& w, int t, int ks) -> bool {
    if constexpr (!C::kQTmem) {
      if (!wait_bar(smem_u32(&c->q_full[t]), q_waits[t] & 1u, wc, 0x12)) return false;
      ++q_waits[t];
      tc_fence_after_sync();
    }
    issue_s(t, skv + C::k_slot(ks) * C::kTileBytes);
    if (!C::kQTmem && w.n[t] == 1) mma_commit(smem_u32(&c->q_empty[t]));
    return true;
  };

  // Where C::kEarlyS0 holds, the next item's S_t(0) goes out right behind
  // this item's last P_t V when its K_0 and Q_t are already here: the
  // tensor pipe runs one thread's MMAs in order, so S_t(0) overwrites P_t
  // only after that product has read it, and the next item's first softmax
  // starts without waiting for the rest of this item.
  constexpr bool kEarly = C::kEarlyS0;
  bool s0_issued = false;  // S_t(0) of this item went out during the previous one
  int held = -1;           // stage that holds this item's K_0 (paired stages)
  for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < p.n_items && ok; ++rnd) {
    const int it = round_item(rnd, p.n_items);
    if (it < 0) continue;
    const Item w = decode_item<NQT, CAUSAL>(it, p);
    const int walk = w.nmax;
    Item wn;
    const bool has_next = next_item<NQT, CAUSAL>(rnd, p, wn);
    if constexpr (C::kQTmem) {
      // the item's Q from its ring stage into Tensor Memory (after the
      // previous item's last S, which read the old Q: this thread's tensor
      // operations run in order), then the stage back to the producer
      int qs;
      uint32_t qpar;
      ring.next<C::kStages>(qs, qpar);
      if (!wait_bar(smem_u32(&c->kv_full[qs]), qpar, wc, 0x12)) break;
      tc_fence_after_sync();
      copy_tile_to_tmem<DT, D>(tbase + C::q_col(), skv + C::k_slot(qs) * C::kTileBytes);
      mma_commit(smem_u32(&c->kv_empty[qs]));
    }
    if (!s0_issued) {
      // S_t(0) for every tile
      int ks = held;
      if (ks < 0) {
        uint32_t kpar;
        ring.next<C::kStages>(ks, kpar);
        if (!wait_bar(smem_u32(&c->kv_full[ks]), kpar, wc, 0x11)) break;
      }
      for (int t = 0; t < NQT && ok; ++t) ok = issue_s0(w, t, ks);
      if (!ok) break;
      mma_commit(smem_u32(&c->kv_empty[ks]));
      held = -1;
    }
    s0_issued = false;

    for (int j = 0; j < walk && ok; ++j) {
      int vs;
      uint32_t vpar;
      ring.next<C::kStages>(vs, vpar);
      if (!wait_bar(smem_u32(&c->kv_full[vs]), vpar, wc, 0x13)) break;
      const bool last = j + 1 == walk;
      const bool ahead = kEarly && last && has_next;  // the next item's S_t(0)
      // stage of the next K: the same one when stages are paired
      int ns = vs;
      uint32_t npar = vpar;
      bool k_ready = C::kPair;
      bool s0_done[2] = {false, false};
      if (!C::kPair && (!last || ahead)) ring.next<C::kStages>(ns, npar);
      const uint32_t sv = skv + C::v_slot(vs) * C::kTileBytes;
      const uint32_t sk = skv + C::k_slot(ns) * C::kTileBytes;
      for (int t = 0; t < NQT && ok; ++t) {
        // S_t(j + 1): behind P_t(j) V, or (S lookahead) ahead of it
        auto next_s = [&]() -> bool {
          if (j + 1 < w.n[t]) {
            if (!k_ready) {
              if (!wait_bar(smem_u32(&c->kv_full[ns]), npar, wc, 0x16)) return false;
              k_ready = true;
            }
            issue_s(t, sk);
            if (!C::kQTmem && j + 2 == w.n[t]) mma_commit(smem_u32(&c->q_empty[t]));
          }
          return true;
        };
        if (C::kSLook && !next_s()) {
          ok = false;
          break;
        }
        if (j < w.n[t]) {
          // first key half as soon as its P and the rescaled O are there
          // (p_full[t][0] counts the softmax and the correction warps),
          // overlapping the softmax of the second half
          const uint32_t pk = p_waits[t];
          if (!wait_bar(smem_u32(&c->p_full[t][0]), pk & 1u, wc, 0x14)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t p_tmem =
              C::kSLook ? tbase + C::s_buf_col((pbuf >> (4u * static_cast<uint32_t>(t) + 2u * (pk & 1u))) & 3u)
                        : tbase + C::s_col(t);
          issue_pv_half<DT, D, 0>(tbase + C::o_col(t), p_tmem, sv, j > 0);
          if (!wait_bar(smem_u32(&c->p_full[t][1 + bar_set(pk, C::kBarSets)]),
                        bar_par(pk, C::kBarSets), wc, 0x18)) {
            ok = false;
            break;
          }
          ++p_waits[t];
          tc_fence_after_sync();
          issue_pv_half<DT, D, 1>(tbase + C::o_col(t), p_tmem, sv, true);
          // O_t is complete for the epilogue after the tile's last block.
          // For earlier blocks the correction warps rescale O_t for block
          // j + 1 only once this product is done: they wait for pv_done
          // (S lookahead), or else for alpha_t(j + 1), which the softmax
          // publishes after S_t(j + 1) completed, and that commit, issued
          // behind this product, tracks it too.
          if (j + 1 == w.n[t])
            mma_commit(smem_u32(&c->o_full[t]));
          else if constexpr (C::kSLook)
            mma_commit(smem_u32(&c->pv_done[t]));
        }
        if (!C::kSLook && !next_s()) {
          ok = false;
          break;
        }
        if constexpr (kEarly) {
          // only where K_0 and Q_t are already here: the other tile's P V
          // must not wait behind them
          // (S lookahead: S products go out in tile order, which the
          // softmax's choice of buffer assumes)
          if (ahead && (!C::kSLook || t == 0 || s0_done[0])) {
            if (!k_ready) k_ready = mbar_test_wait(smem_u32(&c->kv_full[ns]), npar);
            if (k_ready && mbar_test_wait(smem_u32(&c->q_full[t]), q_waits[t] & 1u)) {
              ok = issue_s0(wn, t, ns);
              s0_done[t] = true;
            }
          }
        }
      }
      if (!ok) break;
      if constexpr (!C::kPair) mma_commit(smem_u32(&c->kv_empty[vs]));
      if (!last || ahead) {
        if (!k_ready && !wait_bar(smem_u32(&c->kv_full[ns]), npar, wc, 0x16)) break;
        if constexpr (kEarly) {
          for (int t = 0; t < NQT && ok && ahead; ++t)
            if (!s0_done[t]) ok = issue_s0(wn, t, ns);
          if (!ok) break;
          s0_issued = ahead;
        }
        mma_commit(smem_u32(&c->kv_empty[ns]));
      } else if constexpr (C::kPair) {
        // the last block: this stage also holds the next item's K_0, used
        // by its S_t(0) before the stage is released
        if (has_next)
          held = vs;
        else
          mma_commit(smem_u32(&c->kv_empty[vs]));
      }
    }
  }
  // Wait until every MMA issued above has completed before the CTA frees
  // Tensor Memory.
  mma_commit(smem_u32(&c->drain));
  volatile uint32_t never = 0;
  const WaitCtx wc_never{&never, p.timeout_ns, p.status, p.where};
  wait_bar(smem_u32(&c->drain), 0u, wc_never, 0x17);
}

// ---------------------------------------------------------------------------
// softmax warpgroup of tile t: one thread = one row = one TMEM lane

template <int DT>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<1>(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<2>(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
// two e4m3 codes in the low 16 bits: a in the low byte
__device__ __forceinline__ uint32_t pack2_e4m3(float a, float b) {
  __nv_fp8x2_e4m3 v(make_float2(a, b));
  return static_cast<uint32_t>(*reinterpret_cast<uint16_t*>(&v));
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Largest of the 128 scores of a row: four independent three-input max
// chains of 32 scores each.
__device__ __forceinline__ float max128(const float (&s)[128]) {
  float m[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float* x = s + 32 * k;
    float a = max3f(x[0], x[1], x[2]);
#pragma unroll
    for (int i = 3; i < 31; i += 2) a = max3f(a, x[i], x[i + 1]);
    m[k] = fmaxf(a, x[31]);
  }
  return fmaxf(max3f(m[0], m[1], m[2]), m[3]);
}

// Registers per thread of each warpgroup after setmaxnreg (multiples of 8).
constexpr int kRegsControl = 88;      // producer and MMA-issuer warpgroup
constexpr int kRegsSoftmax = 168;     // each softmax warpgroup: a 128-score row
constexpr int kRegsCorrection = 80;   // correction / epilogue warpgroup

// 2^x for two values on the FMA pipe instead of MUFU (the optional path of
// ATTN_OPT_EXP2_FMA).  Cody and Waite's reduction: x = n + f with n =
// round(x), taken by adding and subtracting 1.5 * 2^23, and |f| <= 1/2;
// then 2^f by a degree-3 polynomial and n added to its exponent field.  The
// coefficients are the minimax fit of the relative error on [-1/2, 1/2]
// that fit_exp2_poly.py computes (Remez exchange), 7.5e-5 at most.  x below
// -126 (masked keys, x = -inf) gives exactly 0, as ex2.approx.ftz does.
__device__ __forceinline__ void exp2_fma2(float x0, float x1, float& e0, float& e1) {
  const uint64_t magic = f2_pack(12582912.f, 12582912.f);   // 1.5 * 2^23
  const uint64_t xx = f2_pack(fmaxf(x0, -127.f), fmaxf(x1, -127.f));
  const uint64_t t2 = f2_add(xx, magic);                     // n in the low mantissa bits
  const uint64_t n2 = f2_add(t2, f2_pack(-12582912.f, -12582912.f));
  const uint64_t fr = f2_fma(n2, f2_pack(-1.f, -1.f), xx);   // f = x - n
  uint64_t q = f2_fma(f2_pack(0.0551716685f, 0.0551716685f), fr,
                      f2_pack(0.242611125f, 0.242611125f));
  q = f2_fma(q, fr, f2_pack(0.693260968f, 0.693260968f));
  q = f2_fma(q, fr, f2_pack(0.999928057f, 0.999928057f));
  float q0, q1, t0, t1;
  f2_unpack(q, q0, q1);
  f2_unpack(t2, t0, t1);
  e0 = x0 < -126.f ? 0.f : __int_as_float(__float_as_int(q0) + (__float_as_int(t0) << 23));
  e1 = x1 < -126.f ? 0.f : __int_as_float(__float_as_int(q1) + (__float_as_int(t1) << 23));
}

// Exponentials of scores OFF .. OFF+LEN-1 of one row, written as P into
// Tensor Memory at taddr_p (16-bit types pack two per column, e4m3 four).
// x = s * scale_log2 - m in packed pairs, p = 2^x on MUFU, or, for XF of
// every 32 scores (the last XF), on the FMA pipe (exp2_fma2).  Returns the
// sum of the fp32 exponentials (before rounding to the P type).
template <int DT, int OFF, int LEN, int XF = 0>
__device__ __forceinline__ float exp_store_chunk(const float (&s)[128], float sl2, float neg_m,
                                                 uint32_t taddr_p) {
  const uint64_t k2 = f2_pack(sl2, sl2);
  const uint64_t b2 = f2_pack(neg_m, neg_m);
  uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
  constexpr int kWords = DT == 3 ? LEN / 4 : LEN / 2;
  uint32_t pk[kWords];
#pragma unroll
  for (int ii = 0; ii < LEN; ii += 4) {
    const int i = OFF + ii;
    float x0, x1, x2, x3;
    f2_unpack(f2_fma(f2_pack(s[i], s[i + 1]), k2, b2), x0, x1);
    f2_unpack(f2_fma(f2_pack(s[i + 2], s[i + 3]), k2, b2), x2, x3);
    float e0, e1, e2, e3;
    if (XF > 0 && (ii % 32) >= 32 - XF) {
      exp2_fma2(x0, x1, e0, e1);
      exp2_fma2(x2, x3, e2, e3);
    } else {
      e0 = ex2_approx(x0);
      e1 = ex2_approx(x1);
      e2 = ex2_approx(x2);
      e3 = ex2_approx(x3);
    }
    acc0 = f2_add(acc0, f2_pack(e0, e1));
    acc1 = f2_add(acc1, f2_pack(e2, e3));
    if constexpr (DT == 3) {
      pk[ii / 4] = pack2_e4m3(e0, e1) | (pack2_e4m3(e2, e3) << 16);
    } else {
      pk[ii / 2] = pack2<DT>(e0, e1);
      pk[ii / 2 + 1] = pack2<DT>(e2, e3);
    }
  }
  if constexpr (kWords == 32)
    tmem_st_x32(taddr_p, pk);
  else if constexpr (kWords == 16)
    tmem_st_x16(taddr_p, pk);
  else
    tmem_st_x8(taddr_p, pk);
  float a0, a1;
  f2_unpack(f2_add(acc0, acc1), a0, a1);
  return a0 + a1;
}

// The subtraction reference moves when a block's max exceeds it by more
// than kRescaleLog2 (base-2 units of the scaled scores); otherwise alpha = 1
// and the correction warpgroup skips the O rescale.  A threshold t > 0 lets
// probabilities reach 2^t: O / l and m + log2 l are unchanged in real
// arithmetic, but the largest probability of a row is then no longer exactly
// 1 and picks up the P type's rounding (2^-8 relative in bf16), which a
// peaked softmax passes straight into O.  The exact running max (0) keeps
// that term exact.
constexpr float kRescaleLog2 = 0.0f;

template <int DT, int D, bool CAUSAL, int XF>
__device__ void role_softmax(int t, Ctrl<Cfg<DT, D>::kSlots>* c, uint32_t tbase,
                             const AttnParams& p) {
  using C = Cfg<DT, D>;
  const WaitCtx wc{&c->abort, p.timeout_ns, p.status, p.where};
  const uint32_t lane = lane_id();
  const uint32_t wq = (threadIdx.x >> 5) & 3u;  // warp quarter = TMEM lane group
  const int r = static_cast<int>(wq * 32u + lane);
  const uint32_t taddr = tbase + ((wq * 32u) << 16) + C::s_col(t);
  const float sl2 = p.scale_log2;
  uint32_t s_waits = 0;
  uint32_t iter = 0;
  // S lookahead: S products fill the three buffers in turn, in issue order
  // (blocks in order, tile 0 before tile 1 within a block); seq3 is the
  // number of S products of the earlier items, mod 3
  [[maybe_unused]] uint32_t seq3 = 0;

  for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < p.n_items; ++rnd) {
    const int it = round_item(rnd, p.n_items);
    if (it < 0) continue;
    const Item w = decode_item<C::kNQT, CAUSAL>(it, p);
    const int qt = w.qt0 + t;
    const int n = w.n[t];
    float m_run = -INFINITY;  // subtraction reference (log2 units)
    float l_run = 0.f;
    float q_bs = 1.0f;  // block scale of this query tile (e4m3 block scaling)
    if constexpr (DT == 3) {
      // the second tile of the last pair lies past N when n_qt is odd: its
      // rows are never stored, and its scale is not read
      if (p.q_block_scale && qt < p.n_qt)
        q_bs = p.q_block_scale[static_cast<size_t>(w.bh) * p.n_qt + qt];
    }
    float* const inv_l_dst = &c->inv_l[iter & 1u][t][r];
    float* const alpha_dst = &c->alpha[t][r];
    float* const alpha_odd_dst = alpha_odd(c) + t * kBlock + r;
    // S lookahead: this tile's S buffer for block 0 (both tiles have one:
    // n[0] >= 1)
    [[maybe_unused]] uint32_t sb = (seq3 + static_cast<uint32_t>(t)) % 3u;
    for (int j = 0; j < n; ++j) {
      // S lookahead: s_full in two sets used in turn, S in buffer sb
      uint32_t sa = taddr;
      if constexpr (C::kSLook) {
        if (!wait_bar(smem_u32(&c->s_full[t][s_waits & 1u]), (s_waits >> 1) & 1u, wc, 0x21)) return;
        sa = taddr - C::s_col(t) + C::s_buf_col(sb);
      } else {
        if (!wait_bar(smem_u32(&c->s_full[t][0]), s_waits & 1u, wc, 0x21)) return;
      }
      ++s_waits;
      tc_fence_after_sync();
      // mask: keys >= N in the last block; keys after the query on the
      // causal diagonal block
      int lim = p.N - j * kBlock;
      if (CAUSAL && j == qt) lim = min(lim, r + 1);

      // The whole row of scores in registers (the softmax warpgroups run
      // with 168 registers per thread).
      float s[kBlock];
      {
        uint32_t raw[kBlock];
        tmem_ld_2x64(sa, raw);
#pragma unroll
        for (int i = 0; i < kBlock; ++i) s[i] = __uint_as_float(raw[i]);
      }
      if (lim < kBlock) {
#pragma unroll
        for (int i = 0; i < kBlock; ++i) s[i] = i < lim ? s[i] : -INFINITY;
      }
      // scale of this block's scores in base-2 units: with block scales,
      // the real score is q_scale * k_scale * (code product)
      float sl2j = sl2;
      if constexpr (DT == 3) {
        if (p.k_block_scale)
          sl2j = sl2 * q_bs * p.k_block_scale[static_cast<size_t>(w.bh) * p.nkv + j];
      }
      const float mx = max128(s) * sl2j;

      float alpha = 1.0f;
      if (mx > m_run + kRescaleLog2) {
        alpha = ex2_approx(m_run - mx);  // 0 on the first block (m_run = -inf)
        m_run = mx;
      }
      // subtraction reference: 0 while every key so far is masked
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      // S lookahead: alpha of block k goes to array k mod 2.  It reuses the
      // array of block k - 2 only after S(k) completed, which was issued
      // after P(k - 2) V, which waited for the correction warps' arrival
      // after their read of alpha(k - 2): no wait is needed here, and the
      // two alpha barriers cannot run two phases ahead of those warps.
      if (C::kSLook && ((s_waits - 1u) & 1u))
        *alpha_odd_dst = alpha;
      else
        *alpha_dst = alpha;
      __syncwarp();
      if (lane == 0) mbar_arrive(sc_bar<C::kSLook>(c, t, s_waits - 1u));

      // P over the first kPCols columns of S (already in registers), in two
      // halves of 64 keys: the first is handed to the MMA issuer while the
      // second is computed
      const float neg_m = -m_use;
      const float sum0 = exp_store_chunk<DT, 0, 64, XF>(s, sl2j, neg_m, sa);
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&c->p_full[t][0]));
      const float sum1 = exp_store_chunk<DT, 64, 64, XF>(s, sl2j, neg_m, sa + C::kPCols / 2);
      l_run = alpha * l_run + (sum0 + sum1);
      tmem_st_wait();
      // hand 1/l to the epilogue before the last P is announced
      if (j == n - 1) *inv_l_dst = __frcp_rn(l_run);
      tc_fence_before_sync();
      __syncwarp();
      if constexpr (C::kSLook) {
        if (lane == 0) mbar_arrive(smem_u32(&c->p_full[t][1 + ((s_waits - 1u) & 1u)]));
        sb = (sb + (t == 0 ? 2u : (j + 1 < w.n[0] ? 2u : 1u))) % 3u;
      } else {
        if (lane == 0) mbar_arrive(smem_u32(&c->p_full[t][1]));
      }
    }
    if constexpr (C::kSLook) seq3 = (seq3 + static_cast<uint32_t>(w.n[0] + w.n[1])) % 3u;
    // LSE (natural log) of the real rows
    const int row = qt * kBlock + r;
    if (row < p.N) {
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      p.lse[static_cast<size_t>(w.bh) * p.N + row] = (m_use + __log2f(l_run)) * 0.6931471805599453f;
    }
    ++iter;
  }
}

// ---------------------------------------------------------------------------
// correction / epilogue warpgroup

// Eight output values (already scaled) as one 16-byte chunk of the output
// type (bf16 for e4m3 inputs)
template <int DT>
__device__ __forceinline__ uint4 pack8_out(const float* v) {
  constexpr int kOut = DT == 1 ? 1 : 2;
  return make_uint4(pack2<kOut>(v[0], v[1]), pack2<kOut>(v[2], v[3]), pack2<kOut>(v[4], v[5]),
                    pack2<kOut>(v[6], v[7]));
}

// The output is staged through shared memory (one 128-row x 64-column box
// at a time, in the 128-byte-swizzled layout the O tensor map uses) and
// written by TMA tensor stores, so that every global write is a whole
// coalesced box; rows past N are clipped by the tensor map.
template <int DT, int D, bool CAUSAL>
__device__ void role_correction(Ctrl<Cfg<DT, D>::kSlots>* c, uint32_t tbase, uint32_t stage,
                                const CUtensorMap* tmO, const AttnParams& p) {
  using C = Cfg<DT, D>;
  constexpr int NQT = C::kNQT;
  const WaitCtx wc{&c->abort, p.timeout_ns, p.status, p.where};
  const uint32_t lane = lane_id();
  const uint32_t wq = (threadIdx.x >> 5) & 3u;
  const int r = static_cast<int>(wq * 32u + lane);
  const uint32_t lane_off = (wq * 32u) << 16;
  const bool issuer = r == 0;  // issues and tracks the TMA stores
  const uint32_t stage_row0 = stage + static_cast<uint32_t>(r) * 128u;
  uint32_t nbox = 0;  // boxes stored (selects the staging buffer)
  uint32_t sc_waits[2] = {0, 0}, o_waits[2] = {0, 0}, pv_waits[2] = {0, 0};
  uint32_t iter = 0;
  bool ok = true;
  // this item's first block of tile t was handled in the previous epilogue
  bool first_done[2] = {false, false};

  for (int rnd = 0; ok && rnd * static_cast<int>(gridDim.x) < p.n_items; ++rnd) {
    const int it = round_item(rnd, p.n_items);
    if (it < 0) continue;
    const Item w = decode_item<NQT, CAUSAL>(it, p);
    Item wn;
    const bool has_next = next_item<NQT, CAUSAL>(rnd, p, wn);
    // the next item's first block of tile t: its alpha (unused) consumed and
    // O_t handed to its first P V, as soon as this item's O_t is read out
    auto first_block_of_next = [&](int t) -> bool {
      if (!wait_bar(sc_bar<C::kSLook>(c, t, sc_waits[t]), sc_par<C::kSLook>(sc_waits[t]), wc, 0x31))
        return false;
      ++sc_waits[t];
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&c->p_full[t][0]));
      first_done[t] = true;
      return true;
    };
    for (int j = 0; j < w.nmax && ok; ++j) {
      for (int t = 0; t < NQT; ++t) {
        if (j >= w.n[t]) continue;
        if (j == 0 && first_done[t]) {
          first_done[t] = false;
          continue;
        }
        const uint32_t scn = sc_waits[t];
        if (!wait_bar(sc_bar<C::kSLook>(c, t, scn), sc_par<C::kSLook>(scn), wc, 0x31)) {
          ok = false;
          break;
        }
        ++sc_waits[t];
        const float alpha = (C::kSLook && (scn & 1u))
                                ? alpha_odd(c)[t * kBlock + r]
                                : c->alpha[t][r];
        if (j > 0) {
          // P_t V_{j-1} has completed: under S lookahead its own commit
          // says so; otherwise alpha_t(j) was published after S_t(j), whose
          // commit came after that product
          if constexpr (C::kSLook) {
            if (!wait_bar(smem_u32(&c->pv_done[t]), pv_waits[t] & 1u, wc, 0x34)) {
              ok = false;
              break;
            }
            ++pv_waits[t];
          }
          tc_fence_after_sync();
          // exact skip: a warp whose 32 rows all kept their max has alpha == 1
          if (!__all_sync(0xffffffffu, alpha == 1.0f)) {
            const uint32_t ta = tbase + lane_off + C::o_col(t);
#pragma unroll 1
            for (int cc = 0; cc < D; cc += 32) {
              uint32_t v[32];
              tmem_ld_x32(ta + cc, v);
              const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                float x0, x1;
                f2_unpack(f2_mul(f2_pack(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), a2),
                          x0, x1);
                v[i] = __float_as_uint(x0);
                v[i + 1] = __float_as_uint(x1);
              }
              tmem_st_x32(ta + cc, v);
            }
            tmem_st_wait();
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&c->p_full[t][0]));
      }
    }
    // epilogue: O / l (times the v descale) -> output dtype
    for (int t = 0; t < NQT && ok; ++t) {
      if (!wait_bar(smem_u32(&c->o_full[t]), o_waits[t] & 1u, wc, 0x33)) {
        ok = false;
        break;
      }
      ++o_waits[t];
      tc_fence_after_sync();
      const float f = c->inv_l[iter & 1u][t][r] * p.out_scale;
      const int qt = w.qt0 + t;
      const uint32_t ta = tbase + lane_off + C::o_col(t);
#pragma unroll 1
      for (int bx = 0; bx < D / 64; ++bx) {
        // 16-byte chunk k of the row sits at chunk k ^ (row mod 8)
        const uint32_t rsw = static_cast<uint32_t>(r) & 7u;
        const uint32_t sbuf = C::kStageBufs == 2 ? (nbox & 1u) * C::kStageBytes : 0u;
        const uint32_t stage_row = stage_row0 + sbuf;
        ++nbox;
        if constexpr (C::kEpiPrefetch) {
          // the box's 64 columns, read and packed while the previous store
          // may still be reading the staging box
          uint4 pk[8];
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            uint32_t v[32];
            tmem_ld_x32(ta + bx * 64 + g * 32, v);
            float x[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(v[i]) * f;
#pragma unroll
            for (int i = 0; i < 4; ++i) pk[4 * g + i] = pack8_out<DT>(x + 8 * i);
          }
          // (no break on failure: every warp goes on through the named barriers)
          if (has_next && bx == D / 64 - 1 && !first_block_of_next(t)) ok = false;
          if (issuer) {
            if constexpr (C::kStageBufs == 2)
              bulk_wait_read_1();
            else
              bulk_wait_read_all();
          }
          named_bar_sync(1, 128);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            st_shared_v4(stage_row + ((static_cast<uint32_t>(k) ^ rsw) << 4), pk[k]);
        } else {
          // the previous store has finished reading the staging box
          if (issuer) bulk_wait_read_all();
          named_bar_sync(1, 128);
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            uint32_t v[32];
            tmem_ld_x32(ta + bx * 64 + g * 32, v);
            float x[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(v[i]) * f;
#pragma unroll
            for (int i = 0; i < 4; ++i)
              st_shared_v4(stage_row + ((static_cast<uint32_t>(4 * g + i) ^ rsw) << 4),
                           pack8_out<DT>(x + 8 * i));
          }
          if (has_next && bx == D / 64 - 1 && !first_block_of_next(t)) ok = false;
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (issuer && qt * kBlock < p.N) {
          tma_store_3d(tmO, stage + sbuf, bx * 64, qt * kBlock, w.bh);
          bulk_commit_group();
        }
      }
    }
    ++iter;
  }
  // no store may still read shared memory (or be in flight) when the CTA
  // exits
  if (issuer) bulk_wait_all();
}

// ---------------------------------------------------------------------------

// XF: exponentials of every 32 computed on the FMA pipe (0: all on MUFU;
// the ATTN_OPT_EXP2_FMA instances use 4)
template <int DT, int D, bool CAUSAL, int XF = 0>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const AttnParams p) {
  using C = Cfg<DT, D>;
  using CtrlT = Ctrl<C::kSlots>;
  static_assert(sizeof(CtrlT) + 1024 <= C::kMiscBytes, "control block budget");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // tiles need 1024-byte alignment (128-byte swizzle atoms)
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* sbase = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t stage = smem_u32(sbase + (C::kQBufTiles + C::kSlots) * C::kTileBytes);
  CtrlT* c = reinterpret_cast<CtrlT*>(sbase + (C::kQBufTiles + C::kSlots) * C::kTileBytes +
                                      C::kStageTotal);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&c->q_full[t]), 1);
      mbar_init(smem_u32(&c->q_empty[t]), 1);
      mbar_init(smem_u32(&c->s_full[t][0]), 1);
      mbar_init(smem_u32(&c->s_full[t][1]), 1);
      mbar_init(smem_u32(&c->p_full[t][0]), 8);
      mbar_init(smem_u32(&c->p_full[t][1]), 4);
      mbar_init(smem_u32(&c->p_full[t][2]), 4);
      mbar_init(smem_u32(&c->sc_full[t]), 4);
      mbar_init(smem_u32(&c->sc_full_odd[t]), 4);
      mbar_init(smem_u32(&c->o_full[t]), 1);
      mbar_init(smem_u32(&c->pv_done[t]), 1);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&c->kv_full[s]), 1);
      mbar_init(smem_u32(&c->kv_empty[s]), 1);
    }
    mbar_init(smem_u32(&c->drain), 1);
    c->abort = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&c->tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  // the tail launch that follows on the stream counts its pieces in these
  // words: clear them here rather than in a launch of their own; that
  // launch may place its CTAs on the SMs this grid leaves (it waits for
  // this grid's completion before it touches the words)
  if (p.flags != nullptr) {
    if (blockIdx.x == 0 && warp == 2)
      for (int i = static_cast<int>(lane); i < 2 * p.tail_items; i += 32) p.flags[i] = 0u;
    if (threadIdx.x == 0) griddep_launch_dependents();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = c->tmem_base;

  // Role dispatch by warpgroup, with the register file split among them:
  // producer / MMA + 2 * softmax + correction must stay within the 4 * 128
  // registers per thread the block is launched with (the host refuses to
  // launch a build with any other count).
  static_assert(kRegsControl + 2 * kRegsSoftmax + kRegsCorrection <= 4 * 128, "register split");
  const uint32_t wg = warp >> 2;
  if (wg == 0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
    if (warp == 0 && lane == 0)
      role_producer<DT, D, CAUSAL>(&tmQ, &tmK, &tmV, sbase, c, p);
    else if (warp == 1 && lane == 0)
      role_mma<DT, D, CAUSAL>(sbase, c, tbase, p);
  } else if (wg == 1 || wg == 2) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    if (static_cast<int>(wg) - 1 < C::kNQT) role_softmax<DT, D, CAUSAL, XF>(wg - 1, c, tbase, p);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCorrection));
    role_correction<DT, D, CAUSAL>(c, tbase, stage, &tmO, p);
  }

  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, C::kTmemCols);
  }
}

}  // namespace wsattn

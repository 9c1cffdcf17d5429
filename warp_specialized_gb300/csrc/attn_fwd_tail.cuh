// attn_fwd_tail.cuh - the forward kernel's second launch for the work the
// static rounds leave over.
//
// The persistent forward kernel gives each CTA whole work items in rounds.
// When the item count is not a multiple of the CTA count, the last round
// leaves SMs idle while the rest finish a whole item (1024 items on 152
// SMs: 6.74 rounds run as 7; 32 items: one round on 32 SMs).  With a caller
// workspace the main kernel runs only the whole rounds and this kernel
// takes the remaining items: their key blocks (units) are shared out over
// its CTAs in contiguous ranges (tail_range_start).  Each CTA walks its
// range with the main kernel's roles, in segments of key blocks [jb, je) of
// one item.  A segment that is not the whole item is a piece: its
// unnormalised O, its subtraction reference m and its sum l go to the
// workspace, and the piece that finds every other piece of the tile done
// merges them (the concept card's "Implementation sketch" rescale, by
// exp2(m_k - M) for the largest reference M) and writes O and LSE.  No CTA
// waits for another.  Behind a main launch the CTAs start as the main
// grid's CTAs leave their SMs (programmatic dependent launch), so the
// ranges are ramped: the CTAs that start first take a little more.
//
// The segment bookkeeping and the merge cost registers; kept out of the
// main kernel, they slow only this share of the work.
#pragma once

#include "attn_fwd_kernel.cuh"
#include "attn_launch.h"

namespace wsattn {

// registers per thread after setmaxnreg in this kernel
constexpr int kTailRegsControl = 88;
constexpr int kTailRegsCorrection = 88;
// largest tail grid (the table of range starts lives in shared memory)
constexpr int kMaxTailGrid = 255;
// the control block of this kernel carries the pieces' m, the CTAs' range
// starts and broadcast words beyond the main kernel's
constexpr int kTailCtrlExtra = 2 * 2 * kBlock * 4 + (kMaxTailGrid + 1) * 4 + 256;

template <int NSLOT>
struct CtrlTail {
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[NSLOT], kv_empty[NSLOT];
  uint64_t s_full[2];
  uint64_t p_full[2][2];
  uint64_t sc_full[2];
  uint64_t o_full[2];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t bcast2[2];    // the pieces' flag counts, per tile (shared by the issuing thread)
  int rs[kMaxTailGrid + 1];  // tail_range_start of every CTA (and the end)
  float alpha[2][kBlock];
  // [segment parity][tile][row]: 1 / l of a whole tile, or l of a piece
  float inv_l[2][2][kBlock];
  float part_m[2][2][kBlock];  // a piece's subtraction reference m (log2 units)
};

template <int DT, int D>
struct TailCfg {
  using C = Cfg<DT, D>;
  static constexpr int kSmemBytes = C::kSmemBytes + kTailCtrlExtra;
  static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
  // the host's restatement of the layout (the tail grid is planned on it)
  static_assert(fwd_region_bytes(D, C::kEsize) == (C::kNQT + C::kSlots) * C::kTileBytes &&
                    fwd_nqt(D, C::kEsize) == C::kNQT && kFwdMiscBytes == C::kMiscBytes &&
                    kFwdSmemLimit == kSmemLimit && kFwdStageBytes == C::kStageBytes && C::kStageBufs == (C::kEsize == 1 ? 2 : 1),
                "host copy of the shared-memory layout");
};

// ---------------------------------------------------------------------------
// Segments: what a tail CTA works on, in order.  A segment is key blocks
// [jb, je) of one tail item: the whole item, or a piece of it where a CTA
// range boundary cuts the item.

struct Seg {
  Item w;
  int jb, je;
  int ti;   // tail item index
  int xs;   // first tail unit of the item
};

// Tail units stay below 2^31 (the tail holds at most 2 G items of at most
// 2^17 blocks); the products below are formed in 64 bits.  CTA c's range
// starts at f(c) = c U / G + A c (G - c) / G: equal shares when A = 0; with
// a ramp A > 0, CTA c's share is about U / G + A (G - 1 - 2c) / G, so the
// CTAs that start first (the tail grid's CTAs take SMs in index order as
// the main grid's CTAs leave them) take more.  A < U / (2G) keeps every
// share positive.
__device__ __forceinline__ int tail_range_start(int c, const AttnParams& p) {
  const long long g = gridDim.x;
  const long long cc = c;
  return static_cast<int>((cc * p.tail_units * g + p.tail_ramp * cc * (g - cc)) / (g * g));
}
template <int NQT, bool CAUSAL>
struct SegIter {
  int u, u_end;  // next tail unit of this CTA, end of its range
  int xs;        // first unit of tail item ti
  int ti;

  __device__ __forceinline__ void init(const AttnParams& p) {
    u = u_end = xs = 0;
    ti = 0;
    if (p.tail_items == 0) return;
    u = tail_range_start(static_cast<int>(blockIdx.x), p);
    u_end = tail_range_start(static_cast<int>(blockIdx.x) + 1, p);
    if (u >= u_end) return;
    if (!CAUSAL) {
      ti = u / p.nkv;
      xs = ti * p.nkv;
      return;
    }
    // causal: items come in levels of B*H items with the same block count
    int it = p.tail_start;
    int acc = 0;
    while (true) {
      const int pair = p.n_pairs - 1 - it / p.BH;
      const int walk = min(pair * NQT + NQT, p.nkv);
      const int left = p.BH - it % p.BH;
      const int span = left * walk;
      if (u < acc + span) {
        const int k = (u - acc) / walk;
        ti = it + k - p.tail_start;
        xs = acc + k * walk;
        return;
      }
      acc += span;
      it += left;
    }
  }

  __device__ __forceinline__ bool next(Seg& sg, const AttnParams& p) {
    if (u >= u_end) return false;
    sg.w = decode_item<NQT, CAUSAL>(p.tail_start + ti, p);
    const int xe = xs + sg.w.nmax;
    sg.jb = u - xs;
    sg.je = (u_end < xe ? u_end : xe) - xs;
    sg.ti = ti;
    sg.xs = xs;
    u = xs + sg.je;
    if (u == xe) {
      ++ti;
      xs = xe;
    }
    return true;
  }
};

// Key blocks of tile t in segment sg: [sg.jb, seg_end(sg, t)), empty when
// the end is not above jb.
__device__ __forceinline__ int seg_end(const Seg& sg, int t) {
  return min(sg.je, sg.w.n[t]);
}

// Pieces of tile t of a tail item, and which of them this segment is.
struct PieceInfo {
  int np;     // pieces holding blocks of the tile (1: the segment is the whole tile)
  int k;      // this segment's piece
  int c0;     // CTA of piece 0
};
// the CTA whose range holds unit u, from the table of range starts rs
__device__ __forceinline__ int tail_cta_rs(int u, const int* rs) {
  int lo = 0, hi = static_cast<int>(gridDim.x) - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (rs[mid] <= u)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}
__device__ __forceinline__ PieceInfo piece_info(const Seg& sg, int t, const int* rs) {
  PieceInfo pi;
  pi.c0 = tail_cta_rs(sg.xs, rs);
  pi.np = tail_cta_rs(sg.xs + sg.w.n[t] - 1, rs) - pi.c0 + 1;
  pi.k = static_cast<int>(blockIdx.x) - pi.c0;
  return pi;
}
// Workspace slot of piece k of the item: the piece is the first tail
// segment of its CTA (slot 0) unless it is the last one of CTA c0 whose
// range starts before the item (slot 1).
__device__ __forceinline__ int piece_slot(const Seg& sg, const PieceInfo& pi, int k,
                                          const int* rs) {
  const int cta = pi.c0 + k;
  const int which = (k == 0 && rs[pi.c0] < sg.xs) ? 1 : 0;
  return cta * 2 + which;
}

// The forward kernel's form of the bounded wait: the limit and the status
// words are read from the kernel parameters where the slow path needs them,
// so that no thread keeps them in registers.  honour_abort = false waits out
// the limit even after another thread gave up (used to drain copies and
// MMAs before the CTA exits).
template <typename CtrlT>
__device__ __forceinline__ bool wait_fwd(uint32_t bar, uint32_t parity, CtrlT* c,
                                         const AttnParams& p, unsigned where,
                                         bool honour_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  volatile uint32_t* abort = &c->abort;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (honour_abort && *abort) return false;
    if (global_timer_ns() - t0 > p.timeout_ns) {
      *abort = 1u;
      atomicCAS(p.status, 0u, kStatusTimeout);
      atomicExch(p.where, where);
      return false;
    }
  }
}


// ---------------------------------------------------------------------------
// producer

template <int DT, int D, bool CAUSAL>
__device__ void role_producer_tail(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                              const CUtensorMap* tmV, uint8_t* sbase,
                              CtrlTail<Cfg<DT, D>::kSlots>* c, const AttnParams& p) {
  using C = Cfg<DT, D>;
  const uint8_t* sq = sbase;
  const uint32_t skv = smem_u32(sbase + C::kNQT * C::kTileBytes);
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
    if (!wait_fwd(smem_u32(&c->kv_empty[st]), par ^ 1u, c, p, 0x02)) return false;
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

  bool k0_loaded = false;  // the segment's first K went out with the previous segment's last V
  SegIter<C::kNQT, CAUSAL> segs;
  segs.init(p);
  Seg sg, sn;
  bool have = segs.next(sg, p);
  bool has_next = have && segs.next(sn, p);
  while (have && ok) {
    const Item& w = sg.w;
    // Q tiles with key blocks in this segment
#pragma unroll
    for (int t = 0; t < C::kNQT; ++t) {
      if (seg_end(sg, t) <= sg.jb) continue;
      const uint32_t full = smem_u32(&c->q_full[t]);
      if (!wait_fwd(smem_u32(&c->q_empty[t]), (q_uses[t] & 1u) ^ 1u, c, p, 0x01)) {
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
      // stages (V_j, next K): K_{j+1}, or the next segment's first K
      if (ok && !k0_loaded) ok = fill(-1, 0, sg.jb * kBlock, w.bh);
      for (int j = sg.jb; j < sg.je && ok; ++j) {
        if (j + 1 < sg.je)
          ok = fill(j * kBlock, w.bh, (j + 1) * kBlock, w.bh);
        else
          ok = fill(j * kBlock, w.bh, has_next ? sn.jb * kBlock : -1, has_next ? sn.w.bh : 0);
      }
      k0_loaded = has_next;
    } else {
      // one tile per stage: K_j, then V_j
      for (int j = sg.jb; j < sg.je && ok; ++j) {
        ok = fill(-1, 0, j * kBlock, w.bh);
        if (ok) ok = fill(j * kBlock, w.bh, -1, 0);
      }
    }
    sg = sn;
    have = has_next;
    if (have) has_next = segs.next(sn, p);
  }
  // Never leave a copy in flight: wait until the last fill of every stage
  // and of every Q tile has landed (immediate on the normal path).
  for (int st = 0; st < C::kStages; ++st) {
    const uint32_t uses =
        stages / C::kStages + (static_cast<uint32_t>(st) < stages % C::kStages ? 1u : 0u);
    if (uses) {
      wait_fwd(smem_u32(&c->kv_full[st]), (uses - 1u) & 1u, c, p, 0x03, false);
    }
  }
  for (int t = 0; t < C::kNQT; ++t) {
    if (q_uses[t]) {
      wait_fwd(smem_u32(&c->q_full[t]), (q_uses[t] - 1u) & 1u, c, p, 0x04, false);
    }
  }
}


// ---------------------------------------------------------------------------
// MMA issuer (one thread)

template <int DT, int D, bool CAUSAL>
__device__ void role_mma_tail(uint8_t* sbase, CtrlTail<Cfg<DT, D>::kSlots>* c, uint32_t tbase,
                         const AttnParams& p) {
  using C = Cfg<DT, D>;
  constexpr int NQT = C::kNQT;
  const uint32_t sq = smem_u32(sbase);
  const uint32_t skv = sq + NQT * C::kTileBytes;
  uint32_t q_waits[2] = {0, 0}, p_waits[2] = {0, 0};
  RingPos ring;
  bool ok = true;

  // S_t(jb), the first S of tile t in segment g, with K_jb in stage ks;
  // false when a wait gave up
  auto issue_s0 = [&](const Seg& g, int t, int ks) -> bool {
    if (!wait_fwd(smem_u32(&c->q_full[t]), q_waits[t] & 1u, c, p, 0x12)) return false;
    ++q_waits[t];
    tc_fence_after_sync();
    issue_qk<DT, D>(tbase + C::s_col(t), sq + t * C::kTileBytes,
                    skv + C::k_slot(ks) * C::kTileBytes);
    mma_commit(smem_u32(&c->s_full[t]));
    if (seg_end(g, t) == g.jb + 1) mma_commit(smem_u32(&c->q_empty[t]));
    return true;
  };

  // Where C::kEarlyS0 holds, the next segment's first S_t goes out right
  // behind this segment's last P_t V when its K and Q_t are already here:
  // the tensor pipe runs one thread's MMAs in order, so that S_t overwrites
  // P_t only after that product has read it, and the next segment's first
  // softmax starts without waiting for the rest of this segment.
  constexpr bool kEarly = C::kEarlyS0;
  bool s0_issued = false;  // this segment's first S went out during the previous one
  int held = -1;           // stage that holds this segment's first K (paired stages)
  SegIter<NQT, CAUSAL> segs;
  segs.init(p);
  Seg sg, sn;
  bool have = segs.next(sg, p);
  bool has_next = have && segs.next(sn, p);
  while (have && ok) {
    if (!s0_issued) {
      int ks = held;
      if (ks < 0) {
        uint32_t kpar;
        ring.next<C::kStages>(ks, kpar);
        if (!wait_fwd(smem_u32(&c->kv_full[ks]), kpar, c, p, 0x11)) break;
      }
      for (int t = 0; t < NQT && ok; ++t)
        if (seg_end(sg, t) > sg.jb) ok = issue_s0(sg, t, ks);
      if (!ok) break;
      mma_commit(smem_u32(&c->kv_empty[ks]));
      held = -1;
    }
    s0_issued = false;

    for (int j = sg.jb; j < sg.je && ok; ++j) {
      int vs;
      uint32_t vpar;
      ring.next<C::kStages>(vs, vpar);
      if (!wait_fwd(smem_u32(&c->kv_full[vs]), vpar, c, p, 0x13)) {
        ok = false;
        break;
      }
      const bool last = j + 1 == sg.je;
      const bool ahead = kEarly && last && has_next;  // the next segment's first S
      // stage of the next K: the same one when stages are paired
      int ns = vs;
      uint32_t npar = vpar;
      bool k_ready = C::kPair;
      bool s0_done[2] = {false, false};
      if (!C::kPair && (!last || ahead)) ring.next<C::kStages>(ns, npar);
      const uint32_t sv = skv + C::v_slot(vs) * C::kTileBytes;
      const uint32_t sk = skv + C::k_slot(ns) * C::kTileBytes;
      for (int t = 0; t < NQT && ok; ++t) {
        const int te = seg_end(sg, t);
        if (j < te) {
          // first key half as soon as its P and the rescaled O are there
          // (p_full[t][0] counts the softmax and the correction warps),
          // overlapping the softmax of the second half
          if (!wait_fwd(smem_u32(&c->p_full[t][0]), p_waits[t] & 1u, c, p, 0x14)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          issue_pv_half<DT, D, 0>(tbase + C::o_col(t), tbase + C::s_col(t), sv, j > sg.jb);
          if (!wait_fwd(smem_u32(&c->p_full[t][1]), p_waits[t] & 1u, c, p, 0x18)) {
            ok = false;
            break;
          }
          ++p_waits[t];
          tc_fence_after_sync();
          issue_pv_half<DT, D, 1>(tbase + C::o_col(t), tbase + C::s_col(t), sv, true);
          // O_t is complete for the epilogue after the tile's last block;
          // for earlier blocks the correction warps need no signal of their
          // own: they rescale O_t for block j + 1 only after alpha_t(j + 1),
          // which the softmax publishes after S_t(j + 1) completed, and that
          // commit tracks this P_t V too
          if (j + 1 == te) mma_commit(smem_u32(&c->o_full[t]));
        }
        if (j + 1 < te) {
          if (!k_ready) {
            if (!wait_fwd(smem_u32(&c->kv_full[ns]), npar, c, p, 0x16)) {
              ok = false;
              break;
            }
            k_ready = true;
          }
          issue_qk<DT, D>(tbase + C::s_col(t), sq + t * C::kTileBytes, sk);
          mma_commit(smem_u32(&c->s_full[t]));
          if (j + 2 == te) mma_commit(smem_u32(&c->q_empty[t]));
        }
        if constexpr (kEarly) {
          // only where the K and Q_t are already here: the other tile's P V
          // must not wait behind them
          if (ahead && seg_end(sn, t) > sn.jb) {
            if (!k_ready) k_ready = mbar_test_wait(smem_u32(&c->kv_full[ns]), npar);
            if (k_ready && mbar_test_wait(smem_u32(&c->q_full[t]), q_waits[t] & 1u)) {
              ok = issue_s0(sn, t, ns);
              s0_done[t] = true;
            }
          }
        }
      }
      if (!ok) break;
      if constexpr (!C::kPair) mma_commit(smem_u32(&c->kv_empty[vs]));
      if (!last || ahead) {
        if (!k_ready && !wait_fwd(smem_u32(&c->kv_full[ns]), npar, c, p, 0x16)) break;
        if constexpr (kEarly) {
          for (int t = 0; t < NQT && ok && ahead; ++t)
            if (!s0_done[t] && seg_end(sn, t) > sn.jb) ok = issue_s0(sn, t, ns);
          if (!ok) break;
          s0_issued = ahead;
        }
        mma_commit(smem_u32(&c->kv_empty[ns]));
      } else if constexpr (C::kPair) {
        // the segment's last block: this stage also holds the next
        // segment's first K, used by its first S before the stage is
        // released
        if (has_next)
          held = vs;
        else
          mma_commit(smem_u32(&c->kv_empty[vs]));
      }
    }
    sg = sn;
    have = has_next;
    if (have) has_next = segs.next(sn, p);
  }
  // Wait until every MMA issued above has completed before the CTA frees
  // Tensor Memory.
  mma_commit(smem_u32(&c->drain));
  wait_fwd(smem_u32(&c->drain), 0u, c, p, 0x17, false);
}


// ---------------------------------------------------------------------------
// softmax warpgroup of tile t

template <int DT, int D, bool CAUSAL>
__device__ void role_softmax_tail(int t, CtrlTail<Cfg<DT, D>::kSlots>* c, uint32_t tbase,
                             const AttnParams& p) {
  using C = Cfg<DT, D>;
  const uint32_t lane = lane_id();
  const uint32_t wq = (threadIdx.x >> 5) & 3u;  // warp quarter = TMEM lane group
  const int r = static_cast<int>(wq * 32u + lane);
  const uint32_t taddr = tbase + ((wq * 32u) << 16) + C::s_col(t);
  const float sl2 = p.scale_log2;
  uint32_t s_waits = 0;
  uint32_t iter = 0;  // segments walked (the parity selects the hand-over slots)

  SegIter<C::kNQT, CAUSAL> segs;
  segs.init(p);
  Seg sg;
  for (; segs.next(sg, p); ++iter) {
    const Item& w = sg.w;
    const int qt = w.qt0 + t;
    const int n = seg_end(sg, t);  // blocks [sg.jb, n) of this tile
    if (n <= sg.jb) continue;
    // the segment holds all of the tile's blocks (else it is one piece)
    const bool whole = sg.jb == 0 && sg.je >= w.n[t];
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
    for (int j = sg.jb; j < n; ++j) {
      if (!wait_fwd(smem_u32(&c->s_full[t]), s_waits & 1u, c, p, 0x21)) return;
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
        tmem_ld_2x64(taddr, raw);
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
      // alpha for the O rescale; the segment's first block has no O to
      // rescale, and publishes none
      if (j > sg.jb) {
        *alpha_dst = alpha;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&c->sc_full[t]));
      }

      // P over the first kPCols columns of S (already in registers), in two
      // halves of 64 keys: the first is handed to the MMA issuer while the
      // second is computed
      const float neg_m = -m_use;
      const float sum0 = exp_store_chunk<DT, 0, 64>(s, sl2j, neg_m, taddr);
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&c->p_full[t][0]));
      const float sum1 = exp_store_chunk<DT, 64, 64>(s, sl2j, neg_m, taddr + C::kPCols / 2);
      l_run = alpha * l_run + (sum0 + sum1);
      tmem_st_wait();
      // hand 1/l (a piece: its reference m and its sum l) to the epilogue
      // before the last P is announced
      if (j == n - 1) {
        if (whole) {
          *inv_l_dst = __frcp_rn(l_run);
        } else {
          *inv_l_dst = l_run;
          c->part_m[iter & 1u][t][r] = m_use;
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&c->p_full[t][1]));
    }
    // LSE (natural log) of the real rows; the epilogue writes it for a
    // piece, once the pieces are merged
    const int row = qt * kBlock + r;
    if (whole && row < p.N) {
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      p.lse[static_cast<size_t>(w.bh) * p.N + row] = (m_use + __log2f(l_run)) * 0.6931471805599453f;
    }
  }
}


// ---------------------------------------------------------------------------
// correction / epilogue warpgroup

// Output stores: the tile is staged through shared memory, one 128-row x
// 64-column box at a time in the 128-byte-swizzled layout the O tensor map
// uses, and written by TMA tensor stores, so that every global write is a
// whole coalesced box; rows past N are clipped by the tensor map.
//
// A piece of a split tile instead leaves its unnormalised O (from Tensor
// Memory), its subtraction reference m and its sum l in the workspace and
// counts itself on the tile's flag; the piece that finds all the others
// done merges them, by the rescale of the concept card's "Implementation
// sketch" (every piece's O and l scaled by exp2(m_k - M) for the largest
// reference M), and writes O and LSE.
template <int DT, int D, bool CAUSAL>
__device__ void role_correction_tail(CtrlTail<Cfg<DT, D>::kSlots>* c, uint32_t tbase, uint32_t stage,
                                uint32_t region, const CUtensorMap* tmO, const AttnParams& p) {
  using C = Cfg<DT, D>;
  constexpr int NQT = C::kNQT;
  const uint32_t lane = lane_id();
  const uint32_t wq = (threadIdx.x >> 5) & 3u;
  const int r = static_cast<int>(wq * 32u + lane);
  const uint32_t lane_off = (wq * 32u) << 16;
  const bool issuer = r == 0;  // issues and tracks the TMA stores, reads and bumps flags
  const uint32_t stage_row = stage + static_cast<uint32_t>(r) * 128u;
  // bytes of the Q tiles and the K/V ring, free after the CTA's last MMA
  constexpr int kRegionBytes = (NQT + C::kSlots) * C::kTileBytes;
  uint32_t sc_waits[2] = {0, 0}, o_waits[2] = {0, 0};
  bool arrived[2] = {false, false};  // the segment's first-block arrival is made
  bool dep_done = false;             // the issuer waited for the grid before
  bool ok = true;

  // This warp's arrival on p_full[t][0]: its rows of O_t are rescaled, or
  // (for the next segment's first block) read out of Tensor Memory.
  auto arrive_p0 = [&](int t) {
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&c->p_full[t][0]));
  };

  // Write tile (qt, bh): get(col, x) yields 16 output values of this row
  // from column col on (already scaled); after the last get, release O_t
  // (release_t >= 0) for the next segment.
  auto store_tile = [&](int qt, int bh, int release_t, auto&& get) {
#pragma unroll 1
    for (int bx = 0; bx < D / 64; ++bx) {
      // the previous store has finished reading the staging box
      if (issuer) bulk_wait_read_all();
      named_bar_sync(1, 128);
#pragma unroll 1
      for (int g = 0; g < 4; ++g) {
        float x[16];
        get(bx * 64 + g * 16, x);
        // 16-byte chunk k of the row sits at chunk k ^ (row mod 8)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint32_t k = static_cast<uint32_t>(2 * g + i);
          st_shared_v4(stage_row + ((k ^ (static_cast<uint32_t>(r) & 7u)) << 4),
                       pack8_out<DT>(x + 8 * i));
        }
      }
      if (release_t >= 0 && bx == D / 64 - 1) arrive_p0(release_t);
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (issuer && qt * kBlock < p.N) {
        tma_store_3d(tmO, stage, bx * 64, qt * kBlock, bh);
        bulk_commit_group();
      }
    }
  };

  SegIter<NQT, CAUSAL> segs;
  segs.init(p);
  Seg sg;
  bool have = segs.next(sg, p);
  uint32_t iter = 0;
  while (have && ok) {
    const Item& w = sg.w;
    // tiles with blocks in the next segment (its first P_t V waits for O_t
    // to be read out here)
    bool next_active[2] = {false, false};
    bool final_seg = true;  // the CTA's last segment
    {
      SegIter<NQT, CAUSAL> look = segs;
      Seg sn;
      if (look.next(sn, p)) {
        final_seg = false;
#pragma unroll
        for (int t = 0; t < NQT; ++t) next_active[t] = seg_end(sn, t) > sn.jb;
      }
    }
    for (int j = sg.jb; j < sg.je && ok; ++j) {
      for (int t = 0; t < NQT; ++t) {
        if (j >= seg_end(sg, t)) continue;
        if (j == sg.jb) {
          // the first block: nothing to rescale; the arrival was made when
          // the previous segment's epilogue had read O_t, if it had one
          if (!arrived[t]) arrive_p0(t);
          arrived[t] = false;
          continue;
        }
        if (!wait_fwd(smem_u32(&c->sc_full[t]), sc_waits[t] & 1u, c, p, 0x31)) {
          ok = false;
          break;
        }
        ++sc_waits[t];
        const float alpha = c->alpha[t][r];
        {
          // P_t V_{j-1} has completed: alpha_t(j) was published after
          // S_t(j), whose commit came after that product
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
        arrive_p0(t);
      }
    }
    // ---- epilogue: O / l (times the v descale) -> output dtype ----
    // The tiles with blocks in this segment, whether the segment holds all
    // of a tile's blocks (whole) or one piece of them.
    bool act[2] = {false, false}, whole[2] = {false, false}, last[2] = {false, false};
    bool wrote[2] = {false, false};  // left in the workspace, O_t handed on
    PieceInfo pis[2];
    bool any_piece = false;
#pragma unroll
    for (int t = 0; t < NQT; ++t) {
      act[t] = seg_end(sg, t) > sg.jb;
      whole[t] = act[t] && sg.jb == 0 && sg.je >= w.n[t];
      if (act[t] && !whole[t]) {
        pis[t] = piece_info(sg, t, c->rs);
        any_piece = true;
      }
    }
    // O of every tile complete.  After the CTA's last segment no MMA or
    // copy uses the Q tiles and the K/V ring any more once this holds, and
    // a merge may stage the other pieces there.
    for (int t = 0; t < NQT && ok; ++t) {
      if (!act[t]) continue;
      if (!wait_fwd(smem_u32(&c->o_full[t]), o_waits[t] & 1u, c, p, 0x33)) {
        ok = false;
        break;
      }
      ++o_waits[t];
    }
    if (!ok) break;
    tc_fence_after_sync();
    auto part_at = [&](int t, int k) {
      return p.part + (static_cast<size_t>(piece_slot(sg, pis[t], k, c->rs)) * NQT + t) *
                          C::kPartFloats;
    };
    if (any_piece) {
      // Settle the pieces of both tiles together: one read of the flags;
      // a piece that is not the last leaves its O, m and l and counts
      // itself (one fence, one round of atomics); a piece that finds (or
      // makes) the count complete merges below.  The flags were cleared by
      // the grid before this one, which may still be running.
      if (issuer) {
        if (!dep_done) {
          griddep_wait();
          dep_done = true;
        }
#pragma unroll
        for (int t = 0; t < NQT; ++t)
          if (act[t] && !whole[t]) c->bcast2[t] = ld_acquire_gpu(p.flags + sg.ti * 2 + t);
      }
      named_bar_sync(1, 128);
      bool any_write = false;
#pragma unroll
      for (int t = 0; t < NQT; ++t) {
        if (!act[t] || whole[t]) continue;
        last[t] = c->bcast2[t] + 1u == static_cast<uint32_t>(pis[t].np);
        any_write |= !last[t];
      }
      named_bar_sync(1, 128);
      if (any_write) {
#pragma unroll
        for (int t = 0; t < NQT; ++t) {
          if (!act[t] || whole[t] || last[t]) continue;
          float* own = part_at(t, pis[t].k);
          float4* own4 = reinterpret_cast<float4*>(own) + r;
          const uint32_t ta = tbase + lane_off + C::o_col(t);
#pragma unroll 1
          for (int cc = 0; cc < D; cc += 16) {
            uint32_t v[16];
            tmem_ld_x16(ta + cc, v);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              own4[(cc / 4 + q) * kBlock] =
                  make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                              __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
          }
          own[D * kBlock + r] = c->part_m[iter & 1u][t][r];
          own[(D + 1) * kBlock + r] = c->inv_l[iter & 1u][t][r];
          // O_t is read out: the next segment may overwrite it (should this
          // piece still turn out to be the last, it merges its own O from
          // the workspace)
          wrote[t] = true;
          if (next_active[t]) arrive_p0(t);
        }
        __threadfence();
        named_bar_sync(1, 128);
        if (issuer) {
#pragma unroll
          for (int t = 0; t < NQT; ++t)
            if (act[t] && !whole[t] && !last[t])
              c->bcast2[t] = atom_add_acq_rel_gpu(p.flags + sg.ti * 2 + t, 1u) + 1u;
        }
        named_bar_sync(1, 128);
#pragma unroll
        for (int t = 0; t < NQT; ++t)
          if (act[t] && !whole[t] && !last[t])
            last[t] = c->bcast2[t] == static_cast<uint32_t>(pis[t].np);
        named_bar_sync(1, 128);
      }
      if (last[0] || last[1]) __threadfence();
    }
    // Merge of tile t (this piece found the count complete): M = largest
    // reference, L = sum of exp2(m_k - M) l_k, O = sum of exp2(m_k - M) O_k
    // / L, summed in piece order whichever piece merges, so the result does
    // not depend on which CTA finished last.  After the CTA's last segment
    // the other pieces' (O, m, l) rows are first copied into the free shared
    // memory (each thread copies, then reads, only its own row, so no
    // barrier is needed), which puts all of the loads in flight at once;
    // otherwise they are read from L2 as they are needed.
    auto merge_tile = [&](int t, int qt, int row, uint32_t ta, int release_t) {
      const PieceInfo& pi = pis[t];
      const float m_own = c->part_m[iter & 1u][t][r];
      const float l_own = c->inv_l[iter & 1u][t][r];
      // pieces read from the workspace: the others, and this one too once
      // its own O was handed on
      const int n_other = pi.np - 1 + (wrote[t] ? 1 : 0);
      const bool staged = final_seg && n_other * (D + 2) * kBlock * 4 <= kRegionBytes;
      const uint32_t m_base = region + static_cast<uint32_t>(n_other * (D / 4) * kBlock) * 16u;
      const uint32_t l_base = m_base + static_cast<uint32_t>(n_other * kBlock) * 4u;
      if (staged) {
        int kk = 0;
        for (int k = 0; k < pi.np; ++k) {
          if (k == pi.k && !wrote[t]) continue;
          const float* pk = part_at(t, k);
          const float4* src = reinterpret_cast<const float4*>(pk) + r;
          const uint32_t dst = region + (static_cast<uint32_t>(kk * (D / 4)) * kBlock + r) * 16u;
#pragma unroll 8
          for (int c4 = 0; c4 < D / 4; ++c4) cp_async_16(dst + c4 * kBlock * 16u, src + c4 * kBlock);
          cp_async_4(m_base + (kk * kBlock + r) * 4u, pk + D * kBlock + r);
          cp_async_4(l_base + (kk * kBlock + r) * 4u, pk + (D + 1) * kBlock + r);
          ++kk;
        }
        cp_async_wait_all();
      }
      auto m_of = [&](int k, int kk) {
        return staged ? ld_shared_f32(m_base + (kk * kBlock + r) * 4u)
                      : __ldcg(part_at(t, k) + D * kBlock + r);
      };
      auto l_of = [&](int k, int kk) {
        return staged ? ld_shared_f32(l_base + (kk * kBlock + r) * 4u)
                      : __ldcg(part_at(t, k) + (D + 1) * kBlock + r);
      };
      // kk: index of piece k among the pieces read from the workspace
      float mx = m_own;
      for (int k = 0, kk = 0; k < pi.np; ++k) {
        if (k != pi.k) mx = fmaxf(mx, m_of(k, kk));
        if (k != pi.k || wrote[t]) ++kk;
      }
      const float a_own = ex2_approx(m_own - mx);
      float lsum = 0.0f;
      for (int k = 0, kk = 0; k < pi.np; ++k) {
        if (k == pi.k) {
          lsum = fmaf(a_own, l_own, lsum);
        } else {
          lsum = fmaf(ex2_approx(m_of(k, kk) - mx), l_of(k, kk), lsum);
        }
        if (k != pi.k || wrote[t]) ++kk;
      }
      const float g = p.out_scale / lsum;
      store_tile(qt, w.bh, release_t, [&](int col, float (&x)[16]) {
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = 0.0f;
        int kk = 0;
#pragma unroll 1
        for (int k = 0; k < pi.np; ++k) {
          if (k == pi.k && !wrote[t]) {
            uint32_t v[16];
            tmem_ld_x16(ta + col, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = fmaf(a_own, __uint_as_float(v[i]), x[i]);
            continue;
          }
          float4 y[4];
          if (staged) {
            const uint32_t src =
                region + (static_cast<uint32_t>(kk * (D / 4) + col / 4) * kBlock + r) * 16u;
#pragma unroll
            for (int q = 0; q < 4; ++q) y[q] = ld_shared_v4f(src + q * kBlock * 16u);
          } else {
            const float4* pk4 =
                reinterpret_cast<const float4*>(part_at(t, k)) + (col / 4) * kBlock + r;
#pragma unroll
            for (int q = 0; q < 4; ++q) y[q] = __ldcg(pk4 + q * kBlock);
          }
          // (this piece's own O, handed on, comes back from the workspace)
          const float ak = k == pi.k ? a_own : ex2_approx(m_of(k, kk) - mx);
          ++kk;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            x[4 * q] = fmaf(ak, y[q].x, x[4 * q]);
            x[4 * q + 1] = fmaf(ak, y[q].y, x[4 * q + 1]);
            x[4 * q + 2] = fmaf(ak, y[q].z, x[4 * q + 2]);
            x[4 * q + 3] = fmaf(ak, y[q].w, x[4 * q + 3]);
          }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] *= g;
      });
      if (row < p.N)
        p.lse[static_cast<size_t>(w.bh) * p.N + row] = (mx + __log2f(lsum)) * 0.6931471805599453f;
    };
    // each tile: store it (whole), merge it (the last piece), or hand its
    // Tensor Memory columns to the next segment
    for (int t = 0; t < NQT; ++t) {
      if (!act[t]) continue;
      const int qt = w.qt0 + t;
      const int row = qt * kBlock + r;
      const uint32_t ta = tbase + lane_off + C::o_col(t);
      // the next segment's first P_t V may overwrite O_t once it is read
      const int release_t = next_active[t] ? t : -1;
      if (whole[t]) {
        const float f = c->inv_l[iter & 1u][t][r] * p.out_scale;
        store_tile(qt, w.bh, release_t, [&](int col, float (&x)[16]) {
          uint32_t v[16];
          tmem_ld_x16(ta + col, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] = __uint_as_float(v[i]) * f;
        });
      } else if (last[t]) {
        merge_tile(t, qt, row, ta, wrote[t] ? -1 : release_t);
      } else if (release_t >= 0 && !wrote[t]) {
        arrive_p0(release_t);
      }
      arrived[t] = release_t >= 0;
    }
    ++iter;
    have = segs.next(sg, p);
  }
  // no store may still read shared memory (or be in flight) when the CTA
  // exits
  if (issuer) bulk_wait_all();
}


// ---------------------------------------------------------------------------

template <int DT, int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tail_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const AttnParams p) {
  using C = Cfg<DT, D>;
  using CtrlT = CtrlTail<C::kSlots>;
  static_assert(sizeof(CtrlT) + 1024 <= C::kMiscBytes + kTailCtrlExtra, "control block budget");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // tiles need 1024-byte alignment (128-byte swizzle atoms)
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* sbase = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t stage = smem_u32(sbase + (C::kNQT + C::kSlots) * C::kTileBytes);
  CtrlT* c = reinterpret_cast<CtrlT*>(sbase + (C::kNQT + C::kSlots) * C::kTileBytes +
                                      C::kStageTotal);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&c->q_full[t]), 1);
      mbar_init(smem_u32(&c->q_empty[t]), 1);
      mbar_init(smem_u32(&c->s_full[t]), 1);
      mbar_init(smem_u32(&c->p_full[t][0]), 8);
      mbar_init(smem_u32(&c->p_full[t][1]), 4);
      mbar_init(smem_u32(&c->sc_full[t]), 4);
      mbar_init(smem_u32(&c->o_full[t]), 1);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&c->kv_full[s]), 1);
      mbar_init(smem_u32(&c->kv_empty[s]), 1);
    }
    mbar_init(smem_u32(&c->drain), 1);
    c->abort = 0u;
    fence_mbar_init();
  }
  for (int i = static_cast<int>(threadIdx.x); i <= static_cast<int>(gridDim.x); i += kThreads)
    c->rs[i] = tail_range_start(i, p);
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
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = c->tmem_base;

  // Role dispatch by warpgroup, with the register file split among them
  // (88 + 2 * 168 + 88: the merging epilogue needs more than the main
  // kernel's correction warps get).
  static_assert(kTailRegsControl + 2 * kRegsSoftmax + kTailRegsCorrection <= 4 * 128,
                "register split");
  const uint32_t wg = warp >> 2;
  if (wg == 0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kTailRegsControl));
    if (warp == 0 && lane == 0)
      role_producer_tail<DT, D, CAUSAL>(&tmQ, &tmK, &tmV, sbase, c, p);
    else if (warp == 1 && lane == 0)
      role_mma_tail<DT, D, CAUSAL>(sbase, c, tbase, p);
  } else if (wg == 1 || wg == 2) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    if (static_cast<int>(wg) - 1 < C::kNQT) role_softmax_tail<DT, D, CAUSAL>(wg - 1, c, tbase, p);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kTailRegsCorrection));
    role_correction_tail<DT, D, CAUSAL>(c, tbase, stage, smem_u32(sbase), &tmO, p);
  }

  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, C::kTmemCols);
  }
  // this grid completes only after the one before it (a no-op when it was
  // launched without programmatic serialization)
  if (threadIdx.x == 0) griddep_wait();
}

}  // namespace wsattn

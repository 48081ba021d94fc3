// fwd_common.cuh -- device helpers shared by the forward kernels: the unit
// schedule (which (head, query-tile pair) a CTA takes next), the kv-tile range
// of a query tile under masks and key counts, and bounded waits.
#pragma once

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

// The r-th unit this CTA processes (-1 when it has no more).  Every role of
// the CTA walks the same sequence.
__device__ __forceinline__ int cta_unit(const FwdArgs& a, int r) {
  int k;
  if (a.sched == 2) {
    // boustrophedon: each round of gridDim.x units alternates direction, so
    // CTAs that got a longer unit in one round get a shorter one in the next
    k = r * (int)gridDim.x + ((r & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x);
  } else {
    k = blockIdx.x + r * gridDim.x;
  }
  return k < a.n_units ? k : -1;
}

// Unit u -> (flat batch*head index, tile pair p: query tiles 2p and 2p+1).
//   sched 0:     head-major (non-causal, and windows), so CTAs running at the
//                same time share the K/V of few heads in L2.
//   sched 2:     longest pairs of every head first (causal work grows with the
//                pair index), dealt in a snake.
//   sched 3:     split-KV; the pairs of one (head, split) are adjacent, so
//                they run together and share that split's K/V in L2.
__device__ __forceinline__ void unit_coords(const FwdArgs& a, int u, int& bh, int& pair,
                                            int& split) {
  const int np = a.n_pairs;
  split = 0;
  if (a.sched == 3) {
    const int rest = u / np;
    pair = u - rest * np;
    bh = rest / a.n_split;
    split = rest - bh * a.n_split;
    return;
  }
  if (a.sched == 2) {
    const int BH = a.B * a.Hq;
    pair = np - 1 - u / BH;
    bh = u - (u / BH) * BH;
    return;
  }
  bh = u / np;
  pair = u - bh * np;
}

// Keys of batch b that exist: seqlens_k[b] clamped to [0, Sk] (the key padding
// mask); all Sk without lengths, and always in the plain kernel.
template <bool kWin>
__device__ __forceinline__ int batch_kv_len(const FwdArgs& a, int b) {
  if (!kWin || !a.seqlens_k) return a.Sk;
  const int n = __ldg(a.seqlens_k + b);
  return n < 0 ? 0 : (n < a.Sk ? n : a.Sk);
}

// kv tiles [lo, hi) that query tile qt sees under the window (wl, wr) among the
// first kv_len keys (empty when the tile lies past Sq or sees no key)
__device__ __forceinline__ void tile_kv_range(const FwdArgs& a, int wl, int wr, int kv_len, int qt,
                                              int& lo, int& hi) {
  lo = hi = 0;
  if (qt * kTile >= a.Sq) return;
  const int last = min(a.Sq, (qt + 1) * kTile) - 1;  // last query row of the tile
  const int lo_key = wl >= 0 ? max(0, qt * kTile - wl) : 0;
  const int hi_key = wr >= 0 ? min(kv_len, last + wr + 1) : kv_len;
  lo = lo_key / kTile;
  hi = max(lo, (hi_key + kTile - 1) / kTile);
}

// A tile's range cut to the kv tiles of `split` (kSplit); may become empty.
template <bool kSplit>
__device__ __forceinline__ void split_kv_range(const FwdArgs& a, int wl, int wr, int kv_len, int qt,
                                               int split, int& lo, int& hi) {
  tile_kv_range(a, wl, wr, kv_len, qt, lo, hi);
  if (kSplit) {
    const int s0 = split * a.split_tiles;
    lo = max(lo, s0);
    hi = max(lo, min(hi, s0 + a.split_tiles));
  }
}

// The kv tiles the two query tiles of a pair stream: lo[t], hi[t] per tile,
// and their union [jlo, jlo + nmax).  An empty tile gets lo = hi = jlo; both
// empty: nmax = 0 and the unit is skipped.
template <bool kSplit>
__device__ __forceinline__ void pair_kv_span(const FwdArgs& a, int wl, int wr, int kv_len, int pair,
                                             int split, int lo[2], int hi[2], int& jlo, int& nmax) {
  split_kv_range<kSplit>(a, wl, wr, kv_len, 2 * pair, split, lo[0], hi[0]);
  split_kv_range<kSplit>(a, wl, wr, kv_len, 2 * pair + 1, split, lo[1], hi[1]);
  const bool e0 = hi[0] <= lo[0], e1 = hi[1] <= lo[1];
  if (e0 && e1) {
    jlo = lo[0];
    nmax = 0;
    return;
  }
  jlo = e0 ? lo[1] : (e1 ? lo[0] : min(lo[0], lo[1]));
  const int jend = e0 ? hi[1] : (e1 ? hi[0] : max(hi[0], hi[1]));
  nmax = jend - jlo;
  if (e0) lo[0] = hi[0] = jlo;
  if (e1) lo[1] = hi[1] = jlo;
}

// Bounded wait done by every lane of a warp; the outcome is made warp-uniform so
// the warp-collective tcgen05.ld/st that follow are never reached by part of it.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait used only while draining at exit: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitTimeoutNs) break;
  }
}

}  // namespace fa

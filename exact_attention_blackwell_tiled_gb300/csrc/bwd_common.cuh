// bwd_common.cuh -- device helpers shared by the backward main kernels
// (64-row and 128-row query blocks, CTA pairs): the visibility window, the kv
// tile -> query block ranges and the deterministic chain's contributors, the
// unit schedule, bounded waits, the TMEM load / store shapes they use, and the
// cluster and 2-CTA (cta_group::2) building blocks of the pair kernel.
#pragma once

#include <climits>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

// The window (wl, wr) a kernel instantiation applies: kMod reads it from the
// arguments, the plain kernel has none or the causal one.
template <bool kMod>
__device__ __forceinline__ int win_left(const BwdArgs& a) {
  return kMod ? a.wl : -1;
}
template <bool kMod>
__device__ __forceinline__ int win_right(const BwdArgs& a) {
  return kMod ? a.wr : (a.causal ? 0 : -1);
}

// Keys of batch b that exist: seqlens_k[b] clamped to [0, Sk] (the key padding
// mask); all Sk without lengths, and always in the plain kernel.
template <bool kMod>
__device__ __forceinline__ int bwd_kv_len(const BwdArgs& a, int b) {
  if (!kMod || !a.seqlens_k) return a.Sk;
  const int n = __ldg(a.seqlens_k + b);
  return n < 0 ? 0 : (n < a.Sk ? n : a.Sk);
}

// QB-row query blocks [lo, hi) with a query that sees a key of kv tile j (of a
// batch with kv_len keys): the queries from (first key - wr) to (last key +
// wl); empty when the tile holds no key of the batch
template <bool kMod, int QB>
__device__ __forceinline__ void bwd_qblk_range(const BwdArgs& a, int j, int kv_len, int& lo,
                                               int& hi) {
  const int wl = win_left<kMod>(a), wr = win_right<kMod>(a);
  const int k0 = j * kTile;
  if (k0 >= kv_len) {
    lo = hi = 0;
    return;
  }
  const int k1 = min(kv_len, k0 + kTile) - 1;
  const int q_lo = wr >= 0 ? max(0, k0 - wr) : 0;
  const int q_hi = wl >= 0 ? min(a.Sq - 1, k1 + wl) : a.Sq - 1;
  lo = q_lo / QB;
  hi = q_hi >= q_lo ? q_hi / QB + 1 : lo;
}

// The first kv tile that adds into 64-row query block iq: the kv tiles that do
// (those whose bwd_qblk_range holds iq) are a contiguous run, since both ends
// of that range grow with j, and the run starts at the first tile whose last
// key reaches the block's first query - wl.  (The bound can overshoot only when
// no tile adds at all, which a caller that adds never meets.)
template <int QB>
__device__ __forceinline__ int qblk_first_contributor(int wl, int iq) {
  return wl >= 0 ? max(0, iq * QB - wl) / kTile : 0;
}

template <bool kMod, int QB>
__device__ __forceinline__ bool tile_adds_to(const BwdArgs& a, int j, int kv_len, int iq) {
  int lo, hi;
  bwd_qblk_range<kMod, QB>(a, j, kv_len, lo, hi);
  return lo <= iq && iq < hi;
}

// The last kv tile that adds into query block iq: the window's bound, cut to
// the batch's kv tiles, then lowered to a tile whose query-block range really
// holds iq (the partial tile at the end of the keys, or a tile that starts past
// the last query but inside its block, can fall short of it).  Called for a
// block that some tile adds into, so the contiguous run of contributors stops
// the descent within a step or two.
template <bool kMod, int QB>
__device__ __forceinline__ int qblk_last_contributor(const BwdArgs& a, int iq, int kv_len) {
  const int wl = win_left<kMod>(a), wr = win_right<kMod>(a);
  const int n_kt = (kv_len + kTile - 1) / kTile;
  const int first = qblk_first_contributor<QB>(wl, iq);
  int last = wr >= 0 ? min(n_kt - 1, (iq * QB + QB - 1 + wr) / kTile) : n_kt - 1;
  while (last > first && !tile_adds_to<kMod, QB>(a, last, kv_len, iq)) --last;
  return last;
}

// The last kv tile <= last, and the first kv tile >= first, that belong to
// deterministic group g.
__device__ __forceinline__ int group_last(int last, int g, int groups) {
  return last - ((last - g) % groups + groups) % groups;
}
__device__ __forceinline__ int group_first(int first, int g, int groups) {
  return first + ((g - first % groups) % groups + groups) % groups;
}

__device__ __forceinline__ bool warp_wait_b(uint32_t bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

// AND of `ok` over the 128 threads of a warpgroup (named barrier `id`); every
// thread of the group must call it the same number of times.
__device__ __forceinline__ bool group_all(bool ok, int id) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.and.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok), "r"(id)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void group_sync(int id) {
  asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}

__device__ __forceinline__ void drain_wait_b(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitTimeoutNs) break;
  }
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// n consecutive 32-bit columns of this thread's lane (n = 8, 16, 32), waited.
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32, "tmem_ld width");
  if constexpr (N == 32) {
    tmem_ld32(taddr, r);
  } else {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
  }
}


// Writes n consecutive 32-bit columns of this thread's lane (no wait).
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const uint32_t (&w)[N]) {
  static_assert(N == 8 || N == 16, "tmem_st width");
  if constexpr (N == 16) {
    tmem_st16(taddr, w);
  } else {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
            taddr),
        "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
        : "memory");
  }
}


// Iterations (q head of the group x query block) of kv tile j.
struct BwdUnit {
  int bhk, j, b, hk, lo, n_blk, n_it;
  int kv_len;  // keys of batch b
};

// The r-th unit this CTA processes under static dealing (-1 when it has no
// more; with a.dyn the units come from a global counter instead, in the order
// bwd_unit decodes: groups of a.head_group kv heads, kv tile major).  Units are either
// head-major (u = bhk * n_ktiles + j, round robin, so CTAs running together
// share the queries of few heads in L2; non-causal and windowed calls) or,
// with causal masking, ordered by ascending kv tile (the longest units first)
// and dealt in a snake so that per-CTA work evens out.  The deterministic dQ chain has each
// tile wait only for tiles of the same head dealt before it (a CTA waiting on
// a tile dealt to it later would wait out its timeout): with the snake it runs
// in ascending tile order; head-major, the deterministic mode deals each
// head's tiles in descending order (bwd_unit) and chains them that way.
__device__ __forceinline__ int bwd_cta_unit(const BwdArgs& a, int r) {
  const int k = a.snake ? r * (int)gridDim.x + ((r & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x
                                                         : (int)blockIdx.x)
                        : (int)blockIdx.x + r * (int)gridDim.x;
  return k < a.n_units ? k : -1;
}

// The same dealing over clusters of two CTAs (the CTA-pair kernel): both CTAs
// of cluster c = blockIdx.x / 2 walk the same pair units.
__device__ __forceinline__ int bwd_cta_unit_pair(const BwdArgs& a, int r) {
  const int id = (int)(blockIdx.x >> 1), n = (int)(gridDim.x >> 1);
  const int k = a.snake ? r * n + ((r & 1) ? n - 1 - id : id) : id + r * n;
  return k < a.n_units ? k : -1;
}

template <bool kMod, int QB>
__device__ __forceinline__ BwdUnit bwd_unit(const BwdArgs& a, int u, int group) {
  BwdUnit w;
  if (a.dyn) {
    // groups of head_group kv heads in turn; in a group, kv tile major
    const int nbhk = a.B * a.Hkv, G = a.head_group, nk = a.n_ktiles;
    const int g = u / (G * nk), h0 = g * G;
    const int gg = min(G, nbhk - h0);
    const int r = u - g * G * nk;
    w.j = r / gg;
    w.bhk = h0 + (r - w.j * gg);
  } else if (a.snake) {
    const int nbhk = a.B * a.Hkv;
    w.j = u / nbhk;
    w.bhk = u - w.j * nbhk;
  } else {
    w.bhk = u / a.n_ktiles;
    w.j = u - w.bhk * a.n_ktiles;
  }
  w.b = w.bhk / a.Hkv;
  w.hk = w.bhk - w.b * a.Hkv;
  w.kv_len = bwd_kv_len<kMod>(a, w.b);
  if (a.desc) w.j = a.n_ktiles - 1 - w.j;  // each head's tiles highest first
  int hi;
  bwd_qblk_range<kMod, QB>(a, w.j, w.kv_len, w.lo, hi);
  w.n_blk = hi - w.lo;
  w.n_it = group * w.n_blk;
  return w;
}

// Pair unit u of a cluster of two CTAs: (batch, kv head, kv tiles 2p and 2p+1);
// the CTA of cluster rank `rank` takes tile 2p + rank (a tile past the last one
// holds no key).  Both CTAs walk the union of the two tiles' query-block
// ranges, so that they meet every block together for the dQ exchange; a block
// outside a tile's own range is fully masked for it and adds nothing.
template <bool kMod, int QB>
__device__ __forceinline__ BwdUnit bwd_unit_pair(const BwdArgs& a, int u, int group, int rank) {
  BwdUnit w;
  const int n_jp = (a.n_ktiles + 1) / 2;
  int jp;
  if (a.snake) {
    const int nbhk = a.B * a.Hkv;
    jp = u / nbhk;
    w.bhk = u - jp * nbhk;
  } else {
    w.bhk = u / n_jp;
    jp = u - w.bhk * n_jp;
  }
  w.b = w.bhk / a.Hkv;
  w.hk = w.bhk - w.b * a.Hkv;
  w.kv_len = bwd_kv_len<kMod>(a, w.b);
  w.j = 2 * jp + rank;
  int lo0, hi0, lo1 = 0, hi1 = 0;
  bwd_qblk_range<kMod, QB>(a, 2 * jp, w.kv_len, lo0, hi0);
  if (2 * jp + 1 < a.n_ktiles) bwd_qblk_range<kMod, QB>(a, 2 * jp + 1, w.kv_len, lo1, hi1);
  int lo, hi;
  if (hi0 <= lo0) {
    lo = lo1, hi = hi1;
  } else if (hi1 <= lo1) {
    lo = lo0, hi = hi0;
  } else {
    lo = min(lo0, lo1), hi = max(hi0, hi1);
  }
  w.lo = lo;
  w.n_blk = hi > lo ? hi - lo : 0;
  w.n_it = group * w.n_blk;
  return w;
}

// ------------------------------------------------------------------ clusters

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of both CTAs of the cluster; release / acquire at cluster scope.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of this CTA's shared address `addr` in CTA `rank`.
__device__ __forceinline__ uint32_t map_peer(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrives once on the mbarrier at shared::cluster address `remote_bar`, with
// relaxed ordering: the arrival publishes no data of this thread (a release
// would first wait for every earlier global write of the thread, measured at
// about 1,000 cycles behind the drain's reduction adds).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar)
               : "memory");
}

// Non-blocking test (test_wait, not try_wait: a try_wait may sleep for a
// system-dependent time, which measured about 1,000 cycles before it saw an
// arrival made by the other CTA of the pair).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on a local mbarrier that another CTA of the cluster completes
// (acquire at cluster scope); gives up like mbar_wait.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int* abort) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitTimeoutNs) {
        *abort = 1;
        return false;
      }
    }
  }
}

// ------------------------------------------------------------------ CTA pairs (tcgen05 cta_group::2)
//
// Two CTAs of a cluster share the tensor cores of their two SMs: one thread of
// rank 0 issues every MMA, which runs its first M/2 rows on rank 0's SM and
// the rest on rank 1's; each SM reads the A rows and the B columns of its half
// from its own shared memory (or TMEM), at the same addresses in both CTAs,
// and writes its own TMEM.  Every tcgen05 allocation, MMA and commit of such a
// kernel names the pair.

// One warp of each CTA of the pair allocates (the same count in both).
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Pair SS MMA from split descriptors; `acc` selects accumulate (1) or overwrite (0).
__device__ __forceinline__ void umma_pair_ss(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi,
                                             uint32_t b_lo, uint32_t b_hi, uint32_t idesc,
                                             uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "mov.b64 da, {%1, %2};\n\t"
      "mov.b64 db, {%3, %4};\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(acc)
      : "memory");
}

// Pair TS MMA: A from each CTA's TMEM at `a_tmem`.
__device__ __forceinline__ void umma_pair_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                             uint32_t b_hi, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(acc)
      : "memory");
}

// Arrives once on the mbarrier at the same offset in both CTAs when every pair
// MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_pair_commit_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}
// ... on this CTA's mbarrier only.
__device__ __forceinline__ void umma_pair_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 3-D tile load into this CTA's shared memory whose bytes are counted on an
// mbarrier of either CTA of the pair (`bar`: a shared::cluster address).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Copies `bytes` (a multiple of 16) of this CTA's shared memory to shared::cluster
// address `dst` (the partner's) through the async proxy; completion counts the
// bytes on the mbarrier at `bar`, in the destination CTA.  The source must have
// been made visible to the async proxy (fence_proxy_async_smem by its writers).
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst, uint32_t src, uint32_t bytes,
                                                  uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "r"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// High word of a shared-memory descriptor with the 64-byte swizzle (layout 4):
// an MN-major operand whose 64-byte rows hold 32 consecutive MN elements of one
// K index, 8 K rows (512 bytes) per swizzle atom; SBO = the next 8 K rows.
__host__ __device__ constexpr uint32_t sdesc_hi_sw64(uint32_t sbo_bytes) {
  return ((sbo_bytes >> 4) & 0x3FFFu) | (1u << 14) | (4u << 29);
}

}  // namespace fa

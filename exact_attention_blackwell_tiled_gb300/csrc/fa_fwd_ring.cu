// fa_fwd_ring.cu -- the head-dimension-64 forward for no mask or the causal one
// (positive scale, no split).
//
// Units and the TMA / tensor-core machinery are those of fwd_kernel: a unit is
// a pair of 128-row query tiles of one (batch, head), one persistent CTA per SM
// walks a list of units, warps 0-7 run the softmax of the two tiles (thread r of
// a group owns query row r) and warp 8 issues the TMA loads.  What differs is
// how a query tile walks its keys, and that each query tile has two MMA-issuing
// threads of its own, one for GEMM 1 (warps 9, 10) and one for GEMM 2 (11, 12).
//
// Each 128-key K/V tile is consumed as two 64-key halves, and every query tile
// owns a ring of three 64-column score buffers in tensor memory:
//   GEMM 1 (k):  S_t[k mod 3] = Q_t K_half(k)^T        (SS, N = 64)
//   GEMM 2 (k):  O_t += P_t[k mod 3] V_half(k)         (TS, P read from TMEM)
// GEMM 1 of a half is issued as soon as GEMM 2 of the half three back is done
// with its buffer, so while the softmax warps work on half k the scores of
// halves k+1 and k+2 are already in TMEM or being computed.  GEMM 1 works per K
// tile: when the tile's two halves land in adjacent buffers (two tiles in
// three) one N = 128 group computes both at the full MMA rate (64 cycles per
// instruction); two N = 64 groups hold the tensor pipe about 2.8 times as long
// (about 89 cycles per N = 64 instruction measured in this kernel's mix).  The
// softmax then runs back to back instead of waiting
// for a GEMM 2 -> GEMM 1 round trip after every block (FlashAttention-4 pages:
// the per-tile phases GEMM 1 -> softmax -> GEMM 2 and the pipeline that overlaps
// the softmax of one block with GEMM 2 of the previous and GEMM 1 of the next).
// Only D = 64 leaves the tensor-memory columns for the ring: per query tile
// 3 x 64 score columns + 64 O columns, 512 for the pair.
//
// Since GEMM 2 no longer completes before the next scores are seen, every
// GEMM 2 signals a barrier of its score buffer.  The softmax waits on it only
// when it has to rescale O at half k (conditional rescale, threshold 8 in the
// log2 domain: GEMM 2 of half k-1 must be done first), and before the epilogue
// reads O.  A buffer's barrier is never more than one phase away from such a
// wait: seeing S(k) implies that GEMM 2 of half k-3 is done (GEMM 1 of half k
// waited for it), and GEMM 2 of half k+2 needs a P that is not written yet.
//
// Four issuing threads: a thread with MMAs queued stalls on its next barrier
// wait until the tensor core has taken them, so one thread serving both tiles
// spends most of its time in such stalls and starves the tensor pipe (measured
// on GB300: about 420 cycles per group of four N = 64 MMAs).  With a thread per
// tile and GEMM each stalls only on its own four MMAs while the others' keep
// the pipe busy.  The Q and K stages are then freed by both GEMM 1 threads and
// the V stages by both GEMM 2 threads: each commits its share after its last
// MMA reading the stage, or, for a K/V tile its query tile does not reach,
// arrives once that tile has landed (so the arrival cannot count toward the
// stage's previous use).
//
// TMEM columns of query tile t: score buffers [256t + 64b, +64) for b = 0..2, P
// (bf16 pairs) over the first 32 columns of its buffer, O [256t + 192, +64).
#include <cuda_bf16.h>

#include "exp2.cuh"
#include "fa_internal.h"
#include "fwd_common.cuh"
#include "ptx.cuh"

namespace fa {

namespace {

struct RingLayout {
  static constexpr int D = 64;
  static constexpr int kTileBytes = kTile * D * 2;   // a Q, K or V tile: 128 rows of 128 bytes
  static constexpr int kHalfBytes = kTileBytes / 2;  // 64 rows
  static constexpr int kRing = 3;                    // score buffers per query tile
  static constexpr int kQStages = 2;                 // each holds both Q tiles of a unit
  static constexpr int kKStages = 3;
  static constexpr int kVStages = 3;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQStages * 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kVStages * kTileBytes;
  static constexpr int kBarQFull = 0;
  static constexpr int kBarQEmpty = kBarQFull + kQStages;
  static constexpr int kBarKFull = kBarQEmpty + kQStages;
  static constexpr int kBarKEmpty = kBarKFull + kKStages;
  static constexpr int kBarVFull = kBarKEmpty + kKStages;
  static constexpr int kBarVEmpty = kBarVFull + kVStages;
  static constexpr int kBarSFull = kBarVEmpty + kVStages;  // [tile][buffer]
  static constexpr int kBarPFull = kBarSFull + 2 * kRing;  // [tile][buffer]
  static constexpr int kBarODone = kBarPFull + 2 * kRing;  // [tile][buffer]: its GEMM 2 done
  static constexpr int kBarOFree = kBarODone + 2 * kRing;  // per tile: epilogue done with O
  static constexpr int kBarDrain = kBarOFree + 2;          // per issuing thread
  static constexpr int kNumBars = kBarDrain + 4;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // TMEM base slot, abort flag
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAllocBytes = kBytes + 1024;  // slack for 1024-byte alignment
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColsPerTile = 256;
  static constexpr uint32_t kColO = 192;  // within a tile's columns
  // exponential split as in fwd_kernel at D = 64: one column pair in eight
  // through the cubic on the FMA pipe
  static constexpr int kPolyPairs = 1;
};
static_assert(RingLayout::kAllocBytes <= 227 * 1024, "shared memory");
static_assert(2 * RingLayout::kColsPerTile == RingLayout::kTmemCols, "tensor memory");
static_assert(RingLayout::kRing * 64 + RingLayout::D <= (int)RingLayout::kColsPerTile,
              "a tile's columns");

constexpr int kRingThreads = 416;  // 8 softmax warps, the producer, four issuers

__global__ void __launch_bounds__(kRingThreads, 1)
    fwd_ring64_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  using L = RingLayout;
  constexpr int D = L::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return sbase + L::kOffBar + 8 * i; };

  if (threadIdx.x == 0) {
    // the stages are freed by both issuing threads
    for (int s = 0; s < L::kQStages; ++s) {
      mbar_init(bar(L::kBarQFull + s), 1);
      mbar_init(bar(L::kBarQEmpty + s), 2);
    }
    for (int s = 0; s < L::kKStages; ++s) {
      mbar_init(bar(L::kBarKFull + s), 1);
      mbar_init(bar(L::kBarKEmpty + s), 2);
    }
    for (int s = 0; s < L::kVStages; ++s) {
      mbar_init(bar(L::kBarVFull + s), 1);
      mbar_init(bar(L::kBarVEmpty + s), 2);
    }
    for (int i = 0; i < 2 * L::kRing; ++i) {
      mbar_init(bar(L::kBarSFull + i), 1);
      mbar_init(bar(L::kBarPFull + i), 128);
      mbar_init(bar(L::kBarODone + i), 1);
    }
    for (int t = 0; t < 2; ++t) mbar_init(bar(L::kBarOFree + t), 128);
    for (int i = 0; i < 4; ++i) mbar_init(bar(L::kBarDrain + i), 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the prologue above overlaps the previous kernel in the stream; q, k, v
  // (which it may have written) are read from here on
  grid_dep_wait();
  grid_dep_launch();
  const uint32_t tmem = *tmem_slot;
  const int group = a.Hq / a.Hkv;
  const int wr = a.causal ? 0 : -1;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    // Per unit: both Q tiles, then K_0, K_1, V_0, K_2, V_1, K_3, ... -- the order
    // in which the MMAs first use them (GEMM 1 runs three halves, i.e. one and a
    // half K tiles, ahead of GEMM 2).
    if (lane == 0) {
      uint32_t k_it = 0, v_it = 0, q_it = 0;
      bool ok = true;
      auto load = [&](bool is_v, int bhk, int j) -> bool {
        uint32_t& it = is_v ? v_it : k_it;
        const int n = is_v ? L::kVStages : L::kKStages;
        const uint32_t st = it % n;
        const uint32_t full = bar((is_v ? L::kBarVFull : L::kBarKFull) + st);
        const uint32_t empty = bar((is_v ? L::kBarVEmpty : L::kBarKEmpty) + st);
        if (!mbar_wait(empty, ((it / n) & 1) ^ 1, abort_flag)) return false;
        mbar_arrive_expect_tx(full, L::kTileBytes);
        tma_load_3d(sbase + (is_v ? L::kOffV : L::kOffK) + st * L::kTileBytes,
                    is_v ? &tm_v : &tm_k, full, 0, j * kTile, bhk);
        ++it;
        return true;
      };
      for (int ri = 0, u = cta_unit(a, 0); ok && u >= 0; u = cta_unit(a, ++ri)) {
        int bh, pair, split;
        unit_coords(a, u, bh, pair, split);
        const int b = bh / a.Hq, h = bh - b * a.Hq;
        const int bhk = b * a.Hkv + h / group;
        int lo[2], hi[2], jlo, nmax;
        pair_kv_span<false>(a, -1, wr, a.Sk, pair, 0, lo, hi, jlo, nmax);
        if (nmax == 0) continue;
        const uint32_t qs = q_it % L::kQStages;
        if (!mbar_wait(bar(L::kBarQEmpty + qs), ((q_it / L::kQStages) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(L::kBarQFull + qs), 2 * L::kTileBytes);
        const uint32_t qdst = sbase + L::kOffQ + qs * 2 * L::kTileBytes;
#pragma unroll
        for (int t = 0; t < 2; ++t)
          tma_load_3d(qdst + t * L::kTileBytes, &tm_q, bar(L::kBarQFull + qs), 0,
                      (2 * pair + t) * kTile, bh);
        ++q_it;
        ok = load(false, bhk, jlo) && (nmax < 2 || load(false, bhk, jlo + 1));
        for (int i = 0; ok && i < nmax; ++i)
          ok = load(true, bhk, jlo + i) && (i + 2 >= nmax || load(false, bhk, jlo + i + 2));
      }
      // Let every issued copy land before the CTA can exit.
      for (uint32_t n = (k_it > (uint32_t)L::kKStages ? k_it - L::kKStages : 0); n < k_it; ++n)
        drain_wait(bar(L::kBarKFull + n % L::kKStages), (n / L::kKStages) & 1);
      for (uint32_t n = (v_it > (uint32_t)L::kVStages ? v_it - L::kVStages : 0); n < v_it; ++n)
        drain_wait(bar(L::kBarVFull + n % L::kVStages), (n / L::kVStages) & 1);
      for (uint32_t n = (q_it > (uint32_t)L::kQStages ? q_it - L::kQStages : 0); n < q_it; ++n)
        drain_wait(bar(L::kBarQFull + n % L::kQStages), (n / L::kQStages) & 1);
    }
  } else if (warp >= 9 && warp <= 10) {
    // ------------------------------------------------------------ GEMM 1 issuers
    // warp 9 for query tile 0, warp 10 for tile 1
    if (lane == 0) {
      const int t = warp - 9;
      constexpr uint32_t kIdescS = idesc_bf16_f32(kTile, 64, false, false);
      constexpr uint32_t kIdescS2 = idesc_bf16_f32(kTile, 128, false, false);
      constexpr uint32_t kHi = sdesc_hi(1024);  // SBO 1024 B, version 1, 128B swizzle
      const uint32_t s_cols = tmem + t * L::kColsPerTile;
      uint32_t k_it = 0, q_it = 0;
      uint32_t gs = 0;  // score halves issued for this tile (all units)
      bool ok = true;
      for (int ri = 0, u = cta_unit(a, 0); ok && u >= 0; u = cta_unit(a, ++ri)) {
        int bh, pair, split;
        unit_coords(a, u, bh, pair, split);
        int lo[2], hi[2], jlo, nmax;
        pair_kv_span<false>(a, -1, wr, a.Sk, pair, 0, lo, hi, jlo, nmax);
        if (nmax == 0) continue;
        // both tiles start at kv tile jlo (no left window); this one reaches m
        // of the unit's nmax kv tiles
        const int m = hi[t] - lo[t], n = 2 * m;
        const uint32_t qs = q_it % L::kQStages;
        if (!mbar_wait(bar(L::kBarQFull + qs), (q_it / L::kQStages) & 1, abort_flag)) {
          ok = false;
          break;
        }
        if (n == 0) mbar_arrive(bar(L::kBarQEmpty + qs));
        const uint32_t q_lo = sdesc_lo(sbase + L::kOffQ + (2 * qs + t) * L::kTileBytes, 16);
        const uint32_t kbase = k_it;  // ring position of K_jlo
        // buffer of the score half with global index g is free once GEMM 2 of
        // half g - 3 is done; that barrier is within one phase: this thread
        // waited for the buffer's use before that one before GEMM 1 of g - 3
        auto buf_free = [&](uint32_t g) -> bool {
          return g < (uint32_t)L::kRing ||
                 mbar_wait(bar(L::kBarODone + t * L::kRing + g % L::kRing),
                           (g / L::kRing - 1) & 1, abort_flag);
        };
        for (int i = 0; ok && i < m; ++i) {
          const uint32_t pos = kbase + i, st = pos % L::kKStages;
          const uint32_t b0 = gs % L::kRing;
          // both halves of K tile i; when their buffers are adjacent (b0 < 2)
          // one N = 128 group computes both, at the full MMA rate
          ok = mbar_wait(bar(L::kBarKFull + st), (pos / L::kKStages) & 1, abort_flag) &&
               buf_free(gs) && buf_free(gs + 1);
          if (!ok) break;
          tc_fence_after();
          const uint32_t k_tile = sbase + L::kOffK + st * L::kTileBytes;
          if (b0 + 1 < (uint32_t)L::kRing) {
            const uint32_t d = s_cols + 64 * b0;
            const uint32_t k_lo = sdesc_lo(k_tile, 16);
            umma_ss_w<0>(d, q_lo, kHi, k_lo, kHi, kIdescS2);
#pragma unroll
            for (int kk = 1; kk < D / 16; ++kk)
              umma_ss_w<1>(d, q_lo + kk * 2, kHi, k_lo + kk * 2, kHi, kIdescS2);
            umma_commit(bar(L::kBarSFull + t * L::kRing + b0));
            umma_commit(bar(L::kBarSFull + t * L::kRing + b0 + 1));
          } else {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const uint32_t b = (b0 + hf) % L::kRing;
              const uint32_t d = s_cols + 64 * b;
              const uint32_t k_lo = sdesc_lo(k_tile + hf * L::kHalfBytes, 16);
              umma_ss_w<0>(d, q_lo, kHi, k_lo, kHi, kIdescS);
#pragma unroll
              for (int kk = 1; kk < D / 16; ++kk)
                umma_ss_w<1>(d, q_lo + kk * 2, kHi, k_lo + kk * 2, kHi, kIdescS);
              umma_commit(bar(L::kBarSFull + t * L::kRing + b));
            }
          }
          gs += 2;
          umma_commit(bar(L::kBarKEmpty + st));
          if (i == m - 1) umma_commit(bar(L::kBarQEmpty + qs));
        }
        // this tile's share of the K tiles only the other tile reaches, each
        // once it has landed
        for (int i = m; ok && i < nmax; ++i) {
          const uint32_t kp = kbase + i;
          ok = mbar_wait(bar(L::kBarKFull + kp % L::kKStages), (kp / L::kKStages) & 1, abort_flag);
          if (ok) mbar_arrive(bar(L::kBarKEmpty + kp % L::kKStages));
        }
        if (!ok) break;
        k_it = kbase + nmax;
        ++q_it;
      }
      // Every issued MMA must complete before TMEM is released.
      umma_commit(bar(L::kBarDrain + t));
      drain_wait(bar(L::kBarDrain + t), 0);
    }
  } else if (warp >= 11) {
    // ------------------------------------------------------------ GEMM 2 issuers
    // warp 11 for query tile 0, warp 12 for tile 1
    if (lane == 0) {
      const int t = warp - 11;
      constexpr uint32_t kIdescO = idesc_bf16_f32(kTile, D, false, true);
      constexpr uint32_t kHi = sdesc_hi(1024);
      const uint32_t s_cols = tmem + t * L::kColsPerTile;
      const uint32_t o_col = s_cols + L::kColO;
      uint32_t v_it = 0;
      uint32_t go = 0;     // P halves consumed for this tile (all units)
      uint32_t units = 0;  // units in which this tile had keys (O-free phases)
      bool ok = true;
      for (int ri = 0, u = cta_unit(a, 0); ok && u >= 0; u = cta_unit(a, ++ri)) {
        int bh, pair, split;
        unit_coords(a, u, bh, pair, split);
        int lo[2], hi[2], jlo, nmax;
        pair_kv_span<false>(a, -1, wr, a.Sk, pair, 0, lo, hi, jlo, nmax);
        if (nmax == 0) continue;
        const int m = hi[t] - lo[t], n = 2 * m;
        const uint32_t vbase = v_it;  // ring position of V_jlo
        for (int k = 0; ok && k < n; ++k) {
          const int i = k >> 1, hf = k & 1;
          const uint32_t pos = vbase + i, st = pos % L::kVStages;
          const uint32_t b = go % L::kRing;
          ok = mbar_wait(bar(L::kBarPFull + t * L::kRing + b), (go / L::kRing) & 1, abort_flag) &&
               (k > 0 || units == 0 ||
                mbar_wait(bar(L::kBarOFree + t), (units - 1) & 1, abort_flag)) &&
               (hf == 1 || mbar_wait(bar(L::kBarVFull + st), (pos / L::kVStages) & 1, abort_flag));
          if (!ok) break;
          tc_fence_after();
          const uint32_t v_lo = sdesc_lo(sbase + L::kOffV + st * L::kTileBytes, kTile * 128);
          const uint32_t p_col = s_cols + 64 * b;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // 16 keys of the half per MMA
            umma_ts_w(o_col, p_col + kk * 8, v_lo + (((4 * hf + kk) * 16 * 128) >> 4), kHi, kIdescO,
                      (k > 0 || kk > 0) ? 1u : 0u);
          umma_commit(bar(L::kBarODone + t * L::kRing + b));
          ++go;
          if (hf == 1) umma_commit(bar(L::kBarVEmpty + st));
        }
        // this tile's share of the V tiles only the other tile reaches
        for (int i = m; ok && i < nmax; ++i) {
          const uint32_t vp = vbase + i;
          ok = mbar_wait(bar(L::kBarVFull + vp % L::kVStages), (vp / L::kVStages) & 1, abort_flag);
          if (ok) mbar_arrive(bar(L::kBarVEmpty + vp % L::kVStages));
        }
        if (!ok) break;
        v_it = vbase + nmax;
        if (n > 0) ++units;
      }
      umma_commit(bar(L::kBarDrain + 2 + t));
      drain_wait(bar(L::kBarDrain + 2 + t), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int t = warp >> 2;          // query tile of the pair this group serves
    const int r = threadIdx.x & 127;  // query row inside the tile == TMEM lane
    const uint32_t t_row = tmem + ((uint32_t)((warp & 3) * 32) << 16) + t * L::kColsPerTile;
    uint32_t x = 0;  // score halves consumed (all units)
    bool ok = true;
    const float c = a.scale_log2;  // > 0 for this kernel
    const float2 c2 = make_float2(c, c);
    for (int ri = 0, u = cta_unit(a, 0); ok && u >= 0; u = cta_unit(a, ++ri)) {
      int bh, pair, split;
      unit_coords(a, u, bh, pair, split);
      const int qt = 2 * pair + t;
      int jlo, jhi;
      split_kv_range<false>(a, -1, wr, a.Sk, qt, 0, jlo, jhi);
      if (jhi == jlo) continue;  // a tile past the last query row
      const int q_row = qt * kTile + r;
      const int lim = wr >= 0 ? min(a.Sk, q_row + 1) : a.Sk;  // keys [0, lim) visible
      const int n = 2 * (jhi - jlo);
      float m_run = -INFINITY, l_run = 0.f;
      for (int k = 0; k < n; ++k) {
        const uint32_t b = x % L::kRing;
        if (!warp_wait(bar(L::kBarSFull + t * L::kRing + b), (x / L::kRing) & 1, abort_flag)) {
          ok = false;
          break;
        }
        ++x;
        tc_fence_after();
        const int kv0 = jlo * kTile + 64 * k;  // first key of the half
        uint32_t v[64];
        tmem_ld64(t_row + 64 * b, v);
        if (kv0 + 64 > lim) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (kv0 + i >= lim) v[i] = __float_as_uint(-INFINITY);
        }
        // four independent max chains (shorter dependency chains)
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < 64; i += 8)
#pragma unroll
          for (int j = 0; j < 4; ++j) mq[j] = fmax3(mq[j], u2f(v[i + 2 * j]), u2f(v[i + 2 * j + 1]));
        float mraw = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        if (mraw != -INFINITY) mraw *= c;
        // Conditional rescale: keep a stale running max unless the new max
        // exceeds it by more than 8 (P then stays <= 2^8).
        float alpha = 1.f;
        bool rescale = false;
        if (k == 0) {
          m_run = mraw;
        } else if (mraw > m_run + 8.0f) {
          alpha = ex2_mufu(m_run - mraw);
          m_run = mraw;
          rescale = true;
        }
        const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
        const float2 nm2 = make_float2(neg_m, neg_m);
        float2 sum2 = make_float2(0.f, 0.f), sum2b = make_float2(0.f, 0.f);
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float2 tt = __ffma2_rn(make_float2(u2f(v[2 * i]), u2f(v[2 * i + 1])), c2, nm2);
          float p0, p1;
          if ((i & 7) < L::kPolyPairs) {
            const float2 pp = ex2_poly2(tt);
            p0 = pp.x, p1 = pp.y;
          } else {
            p0 = ex2_mufu(tt.x), p1 = ex2_mufu(tt.y);
          }
          if (i & 1)
            sum2b = __fadd2_rn(sum2b, make_float2(p0, p1));
          else
            sum2 = __fadd2_rn(sum2, make_float2(p0, p1));
          pk[i] = pack_bf16x2(p0, p1);
        }
        __syncwarp();
        tmem_st32(t_row + 64 * b, pk);
        l_run = l_run * alpha + ((sum2.x + sum2b.x) + (sum2.y + sum2b.y));
        if (__any_sync(0xffffffffu, rescale)) {
          // GEMM 2 of the previous half (global half x-2) must be done before O
          // is rescaled; GEMM 2 of this half waits for this thread's P
          const uint32_t xp = x - 2;
          if (!warp_wait(bar(L::kBarODone + t * L::kRing + xp % L::kRing), (xp / L::kRing) & 1,
                         abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(t_row + L::kColO + cc * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(u2f(o[i]) * alpha);
            tmem_st32(t_row + L::kColO + cc * 32, o);
          }
        }
        tc_fence_before();
        mbar_arrive(bar(L::kBarPFull + t * L::kRing + b));
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16, LSE = ln2 * (m + log2 l).  The unit's
      // last GEMM 2 (global half x-1) is the tile's last.
      const uint32_t xl = x - 1;
      if (!warp_wait(bar(L::kBarODone + t * L::kRing + xl % L::kRing), (xl / L::kRing) & 1,
                     abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool row_ok = q_row < a.Sq;
      const float inv_l = 1.0f / l_run;
      __nv_bfloat16* orow =
          reinterpret_cast<__nv_bfloat16*>(a.o) + ((size_t)bh * a.Sq + (row_ok ? q_row : 0)) * D;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        __syncwarp();  // reconverge after the per-row store before the warp-wide load
        tmem_ld32(t_row + L::kColO + cc * 32, o);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(u2f(o[2 * i]) * inv_l, u2f(o[2 * i + 1]) * inv_l);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (row_ok)
        a.lse[(size_t)bh * a.Sq + q_row] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
      tc_fence_before();
      mbar_arrive(bar(L::kBarOFree + t));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(a.status, (int)FA_ERR_TIMEOUT);
}

}  // namespace

bool fwd_ring64_eligible(const FwdArgs& a, int D, int mode) {
  return D == 64 && mode == 0 && a.n_split <= 1 && a.scale_log2 > 0.f;
}

int launch_fwd_ring64(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const FwdArgs& a, int grid, cudaStream_t stream) {
  using L = RingLayout;
  int dev;
  DeviceInfo info;
  if (!current_device(&dev, &info)) return FA_ERR_CUDA;
  static bool attr_done[64] = {};
  if (dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(fwd_ring64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::kAllocBytes) != cudaSuccess)
      return FA_ERR_CUDA;
    attr_done[dev] = true;
  }
  if (launch_pdl(fwd_ring64_kernel, dim3(grid), dim3(kRingThreads), L::kAllocBytes, stream, tq,
                 tk, tv, a) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // namespace fa

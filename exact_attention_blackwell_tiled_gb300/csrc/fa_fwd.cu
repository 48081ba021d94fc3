// fa_fwd.cu -- forward attention kernel for sm_103a.
//
// One persistent CTA per SM walks a list of work units.  A unit is a PAIR of
// 128-row query tiles of one (batch, head) -- 256 query rows -- that stream the
// same 128-row K/V tiles of the matching kv head (FlashAttention-4 pages: the
// three per-tile phases GEMM 1 -> softmax -> GEMM 2; the pipeline
// "Softmax(S_k) || GEMM 2(P_k V_k) || GEMM 1(Q K_{k+1}^T)"; 128x128 tiles with
// accumulators in tensor memory; conditional rescale with threshold
// log2(256) = 8.0).
//
// Warp roles (320 threads):
//   warps 0-3  softmax of query tile 0 of the pair, warps 4-7 of tile 1: thread r
//              of the group owns query row r (= TMEM lane r).  It reads S from
//              TMEM, masks, updates the running max / sum, writes P (bf16) back
//              over the S columns, rescales its O row in TMEM when the running
//              max moved by more than 8 (log2 units), and writes O and the LSE
//              at the end of the unit.
//   warp 8     TMA producer: both Q tiles of a unit into a 2-stage ring, then
//              K_0, V_0, K_1, V_1, ... into a shared ring, the order the MMA
//              issuer first uses them.
//   warp 9     TMEM allocator and single-thread tcgen05.mma issuer.  Per kv tile
//              j it issues, for tile 0 then tile 1:
//                O_t += P_t(j-1) V_{j-1}   (TS MMA, P read from TMEM)
//                S_t  = Q_t K_j^T          (SS MMA)
//              so while the softmax warps of one tile work, the tensor core
//              runs the other tile's two GEMMs ("ping-pong").
//
// TMEM columns: S/P of tile 0 [0,128), of tile 1 [128,256); O of tile 0
// [256, 256+D), of tile 1 [256+D, 256+2D).
// Scores are handled in base 2: t = s * scale * log2(e), P = 2^(t - m).
#include <cuda_bf16.h>

#include "exp2.cuh"
#include "fa_internal.h"
#include "fwd_common.cuh"
#include "ptx.cuh"

namespace fa {

__device__ int g_fwd_status = 0;

template <int D>
struct FwdLayout {
  static constexpr int kColBlocks = D / 64;         // 64-element (128-byte) column blocks
  static constexpr int kBlockBytes = kTile * 128;   // one 128-row x 64-col block
  static constexpr int kTileBytes = kTile * D * 2;  // a Q, K or V tile
  // Each Q stage holds both Q tiles.  At D = 128 one Q stage buys more K/V
  // stages: the K/V ring must hold V_{j-1} and K_j in use plus enough tiles in
  // flight to hide the TMA latency, while a single Q stage only delays the next
  // unit's first GEMM 1 by the part of one Q load its trailing GEMM 2s don't
  // cover.  Four K/V stages measured as fast as five (1 to 3% faster on the
  // causal shapes), two plus two Q stages 10-15% slower.
  static constexpr int kQStages = (D == 128) ? 1 : 2;
  static constexpr int kKVStages = (D == 128) ? 4 : 6;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kQStages * 2 * kTileBytes;
  static constexpr int kOffBar = kOffKV + kKVStages * kTileBytes;
  static constexpr int kBarQFull = 0;
  static constexpr int kBarQEmpty = kBarQFull + kQStages;
  static constexpr int kBarKVFull = kBarQEmpty + kQStages;
  static constexpr int kBarKVEmpty = kBarKVFull + kKVStages;
  static constexpr int kBarSFull = kBarKVEmpty + kKVStages;  // per tile
  static constexpr int kBarPFull = kBarSFull + 2;            // per tile
  static constexpr int kBarOFinal = kBarPFull + 2;           // per tile: last GEMM 2 done
  static constexpr int kBarOFree = kBarOFinal + 2;           // per tile: epilogue done with O
  static constexpr int kBarDrain = kBarOFree + 2;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // TMEM base slot, abort flag
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAllocBytes = kBytes + 1024;  // slack for 1024-byte alignment
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;
  // Exponential split (FlashAttention-4 pages, key contribution #2): of every 8
  // column pairs of a score row, kPolyPairs go through the cubic on the FMA
  // pipe (two lanes per packed instruction) and the rest through MUFU ex2.
  // Chosen by measurement on GB300, whose MUFU rate is twice B200's.
  static constexpr int kPolyPairs = (D == 64) ? 1 : 0;
};

// kMod: 0 plain (no mask or the causal one), 1 a sliding window, 2 a window
// and the relative-position bias (a.alibi) added to every score.  kSplit: a
// unit covers one split of the kv tiles and writes fp32 parts for the merge.
template <int D, int kMod, bool kSplit>
__global__ void __launch_bounds__(320, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  using L = FwdLayout<D>;
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
    for (int s = 0; s < L::kQStages; ++s) {
      mbar_init(bar(L::kBarQFull + s), 1);
      mbar_init(bar(L::kBarQEmpty + s), 1);
    }
    for (int s = 0; s < L::kKVStages; ++s) {
      mbar_init(bar(L::kBarKVFull + s), 1);
      mbar_init(bar(L::kBarKVEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(L::kBarSFull + t), 1);
      mbar_init(bar(L::kBarPFull + t), 128);
      mbar_init(bar(L::kBarOFinal + t), 1);
      mbar_init(bar(L::kBarOFree + t), 128);
    }
    mbar_init(bar(L::kBarDrain), 1);
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
  constexpr bool kWin = kMod >= 1, kBias = kMod == 2;
  // the window; plain calls carry only the causal flag
  const int wl = kWin ? a.wl : -1;
  const int wr = kWin ? a.wr : (a.causal ? 0 : -1);
  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t kv_it = 0, q_it = 0;
      bool ok = true;
      auto load_kv = [&](const CUtensorMap* tm, int bhk, int j) -> bool {
        const uint32_t st = kv_it % L::kKVStages;
        if (!mbar_wait(bar(L::kBarKVEmpty + st), ((kv_it / L::kKVStages) & 1) ^ 1, abort_flag))
          return false;
        mbar_arrive_expect_tx(bar(L::kBarKVFull + st), L::kTileBytes);
        const uint32_t dst = sbase + L::kOffKV + st * L::kTileBytes;
#pragma unroll
        for (int cb = 0; cb < L::kColBlocks; ++cb)
          tma_load_3d(dst + cb * L::kBlockBytes, tm, bar(L::kBarKVFull + st), cb * 64, j * kTile,
                      bhk);
        ++kv_it;
        return true;
      };
      for (int ri = 0, u = cta_unit(a, 0); ok && u >= 0; u = cta_unit(a, ++ri)) {
        int bh, pair, split;
        unit_coords(a, u, bh, pair, split);
        const int b = bh / a.Hq, h = bh - b * a.Hq;
        const int bhk = b * a.Hkv + h / group;
        int lo[2], hi[2], jlo, nmax;
        pair_kv_span<kSplit>(a, wl, wr, batch_kv_len<kWin>(a, b), pair, split, lo, hi, jlo, nmax);
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
#pragma unroll
          for (int cb = 0; cb < L::kColBlocks; ++cb)
            tma_load_3d(qdst + t * L::kTileBytes + cb * L::kBlockBytes, &tm_q,
                        bar(L::kBarQFull + qs), cb * 64, (2 * pair + t) * kTile, bh);
        ++q_it;
        for (int j = jlo; j < jlo + nmax; ++j) {
          if (!load_kv(&tm_k, bhk, j) || !load_kv(&tm_v, bhk, j)) { ok = false; break; }
        }
      }
      // Let every issued copy land before the CTA can exit.
      for (uint32_t n = (kv_it > (uint32_t)L::kKVStages ? kv_it - L::kKVStages : 0); n < kv_it; ++n)
        drain_wait(bar(L::kBarKVFull + n % L::kKVStages), (n / L::kKVStages) & 1);
      for (uint32_t n = (q_it > (uint32_t)L::kQStages ? q_it - L::kQStages : 0); n < q_it; ++n)
        drain_wait(bar(L::kBarQFull + n % L::kQStages), (n / L::kQStages) & 1);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kTile, kTile, false, false);
      constexpr uint32_t kIdescO = idesc_bf16_f32(kTile, D, false, true);
      constexpr uint32_t kHi = sdesc_hi(1024);  // SBO 1024 B, version 1, 128B swizzle
      uint32_t kv_it = 0, q_it = 0;
      uint32_t p_seen[2] = {0u, 0u};  // P-ready phases consumed, per tile
      uint32_t units_t[2] = {0u, 0u};  // units with work, per tile (O-free phases)
      bool ok = true;
      for (int ri = 0, u = cta_unit(a, 0); ok && u >= 0; u = cta_unit(a, ++ri)) {
        int bh, pair, split;
        unit_coords(a, u, bh, pair, split);
        // kv tile j sits at position p = j - jlo of the pair's range; tile t
        // computes S for positions [plo[t], phi[t]) and O one position behind
        int plo[2], phi[2], jlo, nmax;
        pair_kv_span<kSplit>(a, wl, wr, batch_kv_len<kWin>(a, bh / a.Hq), pair, split, plo, phi,
                             jlo, nmax);
        if (nmax == 0) continue;
        for (int t = 0; t < 2; ++t) {
          plo[t] -= jlo;
          phi[t] -= jlo;
        }
        const uint32_t qs = q_it % L::kQStages;
        if (!mbar_wait(bar(L::kBarQFull + qs), (q_it / L::kQStages) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t q_base = sbase + L::kOffQ + qs * 2 * L::kTileBytes;
        const uint32_t base_it = kv_it;  // ring position of K_0; V_j sits right after K_j
        for (int j = 0; ok && j <= nmax; ++j) {
          const bool need_v = j >= 1;
          const bool need_k = j < nmax;
          const uint32_t v_pos = base_it + 2 * (j - 1) + 1, k_pos = base_it + 2 * j;
          const uint32_t v_st = v_pos % L::kKVStages, k_st = k_pos % L::kKVStages;
          if (need_v && !mbar_wait(bar(L::kBarKVFull + v_st), (v_pos / L::kKVStages) & 1,
                                   abort_flag)) {
            ok = false;
            break;
          }
          if (need_k && !mbar_wait(bar(L::kBarKVFull + k_st), (k_pos / L::kKVStages) & 1,
                                   abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t v_base = sbase + L::kOffKV + v_st * L::kTileBytes;
          const uint32_t k_base = sbase + L::kOffKV + k_st * L::kTileBytes;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (j >= plo[t] + 1 && j <= phi[t]) {
              // GEMM 2: O_t += P_t(j-1) V_{j-1}
              if (!mbar_wait(bar(L::kBarPFull + t), p_seen[t] & 1, abort_flag)) {
                ok = false;
                break;
              }
              ++p_seen[t];
              if (j == plo[t] + 1 && units_t[t] > 0 &&
                  !mbar_wait(bar(L::kBarOFree + t), (units_t[t] - 1) & 1, abort_flag)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t v_lo = sdesc_lo(v_base, L::kBlockBytes);
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk)
                umma_ts_w(tmem + L::kColO + t * D, tmem + t * kTile + kk * 8,
                          v_lo + ((kk * 16 * 128) >> 4), kHi, kIdescO,
                          (j > plo[t] + 1 || kk > 0) ? 1u : 0u);
              if (j == phi[t]) umma_commit(bar(L::kBarOFinal + t));
            }
            if (j >= plo[t] && j < phi[t]) {
              // GEMM 1: S_t = Q_t K_j^T
              const uint32_t q_lo = sdesc_lo(q_base + t * L::kTileBytes, 16);
              const uint32_t k_lo = sdesc_lo(k_base, 16);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * L::kBlockBytes + (kk & 3) * 32) >> 4;
                if (kk == 0)
                  umma_ss_w<0>(tmem + t * kTile, q_lo + off, kHi, k_lo + off, kHi, kIdescS);
                else
                  umma_ss_w<1>(tmem + t * kTile, q_lo + off, kHi, k_lo + off, kHi, kIdescS);
              }
              umma_commit(bar(L::kBarSFull + t));
            }
          }
          if (!ok) break;
          // stages are released in ring order: V_{j-1} then K_j
          if (need_v) umma_commit(bar(L::kBarKVEmpty + v_st));
          if (need_k) umma_commit(bar(L::kBarKVEmpty + k_st));
          // the Q stage is free once the unit's last GEMM 1 has run
          if (j == nmax - 1) umma_commit(bar(L::kBarQEmpty + qs));
        }
        if (!ok) break;
        kv_it = base_it + 2 * nmax;
        ++q_it;
        for (int t = 0; t < 2; ++t)
          if (phi[t] > plo[t]) ++units_t[t];
      }
      // Every issued MMA must complete before TMEM is released.
      umma_commit(bar(L::kBarDrain));
      drain_wait(bar(L::kBarDrain), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int t = warp >> 2;           // query tile of the pair this group serves
    const int r = threadIdx.x & 127;   // query row inside the tile == TMEM lane
    const uint32_t t_row = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t col_s = t * kTile, col_o = L::kColO + t * D;
    uint32_t g = 0, nu = 0;  // S-full phases and units consumed by this group
    bool ok = true;
    for (int ri = 0, u = cta_unit(a, 0); ok && u >= 0; u = cta_unit(a, ++ri)) {
      int bh, pair, split;
      unit_coords(a, u, bh, pair, split);
      const int qt = 2 * pair + t;
      const int kv_len = batch_kv_len<kWin>(a, bh / a.Hq);
      int jlo, jhi;
      split_kv_range<kSplit>(a, wl, wr, kv_len, qt, split, jlo, jhi);
      const int q_row = qt * kTile + r;
      const size_t part_row = ((size_t)split * a.B * a.Hq + bh) * a.Sq + q_row;
      if (jhi == jlo) {
        // no key (of this split) reaches the tile: an empty part, or with a
        // window or padding the whole tile sees no key: O = 0, LSE = -inf
        if (kSplit && q_row < a.Sq) a.lse_part[part_row] = -INFINITY;
        if (!kSplit && kWin && q_row < a.Sq) {
          uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.o) +
                                                 ((size_t)bh * a.Sq + q_row) * D);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) orow[i] = make_uint4(0u, 0u, 0u, 0u);
          a.lse[(size_t)bh * a.Sq + q_row] = -INFINITY;
        }
        continue;
      }
      // keys [lo_row, lim) are visible to this row
      const int lim = wr >= 0 ? min(kv_len, q_row + wr + 1) : kv_len;
      const int lo_row = wl >= 0 ? max(0, q_row - wl) : 0;
      auto hidden = [&](int key) { return key >= lim || (kWin && key < lo_row); };
      // relative-position bias in log2 units: slope * log2(e) per key offset,
      // and the same per unit of raw score (slope2 / c) for the max pass
      const float slope2 = kBias ? a.alibi[bh % a.Hq] * 1.4426950408889634f : 0.f;
      const float kslope = kBias ? slope2 / a.scale_log2 : 0.f;
      const bool kslope_ok = kBias && a.scale_log2 > 0.f && fabsf(kslope) < 1e30f;
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = jlo; j < jhi; ++j) {
        if (!warp_wait(bar(L::kBarSFull + t), g & 1, abort_flag)) { ok = false; break; }
        ++g;
        tc_fence_after();
        const int kv0 = j * kTile;
        const bool masked_tile = kv0 + kTile > lim || (kWin && kv0 < lo_row);
        const float bias0 = slope2 * (float)(kv0 - q_row);  // bias of the tile's first key
        const float c = a.scale_log2;
        float alpha = 1.f;
        bool rescale = false;
        float2 sum2 = make_float2(0.f, 0.f);
        // Conditional rescale: keep a stale running max unless the new max
        // exceeds it by more than 8 (P then stays <= 2^8).
        auto update_max = [&](float tmax) {
          if (j == jlo) {
            m_run = tmax;
          } else if (tmax > m_run + 8.0f) {
            alpha = ex2_mufu(m_run - tmax);
            m_run = tmax;
            rescale = true;
          }
        };
        if (c > 0.f) {
          // Common case.  Pass 1: the whole score row in one TMEM round trip,
          // reduced to its max (masked columns skipped).  The plain kernel keeps
          // the row in registers for pass 2; the score-modified kernels, which
          // carry more live state, reload it.
          float mraw = -INFINITY;
          uint32_t v[kTile];
          {
            tmem_ld128(t_row + col_s, v);
            if (masked_tile) {
#pragma unroll
              for (int i = 0; i < kTile; ++i)
                if (hidden(kv0 + i)) v[i] = __float_as_uint(-INFINITY);
            }
            if (kBias && kslope_ok) {
              // the bias varies along the row: with c > 0 the max of
              // s*c + slope2*i + bias0 is c * max(s + k*i) + bias0, k = slope2 / c
#pragma unroll
              for (int i = 0; i < kTile; i += 2)
                mraw = fmax3(mraw, fmaf(kslope, (float)i, u2f(v[i])),
                             fmaf(kslope, (float)(i + 1), u2f(v[i + 1])));
            } else if (kBias) {
#pragma unroll
              for (int i = 0; i < kTile; i += 2)
                mraw = fmax3(mraw, fmaf(u2f(v[i]), c, fmaf(slope2, (float)i, bias0)),
                             fmaf(u2f(v[i + 1]), c, fmaf(slope2, (float)(i + 1), bias0)));
            } else {
#pragma unroll
              for (int i = 0; i < kTile; i += 2) mraw = fmax3(mraw, u2f(v[i]), u2f(v[i + 1]));
            }
          }
          if (mraw != -INFINITY) mraw = kBias ? (kslope_ok ? fmaf(mraw, c, bias0) : mraw) : mraw * c;
          update_max(mraw);
          const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
          // Pass 2, one half-row (64 scores) per round trip: P = 2^(s*c - m)
          // with one packed FMA per two scores; masked columns are -inf and
          // give P = 0.  Each half of P (32 packed columns) is stored over S
          // columns already read.
          const float2 c2 = make_float2(c, c), nm2 = make_float2(neg_m, neg_m);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t w0[32], w1[32], pk[32];
            if constexpr (kMod == 0) {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                w0[i] = v[h * 64 + i];
                w1[i] = v[h * 64 + 32 + i];
              }
            } else {
              __syncwarp();
              tmem_ld32(t_row + col_s + h * 64, w0);
              tmem_ld32(t_row + col_s + h * 64 + 32, w1);
              if (masked_tile) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                  if (hidden(kv0 + h * 64 + i)) w0[i] = __float_as_uint(-INFINITY);
                  if (hidden(kv0 + h * 64 + 32 + i)) w1[i] = __float_as_uint(-INFINITY);
                }
              }
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const uint32_t* src = (i < 16) ? w0 : w1;
              const int e = (i & 15) * 2;
              float2 add = nm2;
              if (kBias)  // bias of keys kv0 + h*64 + 2i, +1, minus the max
                add = __ffma2_rn(make_float2((float)(h * 64 + 2 * i), (float)(h * 64 + 2 * i + 1)),
                                 make_float2(slope2, slope2),
                                 make_float2(bias0 + neg_m, bias0 + neg_m));
              const float2 tt = __ffma2_rn(make_float2(u2f(src[e]), u2f(src[e + 1])), c2, add);
              float p0, p1;
              if ((i & 7) < L::kPolyPairs) {
                const float2 pp = ex2_poly2(tt);
                p0 = pp.x, p1 = pp.y;
              } else {
                p0 = ex2_mufu(tt.x), p1 = ex2_mufu(tt.y);
              }
              sum2 = __fadd2_rn(sum2, make_float2(p0, p1));
              pk[i] = pack_bf16x2(p0, p1);
            }
            __syncwarp();
            tmem_st32(t_row + col_s + h * 32, pk);
          }
        } else {
          // scale <= 0: two passes over TMEM, the max of s*c through min/max
          // of the raw scores, and masked columns zeroed explicitly (with
          // scale 0, -inf * 0 would be NaN).
          float mraw = (c == 0.f) ? -INFINITY : INFINITY;
#pragma unroll 1
          for (int cb = 0; cb < 4; ++cb) {
            uint32_t w[32];
            __syncwarp();
            tmem_ld32(t_row + col_s + cb * 32, w);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const bool dead = hidden(kv0 + cb * 32 + i);
              const float x = u2f(w[i]);
              if (kBias)  // s*c + bias (0 * s is 0 for the finite scores)
                mraw = dead ? mraw : fmaxf(mraw, fmaf(x, c, fmaf(slope2, (float)(cb * 32 + i), bias0)));
              else if (c == 0.f)
                mraw = dead ? mraw : fmaxf(mraw, 0.f * x);
              else
                mraw = dead ? mraw : fminf(mraw, x);
            }
          }
          const bool none = (kBias || c == 0.f) ? (mraw == -INFINITY) : (mraw == INFINITY);
          update_max(none ? -INFINITY : (kBias ? mraw : (c == 0.f ? 0.f : mraw * c)));
          const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            uint32_t w0[32], w1[32], pk[32];
            __syncwarp();
            tmem_ld32(t_row + col_s + h * 64, w0);
            tmem_ld32(t_row + col_s + h * 64 + 32, w1);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const uint32_t* src = (i < 16) ? w0 : w1;
              const int e = (i & 15) * 2, col = kv0 + h * 64 + 2 * i;
              const float b0 = fmaf(slope2, (float)(col - kv0), bias0) + neg_m;
              const float b1 = fmaf(slope2, (float)(col + 1 - kv0), bias0) + neg_m;
              float p0 = ex2_mufu(fmaf(u2f(src[e]), c, b0));
              float p1 = ex2_mufu(fmaf(u2f(src[e + 1]), c, b1));
              if (hidden(col)) p0 = 0.f;
              if (hidden(col + 1)) p1 = 0.f;
              sum2 = __fadd2_rn(sum2, make_float2(p0, p1));
              pk[i] = pack_bf16x2(p0, p1);
            }
            __syncwarp();
            tmem_st32(t_row + col_s + h * 32, pk);
          }
        }
        l_run = l_run * alpha + (sum2.x + sum2.y);
        // O_t is stable here: S_t(j) completing implies GEMM 2 of tile j-1 has
        // completed, and GEMM 2 of tile j waits for this thread's P.
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(t_row + col_o + cc * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(u2f(o[i]) * alpha);
            tmem_st32(t_row + col_o + cc * 32, o);
          }
        }
        tc_fence_before();
        mbar_arrive(bar(L::kBarPFull + t));
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16, LSE = ln2 * (m + log2 l)
      if (!warp_wait(bar(L::kBarOFinal + t), nu & 1, abort_flag)) { ok = false; break; }
      ++nu;
      tc_fence_after();
      const bool row_ok = q_row < a.Sq;
      if (kSplit) {
        // fp32 part: O / l and the part's LSE; a row with no visible key in
        // this split (its running max still -inf) is an empty part, O = 0 and
        // LSE = -inf.  (l alone does not show it: the polynomial 2^x gives a
        // tiny positive value, not 0, for the -inf of a hidden key.)
        const bool empty = m_run == -INFINITY || !(l_run > 0.f);
        const float inv = empty ? 0.f : 1.0f / l_run;
        // rows grp_row0 .. +3 of the lane group trade 16-byte pieces as in the
        // bf16 epilogue below, in two rounds of four pieces
        const int grp_row0 = qt * kTile + (r & ~3), pc = lane & 3;
        float* pbase = a.o_part + (part_row - (size_t)(r & 3)) * D;  // the group's first row
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          __syncwarp();
          tmem_ld32(t_row + col_o + c * 32, v);
          if (c == D / 32 - 1) {
            tc_fence_before();
            mbar_arrive(bar(L::kBarOFree + t));
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(u2f(v[i]) * inv);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
            for (int wd = 0; wd < 4; ++wd) {
              uint32_t x[4] = {v[16 * hf + wd], v[16 * hf + 4 + wd], v[16 * hf + 8 + wd],
                               v[16 * hf + 12 + wd]};
              xpose4(x, lane);
#pragma unroll
              for (int m = 0; m < 4; ++m) v[16 * hf + 4 * m + wd] = x[m];
            }
            // v[16hf + 4m .. +3] is now piece 4hf + pc of row grp_row0 + m
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              if (grp_row0 + m < a.Sq)
                *reinterpret_cast<uint4*>(pbase + (size_t)m * D + c * 32 + (4 * hf + pc) * 4) =
                    make_uint4(v[16 * hf + 4 * m], v[16 * hf + 4 * m + 1], v[16 * hf + 4 * m + 2],
                               v[16 * hf + 4 * m + 3]);
            }
          }
        }
        if (row_ok)
          a.lse_part[part_row] =
              empty ? -INFINITY : (m_run + __log2f(l_run)) * 0.69314718055994531f;
        continue;
      }
      // a row that sees no key (a window or padding) keeps the running max at
      // -inf: O = 0, LSE = -inf
      const bool no_key = kWin && (m_run == -INFINITY || !(l_run > 0.f));
      const float inv_l = no_key ? 0.f : 1.0f / l_run;
      const float row_lse = no_key ? -INFINITY : (m_run + __log2f(l_run)) * 0.69314718055994531f;
      if constexpr (D == 128) {
        // Each thread holds one row; so that a store instruction writes whole
        // 64-byte row pieces instead of 16 bytes of 32 rows, the four lanes of
        // a group trade 16-byte pieces (a 4x4 transpose): lane 4k+i then writes
        // piece i of rows 4k..4k+3.  O is released after its last TMEM read.
        const int grp_row0 = qt * kTile + (r & ~3), pc = lane & 3;
        __nv_bfloat16* obase = reinterpret_cast<__nv_bfloat16*>(a.o) + (size_t)bh * a.Sq * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          __syncwarp();  // reconverge after the per-row stores before the warp-wide load
          tmem_ld32(t_row + col_o + c * 32, v);
          if (c == D / 32 - 1) {
            tc_fence_before();
            mbar_arrive(bar(L::kBarOFree + t));
          }
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(u2f(v[2 * i]) * inv_l, u2f(v[2 * i + 1]) * inv_l);
#pragma unroll
          for (int wd = 0; wd < 4; ++wd) {  // word wd of each 16-byte piece
            uint32_t x[4] = {w[wd], w[4 + wd], w[8 + wd], w[12 + wd]};
            xpose4(x, lane);
#pragma unroll
            for (int m = 0; m < 4; ++m) w[4 * m + wd] = x[m];
          }
          // w[4m..4m+3] is now piece pc of row grp_row0 + m
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            if (grp_row0 + m < a.Sq)
              *reinterpret_cast<uint4*>(obase + (size_t)(grp_row0 + m) * D + c * 32 + pc * 8) =
                  make_uint4(w[4 * m], w[4 * m + 1], w[4 * m + 2], w[4 * m + 3]);
          }
        }
        if (row_ok) a.lse[(size_t)bh * a.Sq + q_row] = row_lse;
      } else {
        // D = 64: each thread stores its own row, and O is released after the
        // stores (both measured faster here than the D = 128 form, whose
        // shuffles cost the softmax-bound loop more than they save)
        __nv_bfloat16* orow =
            reinterpret_cast<__nv_bfloat16*>(a.o) + ((size_t)bh * a.Sq + (row_ok ? q_row : 0)) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          __syncwarp();  // reconverge after the per-row store before the warp-wide load
          tmem_ld32(t_row + col_o + c * 32, v);
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(u2f(v[2 * i]) * inv_l, u2f(v[2 * i + 1]) * inv_l);
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
        }
        if (row_ok) a.lse[(size_t)bh * a.Sq + q_row] = row_lse;
        tc_fence_before();
        mbar_arrive(bar(L::kBarOFree + t));
      }
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

template <int D>
static int launch_fwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        FwdArgs a, cudaStream_t stream) {
  using L = FwdLayout<D>;
  int dev;
  DeviceInfo info;
  if (!current_device(&dev, &info)) return FA_ERR_CUDA;
  static bool attr_done[64] = {};
  if (dev < 64 && !attr_done[dev]) {
    const void* kernels[] = {
        (const void*)fwd_kernel<D, 0, false>, (const void*)fwd_kernel<D, 1, false>,
        (const void*)fwd_kernel<D, 2, false>, (const void*)fwd_kernel<D, 0, true>,
        (const void*)fwd_kernel<D, 1, true>,  (const void*)fwd_kernel<D, 2, true>};
    for (const void* k : kernels)
      if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAllocBytes) !=
          cudaSuccess)
        return FA_ERR_CUDA;
    attr_done[dev] = true;
  }
  int* status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_fwd_status) != cudaSuccess)
    return FA_ERR_CUDA;
  a.status = status;
  const int sms = info.sm_count;
  int grid;
  if (a.n_split > 1) {
    a.sched = 3;
    a.chunk = 0;
    grid = a.n_units < sms ? a.n_units : sms;
  } else if (a.causal) {
    // longest-first snake over every head.  Also when K/V exceed L2: the CTAs
    // working on one head's pairs at the same time stream its K/V together
    // (measured on GB300 against contiguous per-CTA chunks of a head's pairs:
    // B2 H16 S8192 1,092 -> 1,267 TFLOP/s, S=16k 1,162 -> 1,350, S=32k
    // 1,369 -> 1,418; the chunks also left 24 SMs idle)
    a.sched = 2;
    a.chunk = 0;
    grid = a.n_units < sms ? a.n_units : sms;
  } else {
    a.sched = 0;
    a.chunk = 0;
    grid = a.n_units < sms ? a.n_units : sms;
  }
  record_timing(false, stream);
  // a window other than none / causal, a bias or key lengths select the general
  // kernel
  const bool plain_window = a.wl < 0 && (a.wr < 0 || (a.wr == 0 && a.causal));
  const int mode = a.alibi ? 2 : ((plain_window && !a.seqlens_k) ? 0 : 1);
  if (fwd_ring64_eligible(a, D, mode)) {
    if (launch_fwd_ring64(tq, tk, tv, a, grid, stream) != FA_OK) return FA_ERR_CUDA;
    record_timing(true, stream);
    note_launches(1);
    return FA_OK;
  }
  using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, FwdArgs);
  const KernelFn kernels[2][3] = {{fwd_kernel<D, 0, false>, fwd_kernel<D, 1, false>,
                                   fwd_kernel<D, 2, false>},
                                  {fwd_kernel<D, 0, true>, fwd_kernel<D, 1, true>,
                                   fwd_kernel<D, 2, true>}};
  if (launch_pdl(kernels[a.n_split > 1 ? 1 : 0][mode], dim3(grid), dim3(320), L::kAllocBytes,
                 stream, tq, tk, tv, a) != cudaSuccess)
    return FA_ERR_CUDA;
  record_timing(true, stream);
  note_launches(1);
  return FA_OK;
}

int launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const FwdArgs& a, int D, cudaStream_t stream) {
  if (D == 128) return launch_fwd_d<128>(tq, tk, tv, a, stream);
  if (D == 64) return launch_fwd_d<64>(tq, tk, tv, a, stream);
  return FA_ERR_UNSUPPORTED;
}

int fwd_status_take(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fwd_status, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_fwd_status, &zero, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  }
  return v == 0 ? FA_OK : v;
}

// ------------------------------------------------------------ exp2 test hook

__global__ void exp2_test_kernel(const float* __restrict__ x, float* __restrict__ y, int64_t n,
                                 int which) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
  {
    const float xi = x[i];
    if (which == 2)  // packed path: even elements through lane 0, odd through lane 1
      y[i] = (i & 1) ? ex2_poly2(make_float2(0.0f, xi)).y : ex2_poly2(make_float2(xi, 0.0f)).x;
    else
      y[i] = which ? ex2_poly(xi) : ex2_mufu(xi);
  }
}

int launch_exp2_test(const float* x, float* y, int64_t n, int which, cudaStream_t stream) {
  if (n == 0) return FA_OK;
  int dev;
  DeviceInfo info;
  if (!current_device(&dev, &info)) return FA_ERR_CUDA;
  const int64_t blocks64 = (n + 255) / 256;
  const int grid = (int)(blocks64 < 4L * info.sm_count ? blocks64 : 4L * info.sm_count);
  exp2_test_kernel<<<grid, 256, 0, stream>>>(x, y, n, which);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  note_launches(1);
  return FA_OK;
}

}  // namespace fa

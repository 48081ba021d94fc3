// fa_bwd_pair.cu -- the backward main kernel on pairs of SMs (D = 128, atomic dQ).
//
// FlashAttention-4 pages, key contribution #3: the backward pass runs its
// matrix products in the 2-CTA MMA mode and restructures the dQ reduction so
// that it takes half the global atomic adds.
//
// A cluster of two CTAs takes the kv tiles 2p (rank 0) and 2p+1 (rank 1) of one
// (batch, kv head): 256 keys, K and V of each tile in its own CTA's shared
// memory.  Rank 0 issues every MMA for both (tcgen05.mma.cta_group::2).  Both
// CTAs walk the union of the two tiles' query blocks (a block outside a tile's
// own range is fully masked for it) and, for each 64-row query block i:
//
//   S^T  = K Q_i^T,  dP^T = V dO_i^T    M = 256 keys (128 per SM, from its own
//                                        K / V), N = 64 queries: each CTA
//                                        supplies the 32 queries of its half
//                                        (rank r: rows 32r.. of the block);
//   P^T, dS^T                            the softmax warps of each CTA, on the
//                                        scores of its own keys (TMEM);
//   dV += P^T dO_i,  dK += dS^T Q_i      M = 256 keys (A = P^T / dS^T in each
//                                        SM's TMEM), N = 128 head dims: each
//                                        CTA supplies head dims 64r.. of all
//                                        64 queries;
//   dQ_i^T = K^T dS_i^T                  M = 128 head dims (64 per SM: head
//                                        dims 64r..), N = 64 queries (32 per
//                                        CTA: its half), K = all 256 keys.
//
// A pair MMA splits A by rows and B by columns, but both halves share the
// contraction: each SM multiplies its A rows by the partner's B columns too,
// so both CTAs lay out the contracted index in the same order (head dims in
// natural order for S^T, dP^T; queries for dV, dK; keys for dQ^T).  For dQ^T
// each CTA holds K^T of its head-dim half for both tiles and dS^T of all 256
// keys for its 32 queries, keys in pair order (tile 2p, then 2p+1); the
// softmax warps write the dS^T columns of the partner's queries into the
// partner's shared memory.  Each SM's TMEM then receives 64 head-dim rows of
// dQ_i^T summed over the 256 keys, in 32 columns: lane l holds head dim
// 64r + l % 64 of queries 32 (l / 64) ..  The drain adds them into the fp32
// accumulator: per query block, the pair issues as many adds as one CTA of the
// one-SM kernel, which adds a 128-key partial.
//
// Shared memory of each CTA (same offsets in both, which the pair MMAs need):
//   K, V of its own tile, K-major, 128-byte swizzle (S^T's and dP^T's A);
//   KT0, KT1: K of tiles 2p and 2p+1, head-dim half r (dQ^T's A; one of them
//   repeats this CTA's own half, since an operand address is the same in both
//   CTAs and the partner's KT slot holds partner data there);
//   3 stages of Q_i's and dO_i's rows 32r..32r+31 (S^T's and dP^T's B) and
//   their 64 rows of head-dim half r (dK's and dV's B, MN-major), with LSE2_i
//   and Delta_i beside them (all 64 queries: this CTA's softmax reads them);
//   the dS^T buffer [256 keys][32 queries] bf16, MN-major, 64-byte swizzle,
//   and 2 staging buffers for the 128 rows that go to the partner.
// TMEM (512 columns in each SM): S^T double buffer [0,64) [64,128), dP^T
// [128,192), dQ^T double buffer [192,224) [224,256), dV [256,384), dK [384,512).
//
// Warp roles, both CTAs: warps 0..7 P^T / dS^T (as in the one-SM kernel: warp
// w serves key rows 32 (w % 4).. and queries 32 (w / 4)..), warps 8..11 the dQ
// drain and the dK / dV epilogue, warp 12 the TMA producer, warp 13 the TMEM
// owner.  Rank 0 only: warp 13 issues S^T, warp 14 dP^T, warp 15 dV, dK, dQ^T.
// The TMA loads of both CTAs count their bytes on rank 0's barriers (the MMAs
// wait there); rank 0's commits arrive on the barrier at the same offset in
// both CTAs; the softmax, drain and epilogue warps of both CTAs hand back to
// rank 0's issuers with one arrival per warp, relaxed when it crosses CTAs:
// those hand-backs order TMEM accesses only (tcgen05 fences around them), and
// a cluster-scope release or proxy fence measured about 1,000 cycles each on
// the softmax warps' critical path.  The dS^T rows bound for the partner go
// through a local staging buffer and an async bulk copy (async proxy from end
// to end, so no cluster-scope proxy fence); warp 14 of rank 1 tells rank 0's
// dQ^T issuer when rank 1's buffer is complete.
#include <cuda_bf16.h>

#include <climits>

#include "bwd_common.cuh"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kPQB = 64;   // query rows per block
constexpr int kPD = 128;   // head dim

struct PairSmem {
  static constexpr int kKVBlockBytes = kTile * 128;  // 128 keys x 64 head dims
  static constexpr int kHalfBytes = 32 * 128;        // 32 query rows x 64 head dims
  static constexpr int kRowsBytes = kPQB * 128;      // 64 query rows x 64 head dims
  static constexpr int kOffK = 0;
  static constexpr int kOffV = 2 * kKVBlockBytes;
  static constexpr int kOffKT = 4 * kKVBlockBytes;   // KT0, KT1
  static constexpr int kKVTx = 6 * kKVBlockBytes;    // per CTA
  // stage (3): Q_i's and dO_i's rows 32r..32r+31, both head-dim halves (S^T's
  // and dP^T's B), and their 64 rows of head-dim half r (dK's and dV's B,
  // MN-major)
  static constexpr int kSQP = 0;
  static constexpr int kSQR = kSQP + 2 * kHalfBytes;
  static constexpr int kSDP = kSQR + kRowsBytes;
  static constexpr int kSDR = kSDP + 2 * kHalfBytes;
  static constexpr int kStageBytes = kSDR + kRowsBytes;  // all TMA bytes of a stage
  static constexpr int kStages = 3;
  static constexpr int kOffStage = 6 * kKVBlockBytes;
  static constexpr int kDSBytes = 2 * kTile * 64;  // 256 keys x 32 queries bf16
  static constexpr int kStgBytes = kTile * 64;     // 128 keys x 32 queries bf16
  static constexpr int kOffDS = kOffStage + kStages * kStageBytes;
  static constexpr int kOffStg = kOffDS + kDSBytes;      // 2 staging buffers
  static constexpr int kOffL = kOffStg + 2 * kStgBytes;  // per stage: LSE2 [64], Delta [64]
  static constexpr int kLBytes = 2 * kPQB * 4;
  static constexpr int kOffBar = kOffL + kStages * kLBytes;
  // rank 0 holds the barriers the issuers wait on; "both": the commits arrive
  // on each CTA's copy
  static constexpr int kBarKVFull = 0;                  // rank 0: K, V, KT of both (tx)
  static constexpr int kBarKVEmpty = 1;                 // both: every issuer commits
  static constexpr int kBarQFull = 2;                   // 3, rank 0: both stages' tiles (tx)
  static constexpr int kBarQEmpty = kBarQFull + 3;      // 3, both
  static constexpr int kBarLFull = kBarQEmpty + 3;      // 3, each CTA: LSE2, Delta (tx)
  static constexpr int kBarSFull = kBarLFull + 3;       // 2, both
  static constexpr int kBarPReady = kBarSFull + 2;      // 2, rank 0: 16 softmax warps
  static constexpr int kBarDPFull = kBarPReady + 2;     // both
  static constexpr int kBarDSReady = kBarDPFull + 1;    // 2, rank 0: 16 softmax warps
  static constexpr int kBarDQFull = kBarDSReady + 2;    // 2 (buffer = block parity), both
  static constexpr int kBarDQEmpty = kBarDQFull + 2;    // 2, rank 0: 8 drain warps
  static constexpr int kBarDKVFull = kBarDQEmpty + 2;   // both
  static constexpr int kBarDKVEmpty = kBarDKVFull + 1;  // rank 0: 8 epilogue warps
  static constexpr int kBarSFree = kBarDKVEmpty + 1;    // 2, rank 0
  static constexpr int kBarDrain = kBarSFree + 2;       // 3, rank 0: one per issuer
  static constexpr int kBarDSLocal = kBarDrain + 3;     // each CTA: its 4 local dS^T warps
  static constexpr int kBarDSRecv = kBarDSLocal + 1;    // each CTA: the partner's rows (tx)
  static constexpr int kBarDSPeer = kBarDSRecv + 1;     // rank 0: rank 1's buffer complete
  static constexpr int kNumBars = kBarDSPeer + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // TMEM slot, abort flag
  static constexpr int kBytes = kOffMisc + 16;
  // the launch asks for the largest opt-in size; the layout leaves more than
  // the 1023 bytes of padding a dynamic base can need for 1024-byte alignment
  static constexpr int kAllocBytes = 232448;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 192, kColDV = 256, kColDK = 384;
  static_assert(kOffStage % 1024 == 0 && kStageBytes % 1024 == 0 && kOffDS % 1024 == 0 &&
                    kOffStg % 1024 == 0,
                "swizzle atoms sit on 1024-byte boundaries");
  static_assert(kBytes + 1023 <= kAllocBytes, "shared memory per CTA");
};

constexpr int kPSmxWarps = 8, kPDrainWarp0 = 8, kPTmaWarp = 12, kPScoreWarp = 13;
constexpr int kPThreads = 512;

__global__ void __launch_bounds__(kPThreads, 1)
    bwd_main_pair(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_qh,
                  const __grid_constant__ CUtensorMap tm_doh, const BwdArgs a) {
  using L = PairSmem;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled tiles; the dynamic base is the same
  // in both CTAs, so are all offsets below
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  auto bar = [&](int i) -> uint32_t { return sbase + L::kOffBar + 8 * i; };
  // barrier i of rank 0, as a shared::cluster address
  auto lbar = [&](int i) -> uint32_t { return map_peer(bar(i), 0); };
  auto stage_off = [&](uint32_t it) -> uint32_t {
    return L::kOffStage + (it % L::kStages) * L::kStageBytes;
  };
  auto lse_off = [&](uint32_t it) -> uint32_t { return L::kOffL + (it % L::kStages) * L::kLBytes; };

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kBarKVFull), 1);
    mbar_init(bar(L::kBarKVEmpty), 3);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::kBarQFull + s), 1);
      mbar_init(bar(L::kBarQEmpty + s), 1);
      mbar_init(bar(L::kBarLFull + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kBarSFull + s), 1);
      mbar_init(bar(L::kBarPReady + s), 2 * kPSmxWarps);
      mbar_init(bar(L::kBarDSReady + s), 2 * kPSmxWarps);
      mbar_init(bar(L::kBarDQFull + s), 1);
      mbar_init(bar(L::kBarDQEmpty + s), 2 * 4);
      mbar_init(bar(L::kBarSFree + s), 1);
    }
    mbar_init(bar(L::kBarDPFull), 1);
    mbar_init(bar(L::kBarDKVFull), 1);
    mbar_init(bar(L::kBarDKVEmpty), 2 * 4);
    for (int s = 0; s < 3; ++s) mbar_init(bar(L::kBarDrain + s), 1);
    mbar_init(bar(L::kBarDSLocal), 4);
    mbar_init(bar(L::kBarDSRecv), 1);
    mbar_init(bar(L::kBarDSPeer), 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kPScoreWarp) {
    tmem_alloc_pair(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == kPTmaWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_qh);
    tma_prefetch_desc(&tm_doh);
  }
  tc_fence_before();
  // both CTAs' barriers are initialised before either signals the other
  cluster_sync_all();
  tc_fence_after();
  grid_dep_wait();
  grid_dep_launch();
  const uint32_t tmem = *tmem_slot;
  const int group = a.Hq / a.Hkv;
  // one arrival on rank 0's barrier i: local, or relaxed across the cluster
  auto arrive0 = [&](int i) {
    if (leader)
      mbar_arrive(bar(i));
    else
      mbar_arrive_remote(lbar(i));
  };
  auto next_unit = [&](int r) { return bwd_cta_unit_pair(a, r); };
  auto unit_of = [&](int u) { return bwd_unit_pair<false, kPQB>(a, u, group, (int)rank); };

  if (warp == kPTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0, unit = 0;
      bool ok = true;
      const uint32_t kv_full = lbar(L::kBarKVFull);
      // K and V of this CTA's tile and both tiles' K of head-dim half `rank`,
      // once every issuer is done with the previous ones
      auto load_kv = [&](const BwdUnit& w, uint32_t un) -> bool {
        if (!mbar_wait(bar(L::kBarKVEmpty), (un & 1) ^ 1, abort_flag)) return false;
        if (leader) mbar_arrive_expect_tx(bar(L::kBarKVFull), 2 * L::kKVTx);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          tma_load_3d_pair(sbase + L::kOffK + h * L::kKVBlockBytes, &tm_k, kv_full, h * 64,
                           w.j * kTile, w.bhk);
          tma_load_3d_pair(sbase + L::kOffV + h * L::kKVBlockBytes, &tm_v, kv_full, h * 64,
                           w.j * kTile, w.bhk);
        }
#pragma unroll
        for (int t = 0; t < 2; ++t)
          tma_load_3d_pair(sbase + L::kOffKT + t * L::kKVBlockBytes, &tm_k, kv_full,
                           (int)rank * 64, ((w.j & ~1) + t) * kTile, w.bhk);
        return true;
      };
      for (int ri = 0, u = next_unit(0); ok && u >= 0; u = next_unit(++ri), ++unit) {
        const BwdUnit w = unit_of(u);
        // the unit's first block goes out before its K / V (its stage frees
        // while the previous unit still holds K and V)
        const int early = w.n_it < 1 ? w.n_it : 1;
        for (int t = 0; t < w.n_it; ++t, ++it) {
          if (t == early) {
            if (!load_kv(w, unit)) { ok = false; break; }
          }
          const int gi = t / w.n_blk;
          const int iq = w.lo + (t - gi * w.n_blk);
          const int bh = w.b * a.Hq + w.hk * group + gi;
          const uint32_t st = it % L::kStages;
          if (!mbar_wait(bar(L::kBarQEmpty + st), ((it / L::kStages) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t sdst = sbase + stage_off(it);
          const uint32_t q_full = lbar(L::kBarQFull + st);
          if (leader) mbar_arrive_expect_tx(bar(L::kBarQFull + st), 2 * L::kStageBytes);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            tma_load_3d_pair(sdst + L::kSQP + h * L::kHalfBytes, &tm_qh, q_full, h * 64,
                             iq * kPQB + 32 * (int)rank, bh);
            tma_load_3d_pair(sdst + L::kSDP + h * L::kHalfBytes, &tm_doh, q_full, h * 64,
                             iq * kPQB + 32 * (int)rank, bh);
          }
          tma_load_3d_pair(sdst + L::kSQR, &tm_q, q_full, (int)rank * 64, iq * kPQB, bh);
          tma_load_3d_pair(sdst + L::kSDR, &tm_do, q_full, (int)rank * 64, iq * kPQB, bh);
          const size_t voff = (size_t)bh * a.Sq_pad + (size_t)iq * kPQB;
          mbar_arrive_expect_tx(bar(L::kBarLFull + st), 2 * kPQB * 4);
          const uint32_t ldst = sbase + lse_off(it);
          bulk_load(ldst, a.lse2 + voff, kPQB * 4, bar(L::kBarLFull + st));
          bulk_load(ldst + kPQB * 4, a.delta + voff, kPQB * 4, bar(L::kBarLFull + st));
        }
        if (ok && early == w.n_it && !load_kv(w, unit)) ok = false;
      }
      // no copy into either CTA may be in flight when the pair leaves: rank
      // 0's barriers count both CTAs' tiles
      const uint32_t first = it > (uint32_t)L::kStages ? it - L::kStages : 0;
      if (leader) {
        if (unit > 0) drain_wait_b(bar(L::kBarKVFull), (unit - 1) & 1);
        for (uint32_t n = first; n < it; ++n)
          drain_wait_b(bar(L::kBarQFull + n % L::kStages), (n / L::kStages) & 1);
      }
      for (uint32_t n = first; n < it; ++n)
        drain_wait_b(bar(L::kBarLFull + n % L::kStages), (n / L::kStages) & 1);
    }
  } else if (warp >= kPScoreWarp) {
    if (lane == 0 && !leader && warp == kPScoreWarp + 1) {
      // ------------------------------------------------------------ rank 1: dS^T buffer relay
      // this CTA's dS^T buffer is complete for block it once its 4 local warps
      // have written (and fenced) their rows and the partner's copy has landed
      uint32_t it = 0;
      bool ok = true;
      for (int ri = 0, u = next_unit(0); ok && u >= 0; u = next_unit(++ri)) {
        const BwdUnit w = unit_of(u);
        for (int t = 0; t < w.n_it; ++t, ++it) {
          mbar_arrive_expect_tx(bar(L::kBarDSRecv), L::kStgBytes);
          if (!mbar_wait(bar(L::kBarDSLocal), it & 1, abort_flag) ||
              !mbar_wait_cluster(bar(L::kBarDSRecv), it & 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_remote(lbar(L::kBarDSPeer));
        }
      }
    }
    // ------------------------------------------------------------ MMA issuers (rank 0)
    if (lane == 0 && leader) {
      constexpr uint32_t kIdS = idesc_bf16_f32(2 * kTile, kPQB, false, false);  // S^T, dP^T
      constexpr uint32_t kIdAcc = idesc_bf16_f32(2 * kTile, kPD, false, true);  // dV, dK
      constexpr uint32_t kIdDQ = idesc_bf16_f32(kPD, kPQB, true, true);         // dQ^T
      constexpr uint32_t kHi = sdesc_hi(1024);
      constexpr uint32_t kHi64 = sdesc_hi_sw64(512);
      const int role = warp - kPScoreWarp;  // 0: S^T, 1: dP^T, 2: gradients
      uint32_t it = 0, unit = 0;
      bool ok = true;
      for (int ri = 0, u = next_unit(0); ok && u >= 0; u = next_unit(++ri), ++unit) {
        const BwdUnit w = unit_of(u);
        if (!mbar_wait(bar(L::kBarKVFull), unit & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        if (role < 2) {
          // ---- S^T(i) = K Q_i^T or dP^T(i) = V dO_i^T, both operands K-major
          const uint32_t a_lo = sdesc_lo(sbase + (role == 0 ? L::kOffK : L::kOffV), 16);
          for (int t = 0; t < w.n_it; ++t, ++it) {
            const uint32_t q_base = sbase + stage_off(it);
            if (!mbar_wait(bar(L::kBarQFull + it % L::kStages), (it / L::kStages) & 1,
                           abort_flag)) {
              ok = false;
              break;
            }
            uint32_t d_col, b_lo, done;
            if (role == 0) {
              // the S^T buffer of block it-2 is free once its dV and dK are done
              if (it >= 2 && !mbar_wait(bar(L::kBarSFree + (it & 1)), ((it >> 1) - 1) & 1,
                                        abort_flag)) {
                ok = false;
                break;
              }
              d_col = L::kColS + (it & 1) * kPQB;
              b_lo = sdesc_lo(q_base + L::kSQP, 16);
              done = bar(L::kBarSFull + (it & 1));
            } else {
              // the dP^T columns are free once both CTAs' softmax warps have
              // read dP^T(it-1)
              if (it >= 1 && !mbar_wait_cluster(bar(L::kBarDSReady + ((it - 1) & 1)),
                                                ((it - 1) >> 1) & 1, abort_flag)) {
                ok = false;
                break;
              }
              d_col = L::kColDP;
              b_lo = sdesc_lo(q_base + L::kSDP, 16);
              done = bar(L::kBarDPFull);
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kPD / 16; ++kk) {
              const uint32_t ka = ((kk >> 2) * L::kKVBlockBytes + (kk & 3) * 32) >> 4;
              const uint32_t kb = ((kk >> 2) * L::kHalfBytes + (kk & 3) * 32) >> 4;
              umma_pair_ss(tmem + d_col, a_lo + ka, kHi, b_lo + kb, kHi, kIdS, kk > 0 ? 1u : 0u);
            }
            umma_pair_commit_both(done);
          }
          // K and V may be replaced once every issuer is done with them
          if (ok) umma_pair_commit_both(bar(L::kBarKVEmpty));
        } else {
          // ---- dV += P^T dO, dK += dS^T Q (A from TMEM), dQ^T = K^T dS^T
          if (unit > 0 &&
              !mbar_wait_cluster(bar(L::kBarDKVEmpty), (unit - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          for (int t = 0; t < w.n_it; ++t, ++it) {
            const uint32_t q_base = sbase + stage_off(it);
            // Q_i and dO_i rows of this CTA's head-dim half: MN-major B (K = queries)
            const uint32_t qr_lo = sdesc_lo(q_base + L::kSQR, L::kRowsBytes);
            const uint32_t dr_lo = sdesc_lo(q_base + L::kSDR, L::kRowsBytes);
            const uint32_t s_col = L::kColS + (it & 1) * kPQB;
            if (!mbar_wait_cluster(bar(L::kBarPReady + (it & 1)), (it >> 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // query columns 16kk..16kk+15 of P^T / dS^T: softmax part 16kk/32,
            // whose 32 columns hold P^T in the first 16 and dS^T in the last 16
            auto p_col = [&](int kk) { return s_col + (kk >> 1) * 32 + (kk & 1) * 8; };
#pragma unroll
            for (int kk = 0; kk < kPQB / 16; ++kk)  // dV += P^T dO  (K = queries)
              umma_pair_ts(tmem + L::kColDV, tmem + p_col(kk), dr_lo + ((kk * 16 * 128) >> 4),
                           kHi, kIdAcc, (t > 0 || kk > 0) ? 1u : 0u);
            if (!mbar_wait_cluster(bar(L::kBarDSReady + (it & 1)), (it >> 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kPQB / 16; ++kk)  // dK += dS^T Q
              umma_pair_ts(tmem + L::kColDK, tmem + p_col(kk) + 16,
                           qr_lo + ((kk * 16 * 128) >> 4), kHi, kIdAcc,
                           (t > 0 || kk > 0) ? 1u : 0u);
            // S^T, dP^T (complete before the softmax warps published dS^T), dV
            // and dK of this block are done with the stage and the S^T buffer
            umma_pair_commit_both(bar(L::kBarQEmpty + it % L::kStages));
            umma_pair_commit(bar(L::kBarSFree + (it & 1)));
            // dQ^T(i) into TMEM buffer i%2 once both drains have read dQ^T(i-2),
            // and once both CTAs' dS^T buffers hold block i
            mbar_arrive_expect_tx(bar(L::kBarDSRecv), L::kStgBytes);
            if ((it >= 2 && !mbar_wait_cluster(bar(L::kBarDQEmpty + (it & 1)),
                                               ((it >> 1) - 1) & 1, abort_flag)) ||
                !mbar_wait(bar(L::kBarDSLocal), it & 1, abort_flag) ||
                !mbar_wait_cluster(bar(L::kBarDSRecv), it & 1, abort_flag) ||
                !mbar_wait_cluster(bar(L::kBarDSPeer), it & 1, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t dsb = sbase + L::kOffDS;
#pragma unroll
            for (int kk = 0; kk < 2 * kTile / 16; ++kk) {
              // keys 16kk..: tile 2p, then 2p+1 (KT0, KT1 are contiguous)
              const uint32_t a_addr = sbase + L::kOffKT + kk * 2048;
              umma_pair_ss(tmem + L::kColDQ + (it & 1) * 32, sdesc_lo(a_addr, 16), kHi,
                           sdesc_lo(dsb + kk * 1024, 16), kHi64, kIdDQ, kk > 0 ? 1u : 0u);
            }
            umma_pair_commit_both(bar(L::kBarDQFull + (it & 1)));
          }
          if (ok) {
            umma_pair_commit_both(bar(L::kBarKVEmpty));
            umma_pair_commit_both(bar(L::kBarDKVFull));
          }
        }
      }
      umma_pair_commit(bar(L::kBarDrain + role));
      drain_wait_b(bar(L::kBarDrain + role), 0);
    }
  } else if (warp < kPSmxWarps) {
    // ------------------------------------------------------------ P^T / dS^T
    constexpr int kSC = 32;
    const int quarter = warp & 3;  // TMEM lanes 32*quarter.. = key rows
    const int part = warp >> 2;    // queries kSC*part..: the half that CTA `part` owns
    const int r = quarter * 32 + lane;
    const int c0 = part * kSC;
    const uint32_t t_row = tmem + ((uint32_t)(quarter * 32) << 16);
    // dS^T of these 32 queries goes to CTA `part`, key row 128 rank + r of its
    // buffer (keys in pair order: tile 2p, then 2p+1): written in place when
    // that is this CTA, else into row r of a staging buffer that this warp's
    // lane 0 copies to the partner (32 rows, 2 KB, contiguous in both)
    const bool ds_local = (int)rank == part;
    const uint32_t ds_row =
        ds_local ? (uint32_t)(L::kOffDS + (kTile * (int)rank + r) * 64) : (uint32_t)(L::kOffStg + r * 64);
    const int sw = (r & 7) >> 1;  // 64-byte swizzle: 16-byte chunk c sits at c ^ sw
    const uint32_t peer = rank ^ 1u;
    const uint32_t copy_dst =
        map_peer(sbase + L::kOffDS + (kTile * (int)rank + quarter * 32) * 64, peer);
    const uint32_t copy_bar = map_peer(bar(L::kBarDSRecv), peer);
    uint32_t it = 0;
    bool ok = true;
    for (int ri = 0, u = next_unit(0); ok && u >= 0; u = next_unit(++ri)) {
      const BwdUnit w = unit_of(u);
      const int kv = w.j * kTile + r;
      const bool row_dead = kv >= w.kv_len;
      for (int t = 0; t < w.n_it; ++t, ++it) {
        const int gi = t / w.n_blk;
        const int iq = w.lo + (t - gi * w.n_blk);
        const float4* s_lse2 = reinterpret_cast<const float4*>(smem + lse_off(it) + c0 * 4);
        const float4* s_delta = s_lse2 + kPQB / 4;
        if (!warp_wait_b(bar(L::kBarLFull + it % L::kStages), (it / L::kStages) & 1,
                         abort_flag)) {
          ok = false;
          break;
        }
        float lse[kSC];
#pragma unroll
        for (int q = 0; q < kSC / 4; ++q) {
          const float4 x = s_lse2[q];
          lse[4 * q] = -x.x, lse[4 * q + 1] = -x.y, lse[4 * q + 2] = -x.z, lse[4 * q + 3] = -x.w;
        }
        if (!warp_wait_b(bar(L::kBarSFull + (it & 1)), (it >> 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t s_col = L::kColS + (it & 1) * kPQB + c0;
        // column c is query q0 + c; with causal masking it sees key kv iff c >= kv - q0
        const int q0 = iq * kPQB + c0;
        const int c_lo = a.causal ? kv - q0 : INT_MIN;
        float p[kSC];
        {
          uint32_t v[kSC];
          tmem_ld<kSC>(t_row + s_col, v);
          // two columns per packed FMA (the same rounding as two fmaf); no
          // per-column mask when the whole segment is visible
          const float2 c2 = make_float2(a.scale_log2, a.scale_log2);
          const bool full = !row_dead && c_lo <= 0;
#pragma unroll
          for (int c = 0; c < kSC; c += 2) {
            const float2 t2 = __ffma2_rn(make_float2(u2f(v[c]), u2f(v[c + 1])), c2,
                                         make_float2(lse[c], lse[c + 1]));
            const float x0 = ex2_mufu(t2.x), x1 = ex2_mufu(t2.y);
            if (full) {
              p[c] = x0;
              p[c + 1] = x1;
            } else {
              p[c] = (row_dead || c < c_lo) ? 0.f : x0;
              p[c + 1] = (row_dead || c + 1 < c_lo) ? 0.f : x1;
            }
          }
        }
        {
          uint32_t wbuf[kSC / 2];
#pragma unroll
          for (int e = 0; e < kSC / 2; ++e) wbuf[e] = pack_bf16x2(p[2 * e], p[2 * e + 1]);
          tmem_st<kSC / 2>(t_row + s_col, wbuf);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive0(L::kBarPReady + (it & 1));
        float dl[kSC];
#pragma unroll
        for (int q = 0; q < kSC / 4; ++q) {
          const float4 x = s_delta[q];
          dl[4 * q] = x.x, dl[4 * q + 1] = x.y, dl[4 * q + 2] = x.z, dl[4 * q + 3] = x.w;
        }
        if (!warp_wait_b(bar(L::kBarDPFull), it & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        uint32_t wbuf[kSC / 2];
        {
          uint32_t v[kSC];
          tmem_ld<kSC>(t_row + L::kColDP + c0, v);
#pragma unroll
          for (int e = 0; e < kSC / 2; ++e) {
            // dS = P (dP - Delta), packed (the same roundings as the scalar form)
            const float2 d2 = __fmul2_rn(
                make_float2(p[2 * e], p[2 * e + 1]),
                __fadd2_rn(make_float2(u2f(v[2 * e]), u2f(v[2 * e + 1])),
                           make_float2(-dl[2 * e], -dl[2 * e + 1])));
            const float d0 = d2.x, d1 = d2.y;
            wbuf[e] = pack_bf16x2(d0, d1);
          }
        }
        tmem_st<kSC / 2>(t_row + s_col + kSC / 2, wbuf);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        // dP^T read and dS^T in TMEM: dK(it) and dP^T(it+1) may go
        if (lane == 0) arrive0(L::kBarDSReady + (it & 1));
        // dS^T into shared memory for dQ^T: the buffer (here and in the
        // partner) is free once dQ^T(it-1) is done, staging buffer it%2 once
        // dQ^T(it-2) is (the copy from it had landed before dQ^T(it-2) began)
        const uint32_t prev = it - 1;
        if (ds_local) {
          if (it >= 1 &&
              !warp_wait_b(bar(L::kBarDQFull + (prev & 1)), (prev >> 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
        } else if (it >= 2 &&
                   !warp_wait_b(bar(L::kBarDQFull + (it & 1)), ((it - 2) >> 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t boff = ds_local ? 0u : (it & 1) * (uint32_t)L::kStgBytes;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
          *reinterpret_cast<uint4*>(smem + ds_row + boff + ((ch ^ sw) << 4)) =
              make_uint4(wbuf[4 * ch], wbuf[4 * ch + 1], wbuf[4 * ch + 2], wbuf[4 * ch + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (ds_local) {
            mbar_arrive(bar(L::kBarDSLocal));
          } else if (it >= 1 &&
                     !mbar_wait(bar(L::kBarDQFull + (prev & 1)), (prev >> 1) & 1, abort_flag)) {
            ok = false;
          } else {
            bulk_copy_to_peer(copy_dst, sbase + L::kOffStg + boff + quarter * 32 * 64, 32 * 64,
                              copy_bar);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      }
    }
  } else if (warp < kPTmaWarp) {
    // ------------------------------------------------------------ dQ drain + dK/dV epilogue
    const int r = threadIdx.x - 32 * kPDrainWarp0;  // TMEM lane
    const int wq = warp - kPDrainWarp0;
    const uint32_t t_row = tmem + ((uint32_t)(wq * 32) << 16);
    // lane r of dQ^T holds head dim 64 rank + r % 64 of queries 32 (r / 64) ..
    const int dh = 64 * (int)rank + (r & 63);
    const int qoff = 32 * (r >> 6);

    uint32_t it = 0, unit = 0;
    bool ok = true;
    for (int ri = 0, u = next_unit(0); ok && u >= 0; u = next_unit(++ri), ++unit) {
      const BwdUnit w = unit_of(u);
      for (int t = 0; t < w.n_it; ++t, ++it) {
        const int gi = t / w.n_blk;
        const int iq = w.lo + (t - gi * w.n_blk);
        const int bh = w.b * a.Hq + w.hk * group + gi;
        ok = group_all(warp_wait_b(bar(L::kBarDQFull + (it & 1)), (it >> 1) & 1, abort_flag), 2);
        if (!ok) break;
        tc_fence_after();
        uint32_t v[32];
        tmem_ld32(t_row + L::kColDQ + (it & 1) * 32, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive0(L::kBarDQEmpty + (it & 1));
        // for each query the 32 lanes of a warp add 32 consecutive floats (one
        // 128-byte line per instruction)
        float* dst = a.dq_acc + ((size_t)bh * a.Sq_pad + (size_t)iq * kPQB + qoff) * kPD + dh;
#pragma unroll
        for (int e = 0; e < 32; ++e)
          asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(dst + (size_t)e * kPD),
                       "f"(u2f(v[e]))
                       : "memory");
      }
      if (!ok) break;
      // ---- dK, dV epilogue for key row kv of this CTA's tile
      ok = group_all(warp_wait_b(bar(L::kBarDKVFull), unit & 1, abort_flag), 2);
      if (!ok) break;
      tc_fence_after();
      // the four lanes of a group trade 16-byte pieces (a 4x4 transpose) so
      // that lane 4k+i writes piece i of rows 4k..4k+3: whole 64-byte row
      // pieces per warp instruction
      const int grp = lane & ~3, pc = lane & 3;
      const int row0 = w.j * kTile + wq * 32 + grp;
      __nv_bfloat16* dk_base = reinterpret_cast<__nv_bfloat16*>(a.dk) + (size_t)w.bhk * a.Sk * kPD;
      __nv_bfloat16* dv_base = reinterpret_cast<__nv_bfloat16*>(a.dv) + (size_t)w.bhk * a.Sk * kPD;
#pragma unroll 1
      for (int pass = 0; pass < 2 * (kPD / 32); ++pass) {
        const int c = pass >> 1;
        const bool is_v = (pass & 1) != 0;
        uint32_t vk[32];
        __syncwarp();
        if (w.n_it > 0) {
          tmem_ld32(t_row + (is_v ? L::kColDV : L::kColDK) + c * 32, vk);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) vk[e] = 0u;
        }
        if (pass == 2 * (kPD / 32) - 1) {
          // every TMEM read of dK / dV is done: the accumulators are free
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive0(L::kBarDKVEmpty);
        }
        const float sc = is_v ? 1.f : a.scale;
        uint32_t wk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) wk[e] = pack_bf16x2(u2f(vk[2 * e]) * sc, u2f(vk[2 * e + 1]) * sc);
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
          uint32_t xk[4] = {wk[wd], wk[4 + wd], wk[8 + wd], wk[12 + wd]};
          xpose4(xk, lane);
#pragma unroll
          for (int m = 0; m < 4; ++m) wk[4 * m + wd] = xk[m];
        }
        __nv_bfloat16* base = is_v ? dv_base : dk_base;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          if (row0 + m < a.Sk) {
            const size_t off = (size_t)(row0 + m) * kPD + c * 32 + pc * 8;
            *reinterpret_cast<uint4*>(base + off) =
                make_uint4(wk[4 * m], wk[4 * m + 1], wk[4 * m + 2], wk[4 * m + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  // neither CTA leaves while the pair's MMAs, copies or stores into its shared
  // memory may still run
  cluster_sync_all();
  if (warp == kPScoreWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, L::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(a.status, (int)FA_ERR_TIMEOUT);
}

}  // namespace

bool bwd_pair_eligible(const BwdArgs& a, bool mod) {
  return a.D == kPD && !a.deterministic && !mod;
}

// Clusters of two CTAs, as many as can be resident at once (up to one per
// pair unit).
int launch_bwd_main_pair(const BwdMaps& m, const BwdArgs& a, cudaStream_t stream) {
  using L = PairSmem;
  int dev;
  DeviceInfo info;
  if (!current_device(&dev, &info) || dev >= 64) return FA_ERR_CUDA;
  static int max_clusters[64] = {};
  int& mc = max_clusters[dev];
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = L::kAllocBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  if (mc == 0) {
    if (cudaFuncSetAttribute(bwd_main_pair, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::kAllocBytes) != cudaSuccess)
      return FA_ERR_CUDA;
    cfg.gridDim = dim3(info.sm_count & ~1);
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (const void*)bwd_main_pair, &cfg) != cudaSuccess ||
        n < 1)
      return FA_ERR_CUDA;
    mc = n;
  }
  BwdArgs ap = a;
  ap.n_units = a.B * a.Hkv * ((a.n_ktiles + 1) / 2);
  const int clusters = ap.n_units < mc ? ap.n_units : mc;
  cfg.gridDim = dim3(2 * (clusters > 0 ? clusters : 1));
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, bwd_main_pair, m.q, m.k, m.v, m.dO, m.q_half, m.dO_half, ap) !=
      cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // namespace fa

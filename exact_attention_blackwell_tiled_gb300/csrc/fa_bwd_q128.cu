// fa_bwd_q128.cu -- backward main kernel with 128-row query blocks (D = 128).
//
// The mathematics, the unit schedule and the dQ accumulation modes are those of
// bwd_main in fa_bwd.cu (the textbook gradient of exact attention with P
// recomputed from the saved log-sum-exp; FlashAttention-4 pages, key
// contribution #3: tensor-memory accumulators in the backward pass, and the
// Limitations list's deterministic mode that serialises the reductions through
// semaphores).  What changes is the query step: a unit (batch, kv head,
// 128-row kv tile j) walks 128-row query blocks i, so every GEMM is a full
// M = 128, N = 128 tcgen05 MMA:
//   S^T    = K_j Q_i^T        SS, both operands K-major      TMEM [0,128)
//   P^T    = 2^(S^T*c - LSE2_i) -> bf16 over S^T columns already read
//   dP^T   = V_j dO_i^T       SS                             TMEM [128,256)
//   dS^T   = P^T * (dP^T - Delta_i) -> bf16 in TMEM and shared memory
//   dV    += P^T dO_i         TS, A = P^T from TMEM          TMEM [256,384)
//   dK    += dS^T Q_i         TS, A = dS^T from TMEM         TMEM [384,512)
//   dQ_i^T = K_j^T dS_i^T     SS, both MN-major, written over the dP^T columns
//                             once the softmax warps have read them
// With 64-row blocks the N = 64 MMAs re-read the 128-row K or V operand for
// every 64 queries: 6 KB of shared memory per K = 16 step against 32 cycles of
// tensor work, which measured 54 cycles per step (shared-memory bound).  At
// N = 128 a step reads 8 KB in 64 cycles, which shared memory sustains, and the
// four operand-read streams per 128 queries drop from 352 KB to 256 KB.
//
// TMEM is full (512 columns), so S^T and dP^T are single-buffered and dQ^T
// shares the dP^T columns.  One thread issues, per block i, dV(i), dK(i),
// S^T(i+1), dQ^T(i): S^T(i+1) overwrites the columns dK(i) reads, which the
// in-order execution of one thread's MMAs makes safe without a wait, and it
// goes ahead of dQ^T(i) because the softmax warps wait for it.  Another
// thread issues dP^T(i+1) once the drain has read dQ^T(i).
//
// Warp roles (512 threads, 128 registers):
//   warps 0-7   P^T / dS^T: warp w serves key rows 32*(w%4).. (its TMEM lanes)
//               and query columns 64*(w/4).. of the block.  Its P^T goes to
//               columns 64*(w/4) .. +31 (bf16 pairs), its dS^T to the next 32,
//               both over S^T columns it has already read, so the two column
//               halves never touch each other's columns.
//   warps 8-11  dQ drain (one head-dim row of dQ^T per thread, 184 registers
//               after a setmaxnreg split) and the dK/dV epilogue at the end of
//               a unit.
//   warp 12     TMA producer: K_j, V_j per unit; Q_i, dO_i, LSE2_i, Delta_i per
//               block into a 2-stage ring.  With dynamic dealing (the
//               deterministic mode with the snake order) it also takes each
//               unit number from the global counter.
//   warp 13     TMEM owner; one thread issues S^T, dV, dK and dQ^T.
//   warp 14     one thread issues dP^T.
//   warp 15     deterministic mode: one thread raises the dQ semaphores once
//               the drain warps have added a block (so that no drain warp
//               waits for its adds to reach L2).
// Warps 12-15 run with 72 registers after the setmaxnreg split.
#include <cuda_bf16.h>

#include <climits>

#include "bwd_common.cuh"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kQB2 = 128;  // query rows per block

struct Q128Layout {
  static constexpr int D = 128;
  static constexpr int kBlockBytes = kTile * 128;    // 128 rows x 64 columns bf16
  static constexpr int kTileBytes = kTile * D * 2;   // a 128 x 128 bf16 tile
  static constexpr int kStages = 2;
  static constexpr int kVecBytes = kQB2 * 4;         // LSE2 or Delta of a block
  static constexpr int kStageBytes = 2 * kTileBytes + 2 * kVecBytes;  // Q, dO, LSE2, Delta
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffStage = kOffV + kTileBytes;
  // dS^T [key][query] for the dQ^T MMA: two 64-query column blocks of 128 key
  // rows x 128 bytes, 128-byte swizzled
  static constexpr int kOffDS = kOffStage + kStages * kStageBytes;
  static constexpr int kDSBytes = kTile * kQB2 * 2;
  static constexpr int kOffBar = kOffDS + kDSBytes;
  static constexpr int kBarKVFull = 0, kBarKVEmpty = 1;
  static constexpr int kBarQFull = 2;                 // kStages
  static constexpr int kBarQEmpty = 2 + kStages;      // kStages
  static constexpr int kBarSFull = 2 + 2 * kStages;
  static constexpr int kBarPReady = kBarSFull + 1;
  static constexpr int kBarDPFull = kBarPReady + 1;
  static constexpr int kBarDSReady = kBarDPFull + 1;
  static constexpr int kBarDQFull = kBarDSReady + 1;
  static constexpr int kBarDQEmpty = kBarDQFull + 1;
  static constexpr int kBarDKVFull = kBarDQEmpty + 1;
  static constexpr int kBarDKVEmpty = kBarDKVFull + 1;
  static constexpr int kBarDQAdded = kBarDKVEmpty + 1;    // drain warps -> semaphore warp
  static constexpr int kBarDQAddedFree = kBarDQAdded + 1;  // semaphore warp -> drain warps
  static constexpr int kBarDrain = kBarDQAddedFree + 1;    // 2: one per issuer
  static constexpr int kURing = 8;  // dynamically dealt units posted by the TMA thread
  static constexpr int kBarUFull = kBarDrain + 2;        // kURing
  static constexpr int kBarUEmpty = kBarUFull + kURing;  // kURing
  static constexpr int kNumBars = kBarUEmpty + kURing;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // TMEM slot, abort flag
  static constexpr int kOffURing = kOffMisc + 16;
  static constexpr int kBytes = kOffURing + 4 * kURing;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 128, kColDV = 256, kColDK = 384;
  // warp roles
  static constexpr int kSmxWarps = 8;
  static constexpr int kSmxCols = 64;  // query columns per softmax warp
  static constexpr int kDrainWarp0 = 8;
  static constexpr int kTmaWarp = 12;
  static constexpr int kScoreWarp = 13;  // TMEM owner; S^T and gradient issuer
  static constexpr int kDPWarp = 14;     // dP^T issuer
  static constexpr int kSemWarp = 15;    // raises the deterministic mode's semaphores
  static constexpr int kThreads = 512;
  static constexpr int kSmxThreads = 256;
  static constexpr int kRegsLaunch = 128;  // 65536 / kThreads
  static constexpr int kRegsDrain = 184;   // warps 8-11 after setmaxnreg
  static constexpr int kRegsIssue = 72;    // warps 12-15 after setmaxnreg
};
static_assert(2 * 128 * Q128Layout::kRegsLaunch + 128 * Q128Layout::kRegsDrain +
                      128 * Q128Layout::kRegsIssue ==
                  Q128Layout::kThreads * Q128Layout::kRegsLaunch,
              "the register split must add up to the launch's registers");

static_assert(Q128Layout::kDPWarp == Q128Layout::kScoreWarp + 1 &&
                  Q128Layout::kSemWarp == Q128Layout::kScoreWarp + 2 &&
                  Q128Layout::kThreads == 32 * (Q128Layout::kSemWarp + 1) &&
                  Q128Layout::kTmaWarp % 4 == 0,
              "warps 12-15 (TMA, issuers, semaphores) form the last warpgroup");

// Shared memory the launch asks for: the layout plus whatever of the largest
// opt-in size is left, for aligning the layout to 1024 bytes (the kernel checks
// that the dynamic base leaves enough).
constexpr int kQ128MaxSmem = 232448;
static_assert(Q128Layout::kBytes <= kQ128MaxSmem, "q128 backward layout exceeds shared memory");

}  // namespace

template <bool kMod>
__global__ void __launch_bounds__(Q128Layout::kThreads, 1)
    bwd_main_q128(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_do, const BwdArgs a, int smem_bytes) {
  using L = Q128Layout;
  constexpr int D = L::D;
  extern __shared__ uint8_t smem_raw[];
  // The 128-byte-swizzled tiles need 1024-byte alignment.  The layout leaves
  // less than 1024 bytes of slack, so a dynamic base that needs more padding
  // than that ends the kernel with an error status before anything runs.
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  if (pad + (uint32_t)L::kBytes > (uint32_t)smem_bytes) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicExch(a.status, (int)FA_ERR_UNSUPPORTED);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return sbase + L::kOffBar + 8 * i; };
  auto stage_off = [&](uint32_t it) -> uint32_t {
    return L::kOffStage + (it % L::kStages) * L::kStageBytes;
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kBarKVFull), 1);
    mbar_init(bar(L::kBarKVEmpty), 2);  // both issuers commit
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::kBarQFull + s), 1);
      mbar_init(bar(L::kBarQEmpty + s), 1);
    }
    mbar_init(bar(L::kBarSFull), 1);
    mbar_init(bar(L::kBarPReady), L::kSmxThreads);
    mbar_init(bar(L::kBarDPFull), 1);
    mbar_init(bar(L::kBarDSReady), L::kSmxThreads);
    mbar_init(bar(L::kBarDQFull), 1);
    mbar_init(bar(L::kBarDQEmpty), 128);
    mbar_init(bar(L::kBarDKVFull), 1);
    mbar_init(bar(L::kBarDKVEmpty), 128);
    mbar_init(bar(L::kBarDQAdded), 128);  // every drain thread
    mbar_init(bar(L::kBarDQAddedFree), 1);
    for (int s = 0; s < 2; ++s) mbar_init(bar(L::kBarDrain + s), 1);
    // readers of a posted unit: the softmax and drain warps, both issuing
    // threads and, in the deterministic mode, the semaphore thread
    for (int s = 0; s < L::kURing; ++s) {
      mbar_init(bar(L::kBarUFull + s), 1);
      mbar_init(bar(L::kBarUEmpty + s), L::kSmxWarps + 4 + 2 + (a.deterministic ? 1 : 0));
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == L::kScoreWarp) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish();
  }
  if (warp == L::kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the prologue above overlaps the preprocess kernel; its outputs (LSE2,
  // Delta, the cleared dQ accumulator and semaphores) are read from here on
  grid_dep_wait();
  grid_dep_launch();
  const uint32_t tmem = *tmem_slot;
  const int group = a.Hq / a.Hkv;
  // The r-th unit of this CTA: static dealing computes it in every role;
  // dynamic dealing has the TMA thread take the next number from the global
  // counter and post it in ring slot r % kURing, where the other roles read it.
  // Units are taken in dealing order, so a tile still waits only for tiles
  // taken before it.
  volatile int* uring = reinterpret_cast<volatile int*>(smem + L::kOffURing);
  auto take_unit = [&](int r) -> int {
    if (!a.dyn) return bwd_cta_unit(a, r);
    const int s = r % L::kURing;
    if (!mbar_wait(bar(L::kBarUEmpty + s), ((r / L::kURing) & 1) ^ 1, abort_flag)) return -1;
    int u = atomicAdd(a.unit_counter, 1);
    if (u >= a.n_units) u = -1;
    uring[s] = u;
    mbar_arrive(bar(L::kBarUFull + s));
    return u;
  };
  auto read_unit = [&](int r, bool warp_wide) -> int {
    if (!a.dyn) return bwd_cta_unit(a, r);
    const int s = r % L::kURing;
    bool got = mbar_wait(bar(L::kBarUFull + s), (r / L::kURing) & 1, abort_flag);
    if (warp_wide) got = __all_sync(0xffffffffu, got);
    const int u = got ? uring[s] : -1;
    if (warp_wide) __syncwarp();
    if (!warp_wide || lane == 0) mbar_arrive(bar(L::kBarUEmpty + s));
    return u;
  };
  // Register split (512 threads x 128 at launch): the TMA / issuer warpgroup
  // gives up 56 per thread, the drain warpgroup takes them, so that a drain
  // thread holds its whole 128-column row of dQ^T and releases the columns
  // after one TMEM round trip.  2 x 128 x 128 + 128 x 184 + 128 x 72 = 65536.
  // Each warpgroup runs its setmaxnreg at the top of its own branch.

  // Every barrier below is waited on by its consumers one phase at a time: a
  // phase k+1 can only complete after each consumer has passed phase k (S^T(i+1)
  // follows dK(i), which follows P^T(i) and dS^T(i); dP^T(i+1) follows the
  // drain of dQ^T(i), which follows dS^T(i); the drain of dQ^T(i+1) follows
  // dS^T(i+1), which follows dP^T(i+1)), so a single barrier with the block's
  // parity serves each hand-off.
  if (warp >= L::kTmaWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(L::kRegsIssue));
  if (warp == L::kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0, unit = 0;
      bool ok = true;
      auto load_kv = [&](const BwdUnit& w, uint32_t un) -> bool {
        if (!mbar_wait(bar(L::kBarKVEmpty), (un & 1) ^ 1, abort_flag)) return false;
        mbar_arrive_expect_tx(bar(L::kBarKVFull), 2 * L::kTileBytes);
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
          tma_load_3d(sbase + L::kOffK + cb * L::kBlockBytes, &tm_k, bar(L::kBarKVFull), cb * 64,
                      w.j * kTile, w.bhk);
          tma_load_3d(sbase + L::kOffV + cb * L::kBlockBytes, &tm_v, bar(L::kBarKVFull), cb * 64,
                      w.j * kTile, w.bhk);
        }
        return true;
      };
      for (int ri = 0, u = take_unit(0); ok && u >= 0; u = take_unit(++ri), ++unit) {
        const BwdUnit w = bwd_unit<kMod, kQB2>(a, u, group);
        // the unit's first block's Q / dO go out before its K / V: that stage
        // frees while the previous unit still holds K and V
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
          mbar_arrive_expect_tx(bar(L::kBarQFull + st), 2 * L::kTileBytes + 2 * L::kVecBytes);
#pragma unroll
          for (int cb = 0; cb < 2; ++cb) {
            tma_load_3d(sdst + cb * L::kBlockBytes, &tm_q, bar(L::kBarQFull + st), cb * 64,
                        iq * kQB2, bh);
            tma_load_3d(sdst + L::kTileBytes + cb * L::kBlockBytes, &tm_do,
                        bar(L::kBarQFull + st), cb * 64, iq * kQB2, bh);
          }
          const size_t voff = (size_t)bh * a.Sq_pad + (size_t)iq * kQB2;
          bulk_load(sdst + 2 * L::kTileBytes, a.lse2 + voff, L::kVecBytes,
                      bar(L::kBarQFull + st));
          bulk_load(sdst + 2 * L::kTileBytes + L::kVecBytes, a.delta + voff, L::kVecBytes,
                      bar(L::kBarQFull + st));
        }
        if (ok && early == w.n_it && !load_kv(w, unit)) ok = false;
      }
      if (unit > 0) drain_wait_b(bar(L::kBarKVFull), (unit - 1) & 1);
      for (uint32_t n = (it > (uint32_t)L::kStages ? it - L::kStages : 0); n < it; ++n)
        drain_wait_b(bar(L::kBarQFull + n % L::kStages), (n / L::kStages) & 1);
    }
  } else {
    // ------------------------------------------------------------ MMA issuers
    // Warp 13: S^T and the gradients dV, dK, dQ^T from one thread, so that
    // S^T(i+1) enters the tensor pipe right behind dK(i), the last reader of
    // S^T(i)'s columns, without waiting for dK(i) to complete (the MMAs of one
    // thread run in issue order), and ahead of dQ^T(i), whose result is not
    // needed as soon.  Warp 14: dP^T.  Warp 15 issues nothing; in the
    // deterministic mode it raises the dQ semaphores.
    if (lane == 0 && warp <= L::kDPWarp) {
      constexpr uint32_t kIdS = idesc_bf16_f32(kTile, kQB2, false, false);  // S^T, dP^T
      constexpr uint32_t kIdAcc = idesc_bf16_f32(kTile, D, false, true);    // dV, dK
      constexpr uint32_t kIdDQ = idesc_bf16_f32(D, kQB2, true, true);       // dQ^T
      constexpr uint32_t kHi = sdesc_hi(1024);
      const bool grad = warp == L::kScoreWarp;
      // S^T = K Q_i^T or dP^T = V dO_i^T: M = 128 keys, N = 128 queries,
      // K = head dim; both operands K-major, two 64-column blocks each
      auto issue_kmajor = [&](uint32_t d_col, uint32_t a_lo, uint32_t b_lo) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * L::kBlockBytes + (kk & 3) * 32) >> 4;
          if (kk == 0)
            umma_ss_w<0>(tmem + d_col, a_lo + off, kHi, b_lo + off, kHi, kIdS);
          else
            umma_ss_w<1>(tmem + d_col, a_lo + off, kHi, b_lo + off, kHi, kIdS);
        }
      };
      uint32_t it = 0, unit = 0;
      bool ok = true;
      for (int ri = 0, u = read_unit(0, false); ok && u >= 0; u = read_unit(++ri, false), ++unit) {
        const BwdUnit w = bwd_unit<kMod, kQB2>(a, u, group);
        if (!mbar_wait(bar(L::kBarKVFull), unit & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        if (!grad) {
          // ---- dP^T(i) = V dO_i^T over the columns of dQ^T(i-1), free once
          // the drain has read them
          const uint32_t v_lo = sdesc_lo(sbase + L::kOffV, 16);
          for (int t = 0; t < w.n_it; ++t, ++it) {
            if (!mbar_wait(bar(L::kBarQFull + it % L::kStages), (it / L::kStages) & 1,
                           abort_flag) ||
                (it >= 1 && !mbar_wait(bar(L::kBarDQEmpty), (it - 1) & 1, abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_kmajor(L::kColDP, v_lo, sdesc_lo(sbase + stage_off(it) + L::kTileBytes, 16));
            umma_commit(bar(L::kBarDPFull));
          }
          // V may be replaced once this issuer is done with it
          if (ok) umma_commit(bar(L::kBarKVEmpty));
        } else {
          // ---- S^T(i+1); dV += P^T dO, dK += dS^T Q (A from TMEM); dQ^T = K^T dS^T
          const uint32_t k_lo = sdesc_lo(sbase + L::kOffK, 16);
          // K^T as the MN-major A operand of dQ^T: head-dim rows 64.. are the
          // second column block of K
          const uint32_t kt_lo = sdesc_lo(sbase + L::kOffK, L::kBlockBytes);
          // dS^T as the MN-major B operand: queries 64.. are the second block
          const uint32_t ds_lo = sdesc_lo(sbase + L::kOffDS, L::kDSBytes / 2);
          // dV / dK accumulators are free once the previous unit's epilogue
          // has read them
          if (unit > 0 && !mbar_wait(bar(L::kBarDKVEmpty), (unit - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          // S^T of the unit's first block (S^T(i+1) of later blocks follows dK(i))
          auto issue_s = [&](uint32_t i) -> bool {
            if (!mbar_wait(bar(L::kBarQFull + i % L::kStages), (i / L::kStages) & 1, abort_flag))
              return false;
            tc_fence_after();
            issue_kmajor(L::kColS, k_lo, sdesc_lo(sbase + stage_off(i), 16));
            umma_commit(bar(L::kBarSFull));
            return true;
          };
          if (w.n_it > 0 && !issue_s(it)) {
            ok = false;
            break;
          }
          for (int t = 0; t < w.n_it; ++t, ++it) {
            const uint32_t q_base = sbase + stage_off(it);
            // Q and dO of this block as MN-major B operands (N = head dim,
            // K = queries): two 64-column blocks
            const uint32_t q_mn_lo = sdesc_lo(q_base, L::kBlockBytes);
            const uint32_t do_mn_lo = sdesc_lo(q_base + L::kTileBytes, L::kBlockBytes);
            if (!mbar_wait(bar(L::kBarPReady), it & 1, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // queries 16kk..16kk+15: softmax half kk/4, whose 64 columns hold
            // P^T in the first 32 and dS^T in the last 32 (two bf16 per column)
            auto p_col = [](int kk) { return (uint32_t)(64 * (kk >> 2) + 8 * (kk & 3)); };
#pragma unroll
            for (int kk = 0; kk < kQB2 / 16; ++kk)  // dV += P^T dO  (K = queries)
              umma_ts_w(tmem + L::kColDV, tmem + L::kColS + p_col(kk),
                        do_mn_lo + ((kk * 16 * 128) >> 4), kHi, kIdAcc,
                        (t > 0 || kk > 0) ? 1u : 0u);
            if (!mbar_wait(bar(L::kBarDSReady), it & 1, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kQB2 / 16; ++kk)  // dK += dS^T Q
              umma_ts_w(tmem + L::kColDK, tmem + L::kColS + p_col(kk) + 32,
                        q_mn_lo + ((kk * 16 * 128) >> 4), kHi, kIdAcc,
                        (t > 0 || kk > 0) ? 1u : 0u);
            // S^T, dP^T (done before the softmax warps published P^T / dS^T),
            // dV and dK of this block are complete: the stage can be refilled
            umma_commit(bar(L::kBarQEmpty + it % L::kStages));
            if (t + 1 < w.n_it && !issue_s(it + 1)) {
              ok = false;
              break;
            }
            // dQ^T = K^T dS^T (M = head dim, N = queries, K = keys) over the
            // dP^T columns, which the softmax warps have read (dS^T is ready)
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk) {
              const uint32_t ko = (kk * 16 * 128) >> 4;
              if (kk == 0)
                umma_ss_w<0>(tmem + L::kColDQ, kt_lo + ko, kHi, ds_lo + ko, kHi, kIdDQ);
              else
                umma_ss_w<1>(tmem + L::kColDQ, kt_lo + ko, kHi, ds_lo + ko, kHi, kIdDQ);
            }
            umma_commit(bar(L::kBarDQFull));
          }
          if (ok) {
            umma_commit(bar(L::kBarKVEmpty));
            umma_commit(bar(L::kBarDKVFull));
          }
        }
      }
      const int di = grad ? 0 : 1;
      umma_commit(bar(L::kBarDrain + di));
      drain_wait_b(bar(L::kBarDrain + di), 0);
    }
    if (lane == 0 && warp == L::kSemWarp && a.deterministic) {
      // Block by block, once the drain threads have added it (each one's
      // arrive releases at CTA scope what it added, and this wait acquires
      // it), one add with release order at GPU scope moves the block's
      // semaphore: whoever reads the new count sees the adds.  The drain warps
      // go on meanwhile; the free barrier keeps them at most one block ahead
      // of this thread.
      uint32_t it = 0;
      bool ok = true;
      for (int ri = 0, u = read_unit(0, false); ok && u >= 0; u = read_unit(++ri, false)) {
        const BwdUnit w = bwd_unit<kMod, kQB2>(a, u, group);
        const int g = w.j % a.dq_groups;
        for (int t = 0; t < w.n_it; ++t, ++it) {
          const int gi = t / w.n_blk;
          const int iq = w.lo + (t - gi * w.n_blk);
          const int bh = w.b * a.Hq + w.hk * group + gi;
          if (!mbar_wait(bar(L::kBarDQAdded), it & 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive(bar(L::kBarDQAddedFree));
          int* sem = a.sem + (size_t)g * a.sem_group_stride + (size_t)bh * a.n_qblk + iq;
          asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(sem) : "memory");
        }
      }
    }
  }
  } else if (warp < L::kSmxWarps) {
    // ------------------------------------------------------------ P^T / dS^T
    constexpr int kSC = L::kSmxCols;
    const int quarter = warp & 3;  // TMEM lanes 32*quarter.. = key rows
    const int part = warp >> 2;    // query columns 64*part..
    const int r = quarter * 32 + lane;
    const int c0 = part * kSC;
    const uint32_t t_row = tmem + ((uint32_t)(quarter * 32) << 16);
    // this thread's dS^T row in the 64-query column block of its half
    uint8_t* ds_row = smem + L::kOffDS + part * (L::kDSBytes / 2) + r * 128;
    const int wl = win_left<kMod>(a), wr = win_right<kMod>(a);
    uint32_t it = 0;
    bool ok = true;
    for (int ri = 0, u = read_unit(0, true); ok && u >= 0; u = read_unit(++ri, true)) {
      const BwdUnit w = bwd_unit<kMod, kQB2>(a, u, group);
      const int kv = w.j * kTile + r;
      const bool row_dead = kv >= w.kv_len;
      for (int t = 0; t < w.n_it; ++t, ++it) {
        const int gi = t / w.n_blk;
        const int iq = w.lo + (t - gi * w.n_blk);
        const float4* s_lse2 = reinterpret_cast<const float4*>(
            smem + stage_off(it) + 2 * L::kTileBytes + c0 * 4);
        const float4* s_delta = reinterpret_cast<const float4*>(
            smem + stage_off(it) + 2 * L::kTileBytes + L::kVecBytes + c0 * 4);
        if (!warp_wait_b(bar(L::kBarQFull + it % L::kStages), (it / L::kStages) & 1,
                         abort_flag)) {
          ok = false;
          break;
        }
        // column c is query q0 + c; it sees key kv iff c_lo <= c <= c_hi
        const int q0 = iq * kQB2 + c0;
        const int c_lo = wr >= 0 ? kv - wr - q0 : INT_MIN;
        const int c_hi = wl >= 0 ? kv + wl - q0 : INT_MAX;
        // relative-position bias slope*log2(e)*(kv - q) per column (none in
        // the plain kernel)
        const float slope2 =
            (kMod && a.alibi) ? a.alibi[w.hk * group + gi] * 1.4426950408889634f : 0.f;
        if (!warp_wait_b(bar(L::kBarSFull), it & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the warp's 64 score columns in one TMEM round trip; P^T replaces
        // them in the same registers
        float p[kSC];
        {
          uint32_t v[kSC];
          tmem_ld64(t_row + L::kColS + c0, v);
          // s * c + bias - LSE2, two columns per packed FMA (the same rounding
          // as two fmaf); no per-column mask when the whole segment is visible
          const float2 c2 = make_float2(a.scale_log2, a.scale_log2);
          const bool full = !row_dead && c_lo <= 0 && c_hi >= kSC - 1;
#pragma unroll
          for (int q = 0; q < kSC / 4; ++q) {
            const float4 l4 = s_lse2[q];
            const float lq[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
              const int c = 4 * q + e;
              const float b0 = kMod ? slope2 * (float)(kv - q0 - c) : 0.f;
              const float b1 = kMod ? slope2 * (float)(kv - q0 - c - 1) : 0.f;
              const float2 t2 = __ffma2_rn(make_float2(u2f(v[c]), u2f(v[c + 1])), c2,
                                           make_float2(b0 - lq[e], b1 - lq[e + 1]));
              const float x0 = ex2_mufu(t2.x), x1 = ex2_mufu(t2.y);
              if (full) {
                p[c] = x0;
                p[c + 1] = x1;
              } else {
                p[c] = (row_dead || c < c_lo || c > c_hi) ? 0.f : x0;
                p[c + 1] = (row_dead || c + 1 < c_lo || c + 1 > c_hi) ? 0.f : x1;
              }
            }
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t wbuf[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) wbuf[e] = pack_bf16x2(p[32 * h + 2 * e], p[32 * h + 2 * e + 1]);
          // P^T of queries 32h.. over columns c0 + 16h .. +15, S^T values this
          // thread has already read
          tmem_st16(t_row + L::kColS + c0 + 16 * h, wbuf);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        mbar_arrive(bar(L::kBarPReady));
        if (!warp_wait_b(bar(L::kBarDPFull), it & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t v[32];
          tmem_ld32(t_row + L::kColDP + c0 + 32 * h, v);
          uint32_t wbuf[16];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            // dS = P (dP - Delta), two columns per packed add and multiply (the
            // same roundings as the scalar form)
            const float4 d4 = s_delta[8 * h + q];
            const int c = 32 * h + 4 * q;
            const float2 s01 = __fmul2_rn(
                make_float2(p[c], p[c + 1]),
                __fadd2_rn(make_float2(u2f(v[4 * q]), u2f(v[4 * q + 1])), make_float2(-d4.x, -d4.y)));
            const float2 s23 = __fmul2_rn(
                make_float2(p[c + 2], p[c + 3]),
                __fadd2_rn(make_float2(u2f(v[4 * q + 2]), u2f(v[4 * q + 3])),
                           make_float2(-d4.z, -d4.w)));
            wbuf[2 * q] = pack_bf16x2(s01.x, s01.y);
            wbuf[2 * q + 1] = pack_bf16x2(s23.x, s23.y);
          }
          // dS^T over columns c0 + 32 + 16h .. +15 (their S^T values were read
          // in the P^T pass)
          tmem_st16(t_row + L::kColS + c0 + 32 + 16 * h, wbuf);
          // shared memory, 128-byte swizzle: 16-byte chunks 4h..4h+3 of this
          // key row of the half's 64-query block
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const int chunk = 4 * h + ch;
            *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (r & 7)) << 4)) =
                make_uint4(wbuf[ch * 4], wbuf[ch * 4 + 1], wbuf[ch * 4 + 2], wbuf[ch * 4 + 3]);
          }
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(L::kBarDSReady));
      }
    }
  } else {
    // ------------------------------------------------------------ dQ drain + dK/dV epilogue
    // The four drain warps run independently (no barrier among them: one
    // measured 1-3% slower): a wait that runs out ends that warp's loop, and
    // the others find the abort flag at their next wait.
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(L::kRegsDrain));
    const int r = threadIdx.x - 32 * L::kDrainWarp0;  // TMEM lane: head-dim row of dQ^T, key row of dK/dV
    const int wq = warp - L::kDrainWarp0;
    const uint32_t t_row = tmem + ((uint32_t)(wq * 32) << 16);
    uint32_t it = 0, unit = 0;
    bool ok = true;
    // Deterministic mode: block it - 1's adds, handed to the semaphore warp
    // only after block it's dQ^T has been read (or the unit's dK/dV are
    // ready), so that the arrive, which orders this thread's adds before it
    // (a release at CTA scope), does not hold the drain while they are still
    // on their way to L2.  Each thread arrives for itself; the wait on the
    // free barrier keeps the arrives one barrier phase per block.
    bool handoff_due = false;
    auto hand_off = [&]() -> bool {
      if (!handoff_due) return true;
      handoff_due = false;
      if (it > 1 && !warp_wait_b(bar(L::kBarDQAddedFree), (it - 2) & 1, abort_flag)) return false;
      mbar_arrive(bar(L::kBarDQAdded));
      return true;
    };
    for (int ri = 0, u = read_unit(0, true); ok && u >= 0; u = read_unit(++ri, true), ++unit) {
      const BwdUnit w = bwd_unit<kMod, kQB2>(a, u, group);
      for (int t = 0; t < w.n_it; ++t, ++it) {
        const int gi = t / w.n_blk;
        const int iq = w.lo + (t - gi * w.n_blk);
        const int bh = w.b * a.Hq + w.hk * group + gi;
        ok = warp_wait_b(bar(L::kBarDQFull), it & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        // Row r of dQ^T (head-dim index r, 128 queries) comes out of TMEM in one
        // round trip, and the columns go back to the dP^T issuer before any
        // add: dP^T(i+1) is written over them.  Then, for each query, the 32
        // lanes of a warp add 32 consecutive floats into the fp32 accumulator,
        // one 128-byte line per instruction.
        uint32_t v[128];
        tmem_ld128(t_row + L::kColDQ, v);
        tc_fence_before();
        mbar_arrive(bar(L::kBarDQEmpty));
        int good = hand_off() ? 1 : 0;
        int g = 0, turn = 0;
        int* sem = nullptr;
        if (a.deterministic) {
          // kv tile j adds into accumulator g = j % G after the group's tiles
          // before it in the dealing order (ascending from the block's first
          // contributor with the snake; descending from its last contributor
          // with head-major dealing), the first of them storing
          g = w.j % a.dq_groups;
          turn = a.desc
                     ? (group_last(qblk_last_contributor<kMod, kQB2>(a, iq, w.kv_len), g,
                                   a.dq_groups) -
                        w.j) / a.dq_groups
                     : (w.j - group_first(qblk_first_contributor<kQB2>(win_left<kMod>(a), iq), g,
                                          a.dq_groups)) / a.dq_groups;
          sem = a.sem + (size_t)g * a.sem_group_stride + (size_t)bh * a.n_qblk + iq;
          if (good && turn > 0) {
            // the semaphore counts the group's tiles whose adds are done
            if (lane == 0) {
              const uint64_t t0 = global_timer_ns();
              while (ld_acquire(sem) < turn) {
                if (*abort_flag || global_timer_ns() - t0 > kWaitTimeoutNs) {
                  *abort_flag = 1;
                  good = 0;
                  break;
                }
              }
            }
            good = __shfl_sync(0xffffffffu, good, 0);
            __syncwarp();
          }
        }
        float* dst = a.dq_acc + (size_t)g * a.dq_group_stride +
                     ((size_t)bh * a.Sq_pad + (size_t)iq * kQB2) * D + r;
        if (good) {
          if (a.deterministic && turn == 0) {
#pragma unroll
            for (int e = 0; e < kQB2; ++e) dst[(size_t)e * D] = u2f(v[e]);
          } else {
#pragma unroll
            for (int e = 0; e < kQB2; ++e)
              asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(dst + (size_t)e * D),
                           "f"(u2f(v[e]))
                           : "memory");
          }
        }
        if (a.deterministic && good) handoff_due = true;
        ok = good != 0;
        if (!ok) break;
      }
      if (!ok) break;
      // ---- dK, dV epilogue for key row kv
      {
        const bool ready = warp_wait_b(bar(L::kBarDKVFull), unit & 1, abort_flag);
        ok = hand_off() && ready;  // the unit's last block, it - 1
      }
      if (!ok) break;
      tc_fence_after();
      // Each thread holds one key row; to store whole 64-byte row pieces per
      // warp instruction, the four lanes of a group trade 16-byte pieces (a 4x4
      // transpose) so that lane 4k+i writes piece i of rows 4k..4k+3.
      const int grp = lane & ~3, pc = lane & 3;
      const int row0 = w.j * kTile + wq * 32 + grp;  // first key row of the lane group
      __nv_bfloat16* dk_base = reinterpret_cast<__nv_bfloat16*>(a.dk) + (size_t)w.bhk * a.Sk * D;
      __nv_bfloat16* dv_base = reinterpret_cast<__nv_bfloat16*>(a.dv) + (size_t)w.bhk * a.Sk * D;
#pragma unroll 1
      for (int pass = 0; pass < 2 * (D / 32); ++pass) {
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
        if (pass == 2 * (D / 32) - 1) {
          // every TMEM read of dK / dV is done: the accumulators are free
          tc_fence_before();
          mbar_arrive(bar(L::kBarDKVEmpty));
        }
        const float sc = is_v ? 1.f : a.scale;
        uint32_t wk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) wk[e] = pack_bf16x2(u2f(vk[2 * e]) * sc, u2f(vk[2 * e + 1]) * sc);
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {  // word wd of each 16-byte piece
          uint32_t xk[4] = {wk[wd], wk[4 + wd], wk[8 + wd], wk[12 + wd]};
          xpose4(xk, lane);
#pragma unroll
          for (int m = 0; m < 4; ++m) wk[4 * m + wd] = xk[m];
        }
        // wk[4m..4m+3] is now piece pc of row row0 + m
        __nv_bfloat16* base = is_v ? dv_base : dk_base;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          if (row0 + m < a.Sk) {
            const size_t off = (size_t)(row0 + m) * D + c * 32 + pc * 8;
            *reinterpret_cast<uint4*>(base + off) =
                make_uint4(wk[4 * m], wk[4 * m + 1], wk[4 * m + 2], wk[4 * m + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == L::kScoreWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(a.status, (int)FA_ERR_TIMEOUT);
}

// Launches the main kernel of the 128-row-block backward (D = 128).  The
// preprocess and convert kernels are the same as for the 64-row kernel.
int launch_bwd_main_q128(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const BwdArgs& a, bool mod, int grid,
                         cudaStream_t stream) {
  int dev;
  DeviceInfo info;
  if (!current_device(&dev, &info)) return FA_ERR_CUDA;
  const int smem = (int)(info.smem_optin < (size_t)kQ128MaxSmem ? info.smem_optin : kQ128MaxSmem);
  if (smem < Q128Layout::kBytes) return FA_ERR_UNSUPPORTED;
  static bool attr_done[64] = {};
  if (dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(bwd_main_q128<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess ||
        cudaFuncSetAttribute(bwd_main_q128<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return FA_ERR_CUDA;
    attr_done[dev] = true;
  }
  const auto kernel = mod ? bwd_main_q128<true> : bwd_main_q128<false>;
  // the setmaxnreg split assumes exactly kRegsLaunch registers per thread at
  // launch: a different count could leave the drain warpgroup's request
  // unserved, so such a build is refused
  static bool regs_ok[2] = {false, false};
  if (!regs_ok[mod ? 1 : 0]) {
    cudaFuncAttributes fattr;
    if (cudaFuncGetAttributes(&fattr, kernel) != cudaSuccess) return FA_ERR_CUDA;
    if (fattr.numRegs != Q128Layout::kRegsLaunch) return FA_ERR_UNSUPPORTED;
    regs_ok[mod ? 1 : 0] = true;
  }
  cudaError_t e;
  if (a.deterministic) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(Q128Layout::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, tdo, a, smem);
  } else {
    e = launch_pdl(kernel, dim3(grid), dim3(Q128Layout::kThreads), (size_t)smem, stream, tq, tk,
                   tv, tdo, a, smem);
  }
  if (e != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

}  // namespace fa

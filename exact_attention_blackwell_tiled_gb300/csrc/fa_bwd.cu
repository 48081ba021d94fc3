// fa_bwd.cu -- backward attention kernels for sm_103a.
//
// The pages give no backward mathematics; the kernels compute the textbook
// gradient of exact attention, recomputing P from the saved log-sum-exp
// (FlashAttention-4 pages, key contribution #3: tensor-memory accumulators in
// the backward pass and a restructured dQ reduction with fewer global atomic
// adds; the Limitations list's deterministic mode that serialises the
// reductions through semaphores).
//
//   1. bwd_preprocess  Delta_i = sum_d dO_id O_id and LSE*log2(e) (+inf on padded
//                      rows); clears the semaphores, the status word and (in
//                      the atomic mode) the fp32 dQ accumulator.
//   2. bwd_main        persistent over (batch, kv head, 128-row kv tile j).  K_j
//                      and V_j stay in shared memory; for every q head of the
//                      group and every 64-row query block i that can see tile j:
//                        S^T  = K_j Q_i^T                  (TMEM, rows = keys)
//                        P^T  = 2^(S^T*scale*log2e - LSE2_i) -> bf16 in TMEM
//                        dP^T = V_j dO_i^T                 (TMEM)
//                        dS^T = P^T * (dP^T - Delta_i)     -> bf16 in TMEM and smem
//                        dV_j += P^T dO_i,  dK_j += dS^T Q_i  (TMEM accumulators)
//                        dQ_i^T = K_j^T dS_i^T             (TMEM, rows = head dim)
//                      dQ_i^T goes from TMEM straight into the fp32
//                      accumulator with reduction adds: thread d adds column d
//                      of the 64 query rows, so every warp instruction covers
//                      one 128-byte line (no shared-memory staging, which would
//                      compete with the MMA operand reads for shared-memory
//                      bandwidth).  In the deterministic mode kv tile j adds
//                      into accumulator j % G (G <= 4), in kv-tile order within
//                      its group behind a per-(group, b, h, block) semaphore;
//                      the group's first contributor stores.  At the end of the
//                      unit dK_j * scale and dV_j are written as bf16.
//   3. bwd_dq_convert  dQ = scale * accumulator -> bf16 (deterministic mode: the
//                      sum of the groups' accumulators in fixed order, each
//                      group whose semaphore shows a writer).
//
// bwd_main warp roles, with n = 8 softmax warps (plain D = 128 kernel: 512
// threads, 128 registers) or n = 16 (score-modified and D = 64 kernels: 768
// threads, 80 registers):
//   warps 0..n-1  P^T / dS^T: warp w serves key rows 32*(w%4).. (its TMEM
//                 lanes) and query columns c*(w/4).. of the block, c = 4*64/n
//                 (32 or 16), so each SM sub-partition runs n/4 of them and
//                 their latencies hide behind each other's work;
//   warps n..n+3  dQ drain (one head-dim row per thread) and the dK/dV epilogue;
//   warp n+4      TMA producer: K_j, V_j per unit; Q_i, dO_i, LSE2_i, Delta_i
//                 per block into a 3-stage ring;
//   warp n+5      TMEM owner; one thread issues S^T;
//   warp n+6      one thread issues dP^T (and, at D = 64, dQ^T of the previous
//                 block behind it);
//   warp n+7      one thread issues dV, dK and dQ^T (dV and dK where warp n+6
//                 issues dQ^T).
// TMEM columns: S^T double buffer [0,64) [64,128); P^T and dS^T (bf16 pairs)
// replace it in place: query columns cp..cp+c-1 of S^T are read by the warps
// of part p, which then write their c/2 columns of P^T and c/2 of dS^T over
// them (P^T at cp, dS^T at cp+c/2), so the parts never touch each other's
// columns;
// dP^T [128,192), dQ^T [192,256), dV [256,256+D), dK [256+D,256+2D); at D = 64
// a second dP^T buffer [384,448) takes the odd blocks.
// Three issuing threads: a thread that has MMAs queued and then waits on a
// barrier only continues once the tensor core has taken those MMAs, so a lone
// issuer lets the tensor core run dry at every wait and delays its own view of
// the next event.  S^T (as soon as Q_i has landed and its S^T buffer is free),
// dP^T (as soon as the softmax warps have read the previous one: the one
// loop-carried dependency of the block sequence, so its issuer has nothing else
// queued) and the gradients (dV, dK, dQ^T as the softmax warps publish P^T and
// dS^T) wait on different events, and each one's waits are covered by the MMAs
// the others have queued.  An S^T buffer is handed back once dK of the block
// that used it is done.  The shared dS^T ring has three buffers: the softmax
// warps write buffer i%3 only after S^T(i) is complete, which the S^T issuer
// started after dK(i-2), which the gradient issuer started after dQ^T(i-3), the
// buffer's previous reader; the tensor core completes one thread's MMAs in
// order, so no separate hand-back is needed.  Where the dP^T thread issues
// dQ^T, its order is dP^T(i-1), dQ^T(i-2), dP^T(i): dP^T(i) complete, which the
// softmax warps see before they write dS^T(i), implies dQ^T(i-2) complete.  At
// D = 64 the dQ^T MMA runs with M = 128 by reading the 64-column K block twice;
// lanes 64-127 of its result are ignored.
#include <cuda_bf16.h>

#include <climits>

#include "bwd_common.cuh"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

constexpr int kQB = 64;  // query rows per backward block

// bwd_main warp roles.  The score-modified kernel (masks, bias: more softmax
// work per score) and the D = 64 kernels (half the tensor work per score) run
// 16 softmax warps of 16 query columns each, 768 threads at 80 registers; the
// plain D = 128 kernel 8 of 32 columns, 512 threads at 128 registers, which
// measured faster there.
template <bool kWide>
struct BwdRoles {
  static constexpr int kSmxWarps = kWide ? 16 : 8;  // warps 0..: P^T / dS^T
  static constexpr int kSmxCols = 4 * kQB / kSmxWarps;  // query columns per softmax warp
  static constexpr int kDrainWarp0 = kSmxWarps;    // 4 warps: dQ drain, dK/dV epilogue
  static constexpr int kTmaWarp = kDrainWarp0 + 4;
  static constexpr int kScoreWarp = kTmaWarp + 1;  // TMEM owner, S^T issuer
  static constexpr int kDPWarp = kScoreWarp + 1;   // dP^T issuer
  static constexpr int kGradWarp = kScoreWarp + 2;  // dV / dK / dQ^T issuer
  static constexpr int kThreads = 32 * (kGradWarp + 1);
  static constexpr int kSmxThreads = 32 * kSmxWarps;
  // readers of a dynamically dealt unit: every softmax and drain warp, and the
  // three issuing threads (the TMA thread takes the units)
  static constexpr int kUnitReaders = kSmxWarps + 4 + 3;
  static_assert(kSmxCols == 16 || kSmxCols == 32, "softmax warp column split");
  static_assert(kDrainWarp0 % 4 == 0, "drain warp q reads TMEM lane quarter q");
};

// ------------------------------------------------------------------ preprocess

// Each lane owns 8 consecutive elements (16 bytes) of a row, so a row takes D/8
// lanes and a warp covers 32/(D/8) rows per step; a warp works on kPreUnroll
// steps at once to keep several 16-byte loads in flight.  Row indices over all
// heads are 32-bit (the host bounds them).
constexpr int kPreUnroll = 4;

template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess(const BwdArgs a) {
  grid_dep_wait();    // O (the forward's output) must be complete
  grid_dep_launch();  // the main kernel may launch once every block runs
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerStep = 32 / kLanesPerRow;
  constexpr int kRowsPerWarp = kRowsPerStep * kPreUnroll;
  const uint32_t total_rows = (uint32_t)a.B * a.Hq * a.Sq_pad;
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLanesPerRow, seg = lane % kLanesPerRow;
  const uint32_t warps_per_block = blockDim.x / 32;
  const uint32_t nwarps = gridDim.x * warps_per_block;
  for (uint32_t g = blockIdx.x * warps_per_block + (threadIdx.x >> 5);
       (uint64_t)g * kRowsPerWarp < total_rows; g += nwarps) {
    uint4 ov[kPreUnroll], gv[kPreUnroll];
    bool real[kPreUnroll];
#pragma unroll
    for (int u = 0; u < kPreUnroll; ++u) {
      const uint32_t r = g * kRowsPerWarp + u * kRowsPerStep + sub;
      const uint32_t bh = r / (uint32_t)a.Sq_pad;
      const uint32_t i = r - bh * (uint32_t)a.Sq_pad;
      real[u] = r < total_rows && i < (uint32_t)a.Sq;
      ov[u] = gv[u] = make_uint4(0u, 0u, 0u, 0u);
      if (real[u]) {
        const size_t off = ((size_t)bh * a.Sq + i) * D + seg * 8;
        ov[u] = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.o) + off);
        gv[u] = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.dO) + off);
      }
    }
#pragma unroll
    for (int u = 0; u < kPreUnroll; ++u) {
      const uint32_t r = g * kRowsPerWarp + u * kRowsPerStep + sub;
      const uint32_t* ow = &ov[u].x;
      const uint32_t* gw = &gv[u].x;
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[e]));
        const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[e]));
        acc = fmaf(of.x, gf.x, acc);
        acc = fmaf(of.y, gf.y, acc);
      }
#pragma unroll
      for (int sft = kLanesPerRow / 2; sft > 0; sft >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, sft);
      if (r < total_rows) {
        if (seg == 0) {
          const uint32_t bh = r / (uint32_t)a.Sq_pad;
          const uint32_t i = r - bh * (uint32_t)a.Sq_pad;
          a.delta[r] = acc;
          a.lse2[r] = real[u] ? a.lse[(size_t)bh * a.Sq + i] * 1.4426950408889634f : INFINITY;
        }
        if (a.dq_groups == 1 && !a.deterministic) {
          // the atomic mode adds into a cleared accumulator; the deterministic
          // mode's first contributor of each group stores instead
          float4* dqa = reinterpret_cast<float4*>(a.dq_acc + (size_t)r * D + seg * 8);
          dqa[0] = make_float4(0.f, 0.f, 0.f, 0.f);
          dqa[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  }
  const long long nsem = (long long)a.dq_groups * a.sem_group_stride;
  for (long long s = (long long)blockIdx.x * blockDim.x + threadIdx.x; s < nsem;
       s += (long long)gridDim.x * blockDim.x)
    a.sem[s] = 0;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *a.status = 0;
    *a.unit_counter = 0;
  }
}

// ------------------------------------------------------------------ main kernel

template <int D>
struct BwdSmem {
  static constexpr int kColBlocks = D / 64;
  static constexpr int kKVBlockBytes = kTile * 128;           // 128 rows x 64 cols bf16
  static constexpr int kKVTileBytes = kTile * D * 2;
  static constexpr int kQBlockBytes = kQB * 128;              // 64 rows x 64 cols bf16
  static constexpr int kQTileBytes = kQB * D * 2;
  static constexpr int kStages = 3;
  static constexpr int kStageBytes = 2 * kQTileBytes + 1024;  // Q, dO, LSE2 + Delta (padded)
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKVTileBytes;
  static constexpr int kOffStage = kOffV + kKVTileBytes;
  // dS^T [key][64 queries], a ring of three buffers (block i uses i % 3)
  static constexpr int kDSBufs = 3;
  static constexpr int kOffDS = kOffStage + kStages * kStageBytes;
  static constexpr int kDSBytes = kTile * kQB * 2;
  static constexpr int kOffBar = kOffDS + kDSBufs * kDSBytes;
  static constexpr int kBarKVFull = 0, kBarKVEmpty = 1;
  static constexpr int kBarQFull = 2;                // kStages
  static constexpr int kBarQEmpty = 2 + kStages;     // kStages
  static constexpr int kBarSFull = 2 + 2 * kStages;  // 2
  // P^T / dS^T published, one barrier per block parity: a waiter may lag the
  // softmax warps by a block, never by two blocks of the same parity
  static constexpr int kBarPReady = kBarSFull + 2;   // 2
  // dP^T buffers: two at D = 64, which leaves the TMEM columns for a second
  // one, so that dP^T(i+1) need not wait for the softmax warps to read dP^T(i)
  static constexpr int kDPBufs = (D == 64) ? 2 : 1;
  static constexpr int kBarDPFull = kBarPReady + 2;   // kDPBufs
  static constexpr int kBarDSReady = kBarDPFull + kDPBufs;  // 2
  static constexpr int kBarDQFull = kBarDSReady + 2;
  static constexpr int kBarDQEmpty = kBarDQFull + 1;
  static constexpr int kBarDKVFull = kBarDQEmpty + 1;
  static constexpr int kBarDKVEmpty = kBarDKVFull + 1;
  static constexpr int kBarSFree = kBarDKVEmpty + 1;   // 2: S^T buffer read by dV and dK
  static constexpr int kBarDrain = kBarSFree + 2;      // 3: one per issuer
  // deterministic mode at D = 64: drain warps 0-1 hand each block they have
  // added to lane 0 of drain warp 2, which raises the block's semaphore
  static constexpr int kBarDQAdded = kBarDrain + 3;       // (D = 64 only)
  static constexpr int kBarDQAddedFree = kBarDQAdded + 1;
  // dynamic dealing: a ring of unit numbers taken by the TMA thread
  static constexpr int kURing = 8;
  static constexpr int kBarUFull = kBarDrain + 3 + (D < 128 ? 2 : 0);  // kURing
  static constexpr int kBarUEmpty = kBarUFull + kURing;  // kURing
  static constexpr int kNumBars = kBarUEmpty + kURing;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // TMEM slot, abort flag
  static constexpr int kOffURing = kOffMisc + 16;
  static constexpr int kBytes = kOffURing + 4 * kURing;
  static constexpr int kAllocBytes = kBytes + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 192, kColDV = 256,
                            kColDK = 256 + D;
  static constexpr uint32_t kColDP1 = 256 + 2 * D;  // second dP^T buffer (D = 64)
  static_assert(kDPBufs == 1 || kColDP1 + kQB <= kTmemCols, "second dP^T buffer");
  static __device__ __forceinline__ uint32_t col_dp(uint32_t it) {
    return (kDPBufs == 2 && (it & 1)) ? kColDP1 : kColDP;
  }
};

// kMod: a sliding window and / or the relative-position bias (a.alibi); the
// plain kernel applies no mask or the causal one.
template <int D, bool kMod>
__global__ void __launch_bounds__(BwdRoles<kMod || D == 64>::kThreads, 1)
    bwd_main(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
             const BwdArgs a) {
  using L = BwdSmem<D>;
  using R = BwdRoles<kMod || D == 64>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
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
    mbar_init(bar(L::kBarKVEmpty), 3);  // every issuer commits
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::kBarQFull + s), 1);
      mbar_init(bar(L::kBarQEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) mbar_init(bar(L::kBarSFull + s), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kBarPReady + s), R::kSmxThreads);
      mbar_init(bar(L::kBarDSReady + s), R::kSmxThreads);
    }
    for (int s = 0; s < L::kDPBufs; ++s) mbar_init(bar(L::kBarDPFull + s), 1);
    mbar_init(bar(L::kBarDQFull), 1);
    // the drain threads that read dQ^T: all 128, but in the deterministic mode
    // at D = 64 only drain warps 0-1, which hold its head-dim rows
    mbar_init(bar(L::kBarDQEmpty), (D < 128 && a.deterministic) ? D : 128);
    if (D < 128) {
      mbar_init(bar(L::kBarDQAdded), D);
      mbar_init(bar(L::kBarDQAddedFree), 1);
    }
    mbar_init(bar(L::kBarDKVFull), 1);
    mbar_init(bar(L::kBarDKVEmpty), 128);
    for (int s = 0; s < 2; ++s) mbar_init(bar(L::kBarSFree + s), 1);
    for (int s = 0; s < 3; ++s) mbar_init(bar(L::kBarDrain + s), 1);
    for (int s = 0; s < L::kURing; ++s) {
      mbar_init(bar(L::kBarUFull + s), 1);
      mbar_init(bar(L::kBarUEmpty + s), R::kUnitReaders);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == R::kScoreWarp) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish();
  }
  if (warp == R::kTmaWarp && lane == 0) {
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
  // The r-th unit of this CTA.  Static dealing: computed by every role alike.
  // Dynamic dealing: the TMA thread takes the next unit number from the global
  // counter and posts it in ring slot r % kURing (take_unit); the other roles
  // read it there (read_unit; warp_wide: all lanes of the warp read, lane 0
  // hands the slot back).  -1 ends the walk.
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
  auto unit_of = [&](int u) { return bwd_unit<kMod, kQB>(a, u, group); };

  if (warp == R::kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0, unit = 0;
      bool ok = true;
      // K_j and V_j of a unit, once every issuer is done with the previous ones
      auto load_kv = [&](const BwdUnit& w, uint32_t un) -> bool {
        if (!mbar_wait(bar(L::kBarKVEmpty), (un & 1) ^ 1, abort_flag)) return false;
        mbar_arrive_expect_tx(bar(L::kBarKVFull), 2 * L::kKVTileBytes);
#pragma unroll
        for (int cb = 0; cb < L::kColBlocks; ++cb) {
          tma_load_3d(sbase + L::kOffK + cb * L::kKVBlockBytes, &tm_k, bar(L::kBarKVFull),
                      cb * 64, w.j * kTile, w.bhk);
          tma_load_3d(sbase + L::kOffV + cb * L::kKVBlockBytes, &tm_v, bar(L::kBarKVFull),
                      cb * 64, w.j * kTile, w.bhk);
        }
        return true;
      };
      for (int ri = 0, u = take_unit(0); ok && u >= 0; u = take_unit(++ri), ++unit) {
        const BwdUnit w = unit_of(u);
        // The unit's first block's Q / dO go out before its K / V: its stage
        // frees up while the previous unit still holds K and V, so it has landed
        // by the time K and V can be replaced.  Later blocks follow K and V, which
        // the first S^T needs as much as Q.
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
          mbar_arrive_expect_tx(bar(L::kBarQFull + st), 2 * L::kQTileBytes + 2 * kQB * 4);
#pragma unroll
          for (int cb = 0; cb < L::kColBlocks; ++cb) {
            tma_load_3d(sdst + cb * L::kQBlockBytes, &tm_q, bar(L::kBarQFull + st), cb * 64,
                        iq * kQB, bh);
            tma_load_3d(sdst + L::kQTileBytes + cb * L::kQBlockBytes, &tm_do,
                        bar(L::kBarQFull + st), cb * 64, iq * kQB, bh);
          }
          const size_t voff = (size_t)bh * a.Sq_pad + (size_t)iq * kQB;
          bulk_load(sdst + 2 * L::kQTileBytes, a.lse2 + voff, kQB * 4, bar(L::kBarQFull + st));
          bulk_load(sdst + 2 * L::kQTileBytes + kQB * 4, a.delta + voff, kQB * 4,
                    bar(L::kBarQFull + st));
        }
        if (ok && early == w.n_it && !load_kv(w, unit)) ok = false;
      }
      if (unit > 0) drain_wait_b(bar(L::kBarKVFull), (unit - 1) & 1);
      for (uint32_t n = (it > (uint32_t)L::kStages ? it - L::kStages : 0); n < it; ++n)
        drain_wait_b(bar(L::kBarQFull + n % L::kStages), (n / L::kStages) & 1);
    }
  } else if (warp >= R::kScoreWarp) {
    // ------------------------------------------------------------ MMA issuers
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(kTile, kQB, false, false);  // S^T, dP^T
      constexpr uint32_t kIdAcc = idesc_bf16_f32(kTile, D, false, true);   // dV, dK
      constexpr uint32_t kIdDQ = idesc_bf16_f32(kTile, kQB, true, true);   // dQ^T
      // K^T as the MN-major A operand of dQ^T: the second 64-row head-dim block
      // is the second column block of K (D = 128) or, at D = 64, the first again.
      constexpr uint32_t kLboKT = (D == 128) ? (uint32_t)L::kKVBlockBytes : 0u;
      constexpr uint32_t kHi = sdesc_hi(1024);
      const int role = warp - R::kScoreWarp;  // 0: S^T, 1: dP^T, 2: gradients
      // who issues dQ^T: the gradient thread after dK, or at D = 64 the dP^T
      // thread, behind dP^T of the next block (measured: D = 64 atomic +5 to
      // +7%, its deterministic mode 0 to -3%, D = 128 -12%).  A compile-time
      // choice: testing the mode at run time in the issuing loops cost the
      // atomic mode 2-3%.
      constexpr bool dq_on_dp = (D == 64);
      uint32_t it = 0, unit = 0;
      bool ok = true;
      for (int ri = 0, u = read_unit(0, false); ok && u >= 0; u = read_unit(++ri, false), ++unit) {
        const BwdUnit w = unit_of(u);
        if (!mbar_wait(bar(L::kBarKVFull), unit & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        // dQ^T(j) = K^T dS^T(j) (M = head dim, K = keys) once the softmax warps
        // have published dS^T(j) (waited here when wait_ds) and the drain has
        // emptied the dQ^T columns of block j-1
        auto issue_dq = [&](uint32_t j, bool wait_ds) -> bool {
          if (wait_ds && !mbar_wait(bar(L::kBarDSReady + (j & 1)), (j >> 1) & 1, abort_flag))
            return false;
          if (j > 0 && !mbar_wait(bar(L::kBarDQEmpty), (j - 1) & 1, abort_flag)) return false;
          tc_fence_after();
          const uint32_t kt_lo = sdesc_lo(sbase + L::kOffK, kLboKT);
          const uint32_t dsb_lo =
              sdesc_lo(sbase + L::kOffDS, 1024) + (((j % L::kDSBufs) * L::kDSBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t ko = (kk * 16 * 128) >> 4;
            if (kk == 0)
              umma_ss_w<0>(tmem + L::kColDQ, kt_lo + ko, kHi, dsb_lo + ko, kHi, kIdDQ);
            else
              umma_ss_w<1>(tmem + L::kColDQ, kt_lo + ko, kHi, dsb_lo + ko, kHi, kIdDQ);
          }
          umma_commit(bar(L::kBarDQFull));
          return true;
        };
        if (role < 2) {
          // ---- S^T(i) = K Q_i^T or dP^T(i) = V dO_i^T, both operands K-major
          const uint32_t k_lo = sdesc_lo(sbase + L::kOffK, 16);
          const uint32_t v_lo = sdesc_lo(sbase + L::kOffV, 16);
          auto issue_kmajor = [&](uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t ka = ((kk >> 2) * L::kKVBlockBytes + (kk & 3) * 32) >> 4;
              const uint32_t kb = ((kk >> 2) * L::kQBlockBytes + (kk & 3) * 32) >> 4;
              if (kk == 0)
                umma_ss_w<0>(d_tmem, a_lo + ka, kHi, b_lo + kb, kHi, kIdS);
              else
                umma_ss_w<1>(d_tmem, a_lo + ka, kHi, b_lo + kb, kHi, kIdS);
            }
          };
          for (int t = 0; t < w.n_it; ++t, ++it) {
            const uint32_t q_base = sbase + stage_off(it);
            if (!mbar_wait(bar(L::kBarQFull + it % L::kStages), (it / L::kStages) & 1,
                           abort_flag)) {
              ok = false;
              break;
            }
            if (role == 0) {
              // the S^T buffer of block it-2 is free once its dV and dK are done
              if (it >= 2 && !mbar_wait(bar(L::kBarSFree + (it & 1)), ((it >> 1) - 1) & 1,
                                        abort_flag)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_kmajor(tmem + L::kColS + (it & 1) * kQB, k_lo, sdesc_lo(q_base, 16));
              umma_commit(bar(L::kBarSFull + (it & 1)));
            } else {
              // the dP^T buffer is free once the softmax warps have read the
              // dP^T it held before (block it - kDPBufs)
              constexpr uint32_t kNB = L::kDPBufs;
              if (it >= kNB && !mbar_wait(bar(L::kBarDSReady + ((it - kNB) & 1)),
                                          ((it - kNB) >> 1) & 1, abort_flag)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_kmajor(tmem + L::col_dp(it), v_lo, sdesc_lo(q_base + L::kQTileBytes, 16));
              umma_commit(bar(L::kBarDPFull + it % kNB));
              // dQ^T of the unit's previous block, behind dP^T of this one
              if (dq_on_dp && t > 0 && !issue_dq(it - 1, true)) {
                ok = false;
                break;
              }
            }
          }
          // the unit's last dQ^T, before K may be replaced
          if (ok && dq_on_dp && role == 1 && w.n_it > 0) ok = issue_dq(it - 1, true);
          // K and V may be replaced once both sides are done with them
          if (ok) umma_commit(bar(L::kBarKVEmpty));
        } else {
          // ---- dV += P^T dO, dK += dS^T Q (A from TMEM)
          // dV / dK accumulators are free once the previous unit's epilogue
          // has read them
          if (unit > 0 && !mbar_wait(bar(L::kBarDKVEmpty), (unit - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          for (int t = 0; t < w.n_it; ++t, ++it) {
            const uint32_t q_base = sbase + stage_off(it);
            // Q and dO of this block as MN-major B operands (K = queries)
            const uint32_t q_mn_lo = sdesc_lo(q_base, L::kQBlockBytes);
            const uint32_t do_mn_lo = sdesc_lo(q_base + L::kQTileBytes, L::kQBlockBytes);
            const uint32_t s_col = L::kColS + (it & 1) * kQB;
            if (!mbar_wait(bar(L::kBarPReady + (it & 1)), (it >> 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // query columns 16kk..16kk+15 of P^T / dS^T: softmax warp part
            // 16kk / kSC, whose columns hold P^T in the first half and dS^T in
            // the second (two bf16 per column)
            constexpr int kSC = R::kSmxCols;
            auto p_col = [&](int kk) {
              return s_col + (16 * kk / kSC) * kSC + ((16 * kk) % kSC) / 2;
            };
#pragma unroll
            for (int kk = 0; kk < kQB / 16; ++kk)  // dV += P^T dO  (K = queries)
              umma_ts_w(tmem + L::kColDV, tmem + p_col(kk),
                        do_mn_lo + ((kk * 16 * 128) >> 4), kHi, kIdAcc,
                        (t > 0 || kk > 0) ? 1u : 0u);
            if (!mbar_wait(bar(L::kBarDSReady + (it & 1)), (it >> 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kQB / 16; ++kk)  // dK += dS^T Q
              umma_ts_w(tmem + L::kColDK, tmem + p_col(kk) + kSC / 2,
                        q_mn_lo + ((kk * 16 * 128) >> 4), kHi, kIdAcc,
                        (t > 0 || kk > 0) ? 1u : 0u);
            // S^T, dP^T (done before the softmax warps published P^T / dS^T),
            // dV and dK of this block are complete: the stage and the S^T buffer
            // can be reused
            umma_commit(bar(L::kBarQEmpty + it % L::kStages));
            umma_commit(bar(L::kBarSFree + (it & 1)));
            if (!dq_on_dp && !issue_dq(it, false)) {
              ok = false;
              break;
            }
          }
          if (ok) {
            umma_commit(bar(L::kBarKVEmpty));
            umma_commit(bar(L::kBarDKVFull));
          }
        }
      }
      umma_commit(bar(L::kBarDrain + role));
      drain_wait_b(bar(L::kBarDrain + role), 0);
    }
  } else if (warp < R::kSmxWarps) {
    // ------------------------------------------------------------ P^T / dS^T
    constexpr int kSC = R::kSmxCols;
    const int quarter = warp & 3;  // TMEM lanes 32*quarter.. = key rows
    const int part = warp >> 2;    // query columns kSC*part..
    const int r = quarter * 32 + lane;
    const int c0 = part * kSC;
    const uint32_t t_row = tmem + ((uint32_t)(quarter * 32) << 16);
    uint8_t* ds_rows = smem + L::kOffDS + r * 128;
    uint32_t it = 0;
    bool ok = true;
    for (int ri = 0, u = read_unit(0, true); ok && u >= 0; u = read_unit(++ri, true)) {
      const BwdUnit w = unit_of(u);
      const int kv = w.j * kTile + r;
      const bool row_dead = kv >= w.kv_len;
      for (int t = 0; t < w.n_it; ++t, ++it) {
        const int gi = t / w.n_blk;
        const int iq = w.lo + (t - gi * w.n_blk);
        const float4* s_lse2 = reinterpret_cast<const float4*>(
            smem + stage_off(it) + 2 * L::kQTileBytes + c0 * 4);
        const float4* s_delta = s_lse2 + kQB / 4;
        if (!warp_wait_b(bar(L::kBarQFull + it % L::kStages), (it / L::kStages) & 1,
                         abort_flag)) {
          ok = false;
          break;
        }
        // this warp's LSE2 values, loaded while S^T is still being computed
        float lse[kSC];
#pragma unroll
        for (int q = 0; q < kSC / 4; ++q) {
          const float4 x = s_lse2[q];
          lse[4 * q] = x.x, lse[4 * q + 1] = x.y, lse[4 * q + 2] = x.z, lse[4 * q + 3] = x.w;
        }
        if (!warp_wait_b(bar(L::kBarSFull + (it & 1)), (it >> 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t s_col = L::kColS + (it & 1) * kQB + c0;  // this warp's S^T columns
        // column c is query q0 + c; it sees key kv iff c_lo <= c <= c_hi
        const int q0 = iq * kQB + c0;
        const int wl = win_left<kMod>(a), wr = win_right<kMod>(a);
        const int c_lo = wr >= 0 ? kv - wr - q0 : INT_MIN;
        const int c_hi = wl >= 0 ? kv + wl - q0 : INT_MAX;
        // -LSE2 plus the relative-position bias slope*log2(e)*(kv - q) per column
        // (zero bias: exactly -LSE2)
        if (kMod) {
          const float slope2 =
              a.alibi ? a.alibi[w.hk * group + gi] * 1.4426950408889634f : 0.f;
#pragma unroll
          for (int c = 0; c < kSC; ++c) lse[c] = slope2 * (float)(kv - q0 - c) - lse[c];
        } else {
#pragma unroll
          for (int c = 0; c < kSC; ++c) lse[c] = -lse[c];
        }
        float p[kSC];
        {
          uint32_t v[kSC];
          tmem_ld<kSC>(t_row + s_col, v);
          // s * c - LSE2 for two columns per packed FMA (same rounding as two fmaf)
          const float2 c2 = make_float2(a.scale_log2, a.scale_log2);
          if (!row_dead && c_lo <= 0 && c_hi >= kSC - 1) {
            // every column of this thread's segment is visible (the common case)
#pragma unroll
            for (int c = 0; c < kSC; c += 2) {
              const float2 t2 = __ffma2_rn(make_float2(u2f(v[c]), u2f(v[c + 1])), c2,
                                           make_float2(lse[c], lse[c + 1]));
              p[c] = ex2_mufu(t2.x);
              p[c + 1] = ex2_mufu(t2.y);
            }
          } else {
#pragma unroll
            for (int c = 0; c < kSC; c += 2) {
              const float2 t2 = __ffma2_rn(make_float2(u2f(v[c]), u2f(v[c + 1])), c2,
                                           make_float2(lse[c], lse[c + 1]));
              const float x0 = ex2_mufu(t2.x), x1 = ex2_mufu(t2.y);
              p[c] = (row_dead || c < c_lo || c > c_hi) ? 0.f : x0;
              p[c + 1] = (row_dead || c + 1 < c_lo || c + 1 > c_hi) ? 0.f : x1;
            }
          }
        }
        {
          uint32_t wbuf[kSC / 2];
#pragma unroll
          for (int e = 0; e < kSC / 2; ++e) wbuf[e] = pack_bf16x2(p[2 * e], p[2 * e + 1]);
          tmem_st<kSC / 2>(t_row + s_col, wbuf);  // P^T over the first half of these columns
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        mbar_arrive(bar(L::kBarPReady + (it & 1)));
        float ndl[kSC];  // -Delta
#pragma unroll
        for (int q = 0; q < kSC / 4; ++q) {
          const float4 x = s_delta[q];
          ndl[4 * q] = -x.x, ndl[4 * q + 1] = -x.y, ndl[4 * q + 2] = -x.z, ndl[4 * q + 3] = -x.w;
        }
        if (!warp_wait_b(bar(L::kBarDPFull + it % L::kDPBufs), (it / L::kDPBufs) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t wbuf[kSC / 2];
        {
          uint32_t v[kSC];
          tmem_ld<kSC>(t_row + L::col_dp(it) + c0, v);
          // dS = P (dP - Delta), two columns per packed add and multiply (the same
          // roundings as the scalar form: a - b is a + (-b) exactly)
#pragma unroll
          for (int e = 0; e < kSC / 2; ++e) {
            const float2 d = __fmul2_rn(
                make_float2(p[2 * e], p[2 * e + 1]),
                __fadd2_rn(make_float2(u2f(v[2 * e]), u2f(v[2 * e + 1])),
                           make_float2(ndl[2 * e], ndl[2 * e + 1])));
            wbuf[e] = pack_bf16x2(d.x, d.y);
          }
        }
        // dS^T over the second half of this warp's S^T columns (their S values
        // were consumed above), so the dP^T columns are free as soon as read
        tmem_st<kSC / 2>(t_row + s_col + kSC / 2, wbuf);
        // shared memory, 128-byte swizzle: [key row][64 queries]; this warp's
        // queries are the 16-byte chunks (kSC/8)*part ..
        uint8_t* ds_row = ds_rows + (it % L::kDSBufs) * L::kDSBytes;
#pragma unroll
        for (int ch = 0; ch < kSC / 8; ++ch) {
          const int chunk = part * (kSC / 8) + ch;
          *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (r & 7)) << 4)) =
              make_uint4(wbuf[ch * 4], wbuf[ch * 4 + 1], wbuf[ch * 4 + 2], wbuf[ch * 4 + 3]);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(L::kBarDSReady + (it & 1)));
      }
    }
  } else {
    // ------------------------------------------------------------ dQ drain + dK/dV epilogue
    // The four drain warps run independently (no barrier among them: one
    // measured 1-3% slower): a wait that runs out ends that warp's loop, and
    // the others find the abort flag at their next wait.
    const int r = threadIdx.x - 32 * R::kDrainWarp0;  // TMEM lane: head-dim row of dQ^T, key row of dK/dV
    const int wq = warp - R::kDrainWarp0;
    const uint32_t t_row = tmem + ((uint32_t)(wq * 32) << 16);
    uint32_t it = 0, unit = 0;
    bool ok = true;
    constexpr int kAddWarps = D / 32;  // warps whose lanes hold real head-dim rows
    // D = 64: the other two drain warps read no dQ^T; in the deterministic
    // mode lane 0 of the first of them raises the semaphores (below)
    constexpr bool kSemWarp = kAddWarps < 4;
    // Deterministic mode with the semaphore warp: block it - 1's adds are
    // handed over only once block it's dQ^T is complete (or the unit's dK/dV
    // are), so that the arrive, which orders this thread's adds before it (a
    // release at CTA scope), does not hold the drain while they are on their
    // way to L2.  The free barrier keeps the arrives one phase per block.
    bool handoff_due = false;
    auto hand_off = [&]() -> bool {
      if (!handoff_due) return true;
      handoff_due = false;
      if (it > 1 && !warp_wait_b(bar(L::kBarDQAddedFree), (it - 2) & 1, abort_flag)) return false;
      mbar_arrive(bar(L::kBarDQAdded));
      return true;
    };
    for (int ri = 0, u = read_unit(0, true); ok && u >= 0; u = read_unit(++ri, true), ++unit) {
      const BwdUnit w = unit_of(u);
      for (int t = 0; t < w.n_it; ++t, ++it) {
        const int gi = t / w.n_blk;
        const int iq = w.lo + (t - gi * w.n_blk);
        const int bh = w.b * a.Hq + w.hk * group + gi;
        if (kSemWarp && a.deterministic && wq >= kAddWarps) {
          if (wq == kAddWarps) {
            // once drain warps 0-1 have added block it (their arrives release
            // at CTA scope what each thread added, this wait acquires it), one
            // add with release order at GPU scope moves its semaphore
            int good = 1;
            if (lane == 0) {
              if (!mbar_wait(bar(L::kBarDQAdded), it & 1, abort_flag)) {
                good = 0;
              } else {
                mbar_arrive(bar(L::kBarDQAddedFree));
                int* sem = a.sem + (size_t)(w.j % a.dq_groups) * a.sem_group_stride +
                           (size_t)bh * a.n_qblk + iq;
                asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(sem) : "memory");
              }
            }
            ok = __shfl_sync(0xffffffffu, good, 0) != 0;
            if (!ok) break;
          }
          continue;
        }
        ok = warp_wait_b(bar(L::kBarDQFull), it & 1, abort_flag);
        if (ok && kSemWarp && a.deterministic) ok = hand_off();
        if (!ok) break;
        tc_fence_after();
        // Row r of dQ^T (head-dim index r, 64 queries) goes straight from TMEM
        // to the fp32 accumulator: for each query the 32 lanes of a warp add
        // 32 consecutive floats, one 128-byte line per instruction.
        int good = 1;
        if (!a.deterministic) {
          // two 32-column halves, so that only 32 values are live at a time;
          // the columns are released once the second half is read
          float* dst = a.dq_acc + ((size_t)bh * a.Sq_pad + (size_t)iq * kQB) * D + r;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t v[32];
            tmem_ld32(t_row + L::kColDQ + hf * 32, v);
            if (hf == 1) {
              tc_fence_before();
              mbar_arrive(bar(L::kBarDQEmpty));
            }
            if (r < D) {
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(
                                 dst + (size_t)(hf * 32 + e) * D),
                             "f"(u2f(v[e]))
                             : "memory");
                // D = 128: a pause after every eight adds spreads a block's
                // adds over its period; issued in one burst, they hold up the
                // shared-memory and barrier operations of the softmax warps
                // on the same SM sub-partitions (measured: +2.2% at B2 H16
                // S8192 causal, +2.5% at B4 H16 S2048; at D = 64, whose blocks
                // are shorter, the drain then falls behind: -11%)
                if (D == 128 && (e & 7) == 7) __nanosleep(16);
              }
            }
          }
        } else {
          // deterministic mode: kv tile j adds into accumulator g = j % G after
          // the group's tiles before it in the dealing order, the first of
          // them storing instead of adding: from the block's first contributor
          // up (ascending order), or from its last contributor down (each
          // head's tiles dealt highest first; causal tiles then reach a block
          // in chain order, tile j starting at block 2j)
          const int g = w.j % a.dq_groups;
          const int turn =
              a.desc ? (group_last(qblk_last_contributor<kMod, kQB>(a, iq, w.kv_len), g, a.dq_groups) -
                        w.j) / a.dq_groups
                     : (w.j - group_first(qblk_first_contributor<kQB>(win_left<kMod>(a), iq), g,
                                          a.dq_groups)) / a.dq_groups;
          float* dst = a.dq_acc + (size_t)g * a.dq_group_stride +
                       ((size_t)bh * a.Sq_pad + (size_t)iq * kQB) * D + r;
          int* sem = a.sem + (size_t)g * a.sem_group_stride + (size_t)bh * a.n_qblk + iq;
          if (wq < kAddWarps && turn > 0) {
            // the semaphore counts the group's finished adding warps (with
            // the semaphore warp: the group's finished tiles)
            if (lane == 0) {
              const uint64_t t0 = global_timer_ns();
              while (ld_acquire(sem) < turn * (kSemWarp ? 1 : kAddWarps)) {
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
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t v[32];
            tmem_ld32(t_row + L::kColDQ + hf * 32, v);
            if (hf == 1) {
              tc_fence_before();
              mbar_arrive(bar(L::kBarDQEmpty));
            }
            if (good && r < D) {
              if (turn == 0) {
#pragma unroll
                for (int e = 0; e < 32; ++e) dst[(size_t)(hf * 32 + e) * D] = u2f(v[e]);
              } else {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(
                                   dst + (size_t)(hf * 32 + e) * D),
                               "f"(u2f(v[e]))
                               : "memory");
              }
            }
          }
          if (wq < kAddWarps && good) {
            if (kSemWarp) {
              handoff_due = true;
            } else {
              // the warp barrier orders every lane's adds before lane 0's
              // release, which makes them visible before the count moves
              __syncwarp();
              if (lane == 0)
                asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(sem) : "memory");
            }
          }
        }
        ok = good != 0;
        if (!ok) break;
      }
      if (!ok) break;
      // ---- dK, dV epilogue for key row kv
      ok = warp_wait_b(bar(L::kBarDKVFull), unit & 1, abort_flag);
      if (kSemWarp && wq < kAddWarps && !hand_off()) ok = false;  // the unit's last block
      if (!ok) break;
      tc_fence_after();
      // Each thread holds one key row; to store whole 64-byte row pieces per
      // warp instruction, the four lanes of a group trade 16-byte pieces (a 4x4
      // transpose) so that lane 4k+i writes piece i of rows 4k..4k+3.
      const int grp = lane & ~3, pc = lane & 3;
      const int row0 = w.j * kTile + wq * 32 + grp;  // first key row of the lane group
      __nv_bfloat16* dk_base = reinterpret_cast<__nv_bfloat16*>(a.dk) + (size_t)w.bhk * a.Sk * D;
      __nv_bfloat16* dv_base = reinterpret_cast<__nv_bfloat16*>(a.dv) + (size_t)w.bhk * a.Sk * D;
      // 32 columns of dK, then of dV, per pass (the register budget of 768
      // threads holds one 32-column group at a time)
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
  if (warp == R::kScoreWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(a.status, (int)FA_ERR_TIMEOUT);
}

// ------------------------------------------------------------------ dQ convert

template <int D>
__global__ void __launch_bounds__(256) bwd_dq_convert(const BwdArgs a) {
  grid_dep_wait();  // every dQ reduction of the main kernel must be complete
  // 8 elements (two 16-byte loads, one 16-byte store) per thread; row indices
  // over all heads are 32-bit (the host bounds them)
  constexpr uint32_t kPerRow = D / 8;
  const uint64_t total = (uint64_t)a.B * a.Hq * a.Sq * kPerRow;
  for (uint64_t x = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; x < total;
       x += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t row = (uint32_t)(x / kPerRow);
    const uint32_t c8 = (uint32_t)(x - (uint64_t)row * kPerRow);
    const uint32_t bh = row / (uint32_t)a.Sq;
    const uint32_t i = row - bh * (uint32_t)a.Sq;
    const float* base = a.dq_acc + ((size_t)bh * a.Sq_pad + i) * D + c8 * 8;
    float4 x0 = reinterpret_cast<const float4*>(base)[0];
    float4 x1 = reinterpret_cast<const float4*>(base)[1];
    if (a.deterministic) {
      // the groups' accumulators in fixed order; a group that no kv tile
      // wrote for this query block (its semaphore, the count of warps that
      // added, is 0) holds stale memory and is skipped
      const int* sem = a.sem + (size_t)bh * a.n_qblk + i / (uint32_t)a.qblk_rows;
      if (__ldg(sem) == 0) x0 = x1 = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int g = 1; g < a.dq_groups; ++g) {
        if (__ldg(sem + (size_t)g * a.sem_group_stride) == 0) continue;
        const float4* src = reinterpret_cast<const float4*>(base + (size_t)g * a.dq_group_stride);
        const float4 y0 = src[0], y1 = src[1];
        x0.x += y0.x, x0.y += y0.y, x0.z += y0.z, x0.w += y0.w;
        x1.x += y1.x, x1.y += y1.y, x1.z += y1.z, x1.w += y1.w;
      }
    }
    uint4 w;
    w.x = pack_bf16x2(x0.x * a.scale, x0.y * a.scale);
    w.y = pack_bf16x2(x0.z * a.scale, x0.w * a.scale);
    w.z = pack_bf16x2(x1.x * a.scale, x1.y * a.scale);
    w.w = pack_bf16x2(x1.z * a.scale, x1.w * a.scale);
    reinterpret_cast<uint4*>(a.dq)[x] = w;
  }
}

std::atomic<int> g_bwd_kernel{FA_BWD_KERNEL_AUTO};

template <int D>
static int launch_bwd_d(const BwdMaps& m, const BwdArgs& a, cudaStream_t stream) {
  const CUtensorMap &tq = m.q, &tk = m.k, &tv = m.v, &tdo = m.dO;
  using L = BwdSmem<D>;
  int dev;
  DeviceInfo info;
  if (!current_device(&dev, &info)) return FA_ERR_CUDA;
  static bool attr_done[64] = {};
  if (dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(bwd_main<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::kAllocBytes) != cudaSuccess ||
        cudaFuncSetAttribute(bwd_main<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::kAllocBytes) != cudaSuccess)
      return FA_ERR_CUDA;
    attr_done[dev] = true;
  }
  const int sms = info.sm_count;
  // 1. preprocess
  {
    const long long rows = (long long)a.B * a.Hq * a.Sq_pad;
    constexpr long long kRowsPerBlock = 8LL * (32 / (D / 8)) * kPreUnroll;  // 8 warps
    long long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    if (blocks > 8LL * sms) blocks = 8LL * sms;
    if (blocks < 1) blocks = 1;
    if (launch_pdl(bwd_preprocess<D>, dim3((int)blocks), dim3(256), 0, stream, a) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  // 2. main: one CTA per SM (all resident, which the deterministic mode's
  //    in-order semaphore chain relies on)
  {
    const int grid = a.n_units < sms ? a.n_units : sms;
    // a window other than none / causal, a bias or key lengths select the
    // general kernel
    const bool mod =
        a.alibi || a.seqlens_k || !(a.wl < 0 && (a.wr < 0 || (a.wr == 0 && a.causal)));
    const auto kernel = mod ? bwd_main<D, true> : bwd_main<D, false>;
    const int threads =
        (mod || D == 64) ? BwdRoles<true>::kThreads : BwdRoles<false>::kThreads;
    record_timing(false, stream);
    if (a.qblk_rows == 128) {
      // the deterministic mode deals units from the global counter in the
      // static order: the snake's over all heads, or head-major (groups of one
      // kv head, each head's tiles highest first).  Measured against static
      // dealing: B2 H16 S8192 causal 899 -> 986 TFLOP/s, non-causal 889 -> 904,
      // B8 H16 S2048 non-causal 829 -> 850; a CTA whose unit waited on the
      // semaphore chain takes its next unit later instead of holding one dealt
      // in advance
      BwdArgs aq = a;
      aq.dyn = a.deterministic ? 1 : 0;
      aq.head_group = a.snake ? a.B * a.Hkv : 1;
      const int rc = launch_bwd_main_q128(tq, tk, tv, tdo, aq, mod, grid, stream);
      if (rc != FA_OK) return rc;
    } else if (g_bwd_kernel.load(std::memory_order_relaxed) == FA_BWD_KERNEL_PAIR &&
               bwd_pair_eligible(a, mod)) {
      const int rc = launch_bwd_main_pair(m, a, stream);
      if (rc != FA_OK) return rc;
    } else if (a.deterministic) {
      BwdArgs am = a;
      // (D = 128 deterministic calls run the 128-row kernel.)  With the snake
      // order, units come from the global counter over all heads, in the
      // snake's order (D = 64, B2 H16 S8192 causal: 369 -> 393 TFLOP/s
      // against the static snake)
      am.dyn = a.snake;
      am.head_group = a.B * a.Hkv;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(grid);
      cfg.blockDim = dim3(threads);
      cfg.dynamicSmemBytes = L::kAllocBytes;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeCooperative;
      attr[0].val.cooperative = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, tdo, am) != cudaSuccess)
        return FA_ERR_CUDA;
    } else {
      // dynamic dealing at D = 128 with the snake (measured against the static
      // snake at B2 H16 S8192 causal: 1,159 -> 1,173 TFLOP/s; at D = 64 it
      // measured 1-4% slower and stays static)
      BwdArgs am = a;
      am.dyn = (D == 128) ? a.snake : 0;
      if (launch_pdl(kernel, dim3(grid), dim3(threads), L::kAllocBytes, stream, tq, tk, tv,
                     tdo, am) != cudaSuccess)
        return FA_ERR_CUDA;
    }
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    record_timing(true, stream);
  }
  // 3. dQ convert
  int launches = 2;
  if (a.Sq > 0) {
    const long long total = (long long)a.B * a.Hq * a.Sq * (D / 8);
    long long blocks = (total + 255) / 256;
    if (blocks > 16LL * sms) blocks = 16LL * sms;
    if (launch_pdl(bwd_dq_convert<D>, dim3((int)blocks), dim3(256), 0, stream, a) !=
        cudaSuccess)
      return FA_ERR_CUDA;
    ++launches;
  }
  note_launches(launches);
  return FA_OK;
}

int launch_bwd(const BwdMaps& m, const BwdArgs& a, cudaStream_t stream) {
  if (a.D == 128) return launch_bwd_d<128>(m, a, stream);
  if (a.D == 64) return launch_bwd_d<64>(m, a, stream);
  return FA_ERR_UNSUPPORTED;
}

// ------------------------------------------------------------------ wait test hook

// One thread runs one of the kernels' bounded waits on something that may
// never happen, and writes FA_OK or FA_ERR_TIMEOUT to *status.
//   which 0: the deterministic mode's semaphore spin, on *flag reaching 1;
//   which 1: an mbarrier wait on a phase that nothing completes.
__global__ void wait_test_kernel(const int* flag, int which, int* status) {
  __shared__ uint64_t mbar;
  __shared__ int abort_word;
  if (threadIdx.x == 0) {
    abort_word = 0;
    mbar_init(smem_u32(&mbar), 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  bool ok = true;
  if (which == 0) {
    const uint64_t t0 = global_timer_ns();
    while (ld_acquire(flag) < 1) {
      if (global_timer_ns() - t0 > kWaitTimeoutNs) {
        ok = false;
        break;
      }
    }
  } else {
    ok = mbar_wait(smem_u32(&mbar), 0, &abort_word);
  }
  *status = ok ? (int)FA_OK : (int)FA_ERR_TIMEOUT;
}

int launch_wait_test(const int* flag, int which, int* status, cudaStream_t stream) {
  wait_test_kernel<<<1, 32, 0, stream>>>(flag, which, status);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  note_launches(1);
  return FA_OK;
}

}  // namespace fa

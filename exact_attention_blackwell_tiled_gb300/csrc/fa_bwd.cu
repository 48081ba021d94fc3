// fa_bwd.cu -- backward attention kernels for sm_103a.
//
// The pages give no backward mathematics; the kernels compute the textbook
// gradient of exact attention, recomputing P from the saved log-sum-exp
// (FlashAttention-4 pages, key contribution #3: tensor-memory accumulators in
// the backward pass; the dQ reduction through global atomic adds, and the
// deterministic mode of the Limitations list that serialises those reductions
// through semaphores).
//
//   1. bwd_preprocess  Delta_i = sum_d dO_id O_id, LSE*log2(e) (+inf on padded
//                      rows), clears the fp32 dQ accumulator, the semaphores and
//                      the status word.
//   2. bwd_main        persistent over (batch, kv head, 128-row kv tile j).  K_j
//                      and V_j stay in shared memory; for every q head of the
//                      group and every q tile i that can see tile j:
//                        S^T  = K_j Q_i^T              (TMEM, rows = keys)
//                        P^T  = 2^(S^T*scale*log2e - LSE2_i)   -> bf16 in TMEM
//                        dP^T = V_j dO_i^T             (TMEM)
//                        dS^T = P^T * (dP^T - Delta_i) -> bf16 in TMEM and smem
//                        dV_j += P^T dO_i,  dK_j += dS^T Q_i   (TMEM accumulators)
//                        dQ_i  = dS K_j  (TMEM) -> fp32 atomic add into the
//                                accumulator (deterministic mode: in kv-tile
//                                order behind a per-(b, h, i) semaphore)
//                      then dK_j * scale and dV_j are written as bf16.
//   3. bwd_dq_convert  dQ = scale * accumulator -> bf16.
//
// bwd_main warp roles (192 threads): warps 0-3 compute P/dS and drain dQ and
// dK/dV (thread r owns TMEM lane r); warp 4 issues TMA loads; warp 5 owns TMEM
// and issues every tcgen05.mma from one thread.
// TMEM columns: S^T/P^T [0,128), dP^T/dS^T [128,256), dV [256,256+D),
// dK [256+D,256+2D); dQ: D=64 [384,448), D=128 two 64-column halves in the
// columns P^T and dS^T leave free, [64,128) and [192,256).
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

// ------------------------------------------------------------------ preprocess

template <int D>
__global__ void bwd_preprocess(const BwdArgs a) {
  // one warp per (b, h, padded row)
  const int warps_per_block = blockDim.x / 32;
  const long long total_rows = (long long)a.B * a.Hq * a.Sq_pad;
  const int lane = threadIdx.x & 31;
  const long long gwarp = (long long)blockIdx.x * warps_per_block + (threadIdx.x >> 5);
  const long long nwarps = (long long)gridDim.x * warps_per_block;
  constexpr int kPer = D / 32;  // elements per lane
  for (long long r = gwarp; r < total_rows; r += nwarps) {
    const long long bh = r / a.Sq_pad;
    const int i = (int)(r - bh * a.Sq_pad);
    float acc = 0.f;
    if (i < a.Sq) {
      const size_t off = ((size_t)bh * a.Sq + i) * D + lane * kPer;
      const __nv_bfloat16* o = reinterpret_cast<const __nv_bfloat16*>(a.o) + off;
      const __nv_bfloat16* g = reinterpret_cast<const __nv_bfloat16*>(a.dO) + off;
#pragma unroll
      for (int e = 0; e < kPer; ++e) acc += __bfloat162float(o[e]) * __bfloat162float(g[e]);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) {
      a.delta[r] = acc;
      a.lse2[r] = (i < a.Sq) ? a.lse[bh * a.Sq + i] * 1.4426950408889634f : INFINITY;
    }
    float* dqa = a.dq_acc + (size_t)r * D + lane * kPer;
#pragma unroll
    for (int e = 0; e < kPer; ++e) dqa[e] = 0.f;
  }
  const long long nsem = (long long)a.B * a.Hq * a.n_qtiles;
  for (long long s = (long long)blockIdx.x * blockDim.x + threadIdx.x; s < nsem;
       s += (long long)gridDim.x * blockDim.x)
    a.sem[s] = 0;
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.status = 0;
}

// ------------------------------------------------------------------ main kernel

template <int D>
struct BwdLayoutSmem {
  static constexpr int kColBlocks = D / 64;
  static constexpr int kBlockBytes = kTile * 128;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ0 = kOffV + kTileBytes;  // stage s: Q at kOffQ0 + s*2*kTileBytes,
                                                     // dO right after it
  static constexpr int kOffDS = kOffQ0 + 4 * kTileBytes;  // dS^T, 128 keys x 128 queries bf16
  static constexpr int kDSBytes = kTile * kTile * 2;
  static constexpr int kOffBar = kOffDS + kDSBytes;
  static constexpr int kBarKVFull = 0;
  static constexpr int kBarKVEmpty = 1;
  static constexpr int kBarQFull = 2;   // 2 stages
  static constexpr int kBarQEmpty = 4;  // 2 stages
  static constexpr int kBarSFull = 6;
  static constexpr int kBarPReady = 7;
  static constexpr int kBarDSReady = 8;
  static constexpr int kBarDQFull = 9;
  static constexpr int kBarDQEmpty = 10;
  static constexpr int kBarDKVFull = 11;
  static constexpr int kBarDKVEmpty = 12;
  static constexpr int kBarDrain = 13;
  static constexpr int kNumBars = 14;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAllocBytes = kBytes + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  __host__ __device__ static constexpr uint32_t col_dq(int half) {
    return D == 64 ? 384u : (half == 0 ? 64u : 192u);
  }
};

// q tiles that kv tile j contributes to: [lo, n_qtiles)
__device__ __forceinline__ int bwd_q_lo(const BwdArgs& a, int j) {
  if (!a.causal) return 0;
  return (j * kTile < a.Sq) ? j : a.n_qtiles;
}

__device__ __forceinline__ bool warp_wait_b(uint32_t bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
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

template <int D>
__global__ void __launch_bounds__(192, 1)
    bwd_main(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
             const BwdArgs a) {
  using L = BwdLayoutSmem<D>;
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
    mbar_init(bar(L::kBarKVFull), 1);
    mbar_init(bar(L::kBarKVEmpty), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kBarQFull + s), 1);
      mbar_init(bar(L::kBarQEmpty + s), 1);
    }
    mbar_init(bar(L::kBarSFull), 1);
    mbar_init(bar(L::kBarPReady), 128);
    mbar_init(bar(L::kBarDSReady), 128);
    mbar_init(bar(L::kBarDQFull), 1);
    mbar_init(bar(L::kBarDQEmpty), 128);
    mbar_init(bar(L::kBarDKVFull), 1);
    mbar_init(bar(L::kBarDKVEmpty), 128);
    mbar_init(bar(L::kBarDrain), 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int group = a.Hq / a.Hkv;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0, unit = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.n_units; u += gridDim.x, ++unit) {
        const int bhk = u / a.n_ktiles;
        const int j = u - bhk * a.n_ktiles;
        const int b = bhk / a.Hkv, hk = bhk - (bhk / a.Hkv) * a.Hkv;
        if (!mbar_wait(bar(L::kBarKVEmpty), (unit & 1) ^ 1, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(L::kBarKVFull), 2 * L::kTileBytes);
#pragma unroll
        for (int cb = 0; cb < L::kColBlocks; ++cb) {
          tma_load_3d(sbase + L::kOffK + cb * L::kBlockBytes, &tm_k, bar(L::kBarKVFull), cb * 64,
                      j * kTile, bhk);
          tma_load_3d(sbase + L::kOffV + cb * L::kBlockBytes, &tm_v, bar(L::kBarKVFull), cb * 64,
                      j * kTile, bhk);
        }
        const int lo = bwd_q_lo(a, j);
        for (int gi = 0; ok && gi < group; ++gi) {
          const int bh = b * a.Hq + hk * group + gi;
          for (int i = lo; i < a.n_qtiles; ++i, ++it) {
            const uint32_t st = it & 1;
            if (!mbar_wait(bar(L::kBarQEmpty + st), ((it >> 1) & 1) ^ 1, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar(L::kBarQFull + st), 2 * L::kTileBytes);
            const uint32_t qdst = sbase + L::kOffQ0 + st * 2 * L::kTileBytes;
#pragma unroll
            for (int cb = 0; cb < L::kColBlocks; ++cb) {
              tma_load_3d(qdst + cb * L::kBlockBytes, &tm_q, bar(L::kBarQFull + st), cb * 64,
                          i * kTile, bh);
              tma_load_3d(qdst + L::kTileBytes + cb * L::kBlockBytes, &tm_do,
                          bar(L::kBarQFull + st), cb * 64, i * kTile, bh);
            }
          }
        }
      }
      if (unit > 0) drain_wait_b(bar(L::kBarKVFull), (unit - 1) & 1);
      for (uint32_t n = (it > 2 ? it - 2 : 0); n < it; ++n)
        drain_wait_b(bar(L::kBarQFull + (n & 1)), (n >> 1) & 1);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kTile, kTile, false, false);
      constexpr uint32_t kIdescAcc = idesc_bf16_f32(kTile, D, false, true);
      constexpr uint32_t kIdescDQ = idesc_bf16_f32(kTile, 64, true, true);
      uint32_t it = 0, unit = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.n_units; u += gridDim.x, ++unit) {
        const int j = u % a.n_ktiles;
        const int n_it = group * (a.n_qtiles - bwd_q_lo(a, j));
        if (unit > 0 && !mbar_wait(bar(L::kBarDKVEmpty), (unit - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        if (!mbar_wait(bar(L::kBarKVFull), unit & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t k_base = sbase + L::kOffK, v_base = sbase + L::kOffV;
        for (int t = 0; t < n_it; ++t, ++it) {
          const uint32_t st = it & 1;
          const uint32_t q_base = sbase + L::kOffQ0 + st * 2 * L::kTileBytes;
          const uint32_t do_base = q_base + L::kTileBytes;
          if (!mbar_wait(bar(L::kBarQFull + st), (it >> 1) & 1, abort_flag)) { ok = false; break; }
          // previous dQ drained (its columns overlap S^T / dP^T when D = 128)
          if (it > 0 && !mbar_wait(bar(L::kBarDQEmpty), (it - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * L::kBlockBytes + (kk & 3) * 32;
            umma_ss(tmem + L::kColS, sdesc_sw128(k_base + off, 16, 1024),
                    sdesc_sw128(q_base + off, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * L::kBlockBytes + (kk & 3) * 32;
            umma_ss(tmem + L::kColDP, sdesc_sw128(v_base + off, 16, 1024),
                    sdesc_sw128(do_base + off, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
          }
          umma_commit(bar(L::kBarSFull));
          if (!mbar_wait(bar(L::kBarPReady), it & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)  // dV += P^T dO  (K = queries)
            umma_ts(tmem + L::kColDV, tmem + L::kColS + kk * 8,
                    sdesc_sw128(do_base + kk * 16 * 128, L::kBlockBytes, 1024), kIdescAcc,
                    (t > 0 || kk > 0) ? 1u : 0u);
          if (!mbar_wait(bar(L::kBarDSReady), it & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)  // dK += dS^T Q
            umma_ts(tmem + L::kColDK, tmem + L::kColDP + kk * 8,
                    sdesc_sw128(q_base + kk * 16 * 128, L::kBlockBytes, 1024), kIdescAcc,
                    (t > 0 || kk > 0) ? 1u : 0u);
          const uint32_t ds_base = sbase + L::kOffDS;
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {  // dQ = dS K  (K = keys)
#pragma unroll
            for (int hf = 0; hf < D / 64; ++hf)
              umma_ss(tmem + L::col_dq(hf),
                      sdesc_sw128(ds_base + kk * 16 * 128, L::kBlockBytes, 1024),
                      sdesc_sw128(k_base + hf * L::kBlockBytes + kk * 16 * 128, L::kBlockBytes,
                                  1024),
                      kIdescDQ, kk > 0 ? 1u : 0u);
          }
          umma_commit(bar(L::kBarQEmpty + st));
          umma_commit(bar(L::kBarDQFull));
        }
        if (!ok) break;
        umma_commit(bar(L::kBarKVEmpty));
        umma_commit(bar(L::kBarDKVFull));
      }
      umma_commit(bar(L::kBarDrain));
      drain_wait_b(bar(L::kBarDrain), 0);
    }
  } else {
    // ------------------------------------------------------------ P / dS / drains
    const int r = threadIdx.x;  // key row of the kv tile (and q row for the dQ drain)
    const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16);
    uint32_t it = 0, unit = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < a.n_units; u += gridDim.x, ++unit) {
      const int bhk = u / a.n_ktiles;
      const int j = u - bhk * a.n_ktiles;
      const int b = bhk / a.Hkv, hk = bhk - (bhk / a.Hkv) * a.Hkv;
      const int kv = j * kTile + r;
      const int lo = bwd_q_lo(a, j);
      const int n_qt = a.n_qtiles - lo;
      const int n_it = group * n_qt;
      for (int t = 0; t < n_it; ++t, ++it) {
        const int gi = t / n_qt;
        const int i = lo + (t - gi * n_qt);
        const int bh = b * a.Hq + hk * group + gi;
        const size_t vec_off = (size_t)bh * a.Sq_pad + (size_t)i * kTile;
        // LSE2 / Delta of the 128 queries: every lane reads the same addresses
        // (broadcast through L1).
        const float4* lse4 = reinterpret_cast<const float4*>(a.lse2 + vec_off);
        const float4* del4 = reinterpret_cast<const float4*>(a.delta + vec_off);
        if (!warp_wait_b(bar(L::kBarSFull), it & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        // ---- P^T row: key kv, queries i*128 + c
        float p[kTile];
        const bool row_dead = kv >= a.Sk;
        const int causal_lim = a.causal ? kv - i * kTile : -1;  // queries c < lim are masked
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t v[32];
          tmem_ld32(t_row + L::kColS + c4 * 32, v);
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 l = __ldg(lse4 + c4 * 8 + e4);
            const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = c4 * 32 + e4 * 4 + e;
              float x = ex2_mufu(u2f(v[e4 * 4 + e]) * a.scale_log2 - lv[e]);
              if (row_dead || c < causal_lim) x = 0.f;
              p[c] = x;
            }
          }
        }
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          uint32_t w[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) w[e] = pack_bf16x2(p[c2 * 64 + 2 * e], p[c2 * 64 + 2 * e + 1]);
          tmem_st32(t_row + L::kColS + c2 * 32, w);
        }
        tc_fence_before();
        mbar_arrive(bar(L::kBarPReady));
        // ---- dS^T row = P^T * (dP^T - Delta); written packed over the dP^T
        // columns already read, and to shared memory for the dQ MMA
        uint8_t* ds_row = smem + L::kOffDS + r * 128;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t v[32];
          tmem_ld32(t_row + L::kColDP + c4 * 32, v);
          uint32_t w[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 dl = __ldg(del4 + c4 * 8 + e4);
            const int c = c4 * 32 + e4 * 4;
            const float d0 = p[c] * (u2f(v[e4 * 4]) - dl.x);
            const float d1 = p[c + 1] * (u2f(v[e4 * 4 + 1]) - dl.y);
            const float d2 = p[c + 2] * (u2f(v[e4 * 4 + 2]) - dl.z);
            const float d3 = p[c + 3] * (u2f(v[e4 * 4 + 3]) - dl.w);
            w[e4 * 2] = pack_bf16x2(d0, d1);
            w[e4 * 2 + 1] = pack_bf16x2(d2, d3);
          }
          asm volatile(
              "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
              "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(
                  t_row + L::kColDP + c4 * 16),
              "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
              "r"(w[7]), "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]),
              "r"(w[14]), "r"(w[15])
              : "memory");
          // shared memory, 128-byte swizzle: [query block][key row][64 queries]
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const int qcol = c4 * 32 + ch * 8;  // first query of this 16-byte chunk
            const int blk = qcol >> 6;
            const int chunk = (qcol & 63) >> 3;
            uint4* dst = reinterpret_cast<uint4*>(ds_row + blk * L::kBlockBytes +
                                                  ((chunk ^ (r & 7)) << 4));
            *dst = make_uint4(w[ch * 4], w[ch * 4 + 1], w[ch * 4 + 2], w[ch * 4 + 3]);
          }
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(L::kBarDSReady));
        // ---- dQ drain: thread r now owns query row i*128 + r
        if (!warp_wait_b(bar(L::kBarDQFull), it & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        int* sem = a.sem + (size_t)bh * a.n_qtiles + i;
        if (a.deterministic) {
          // Each of the 4 warps of kv tile j adds its 32 rows once tile j-1's
          // four warps have finished: the semaphore counts warps, target 4*j.
          int good = 1;
          if (lane == 0) {
            const uint64_t t0 = global_timer_ns();
            while (ld_acquire(sem) != 4 * j) {
              if (*abort_flag || global_timer_ns() - t0 > kWaitTimeoutNs) {
                *abort_flag = 1;
                good = 0;
                break;
              }
            }
          }
          good = __shfl_sync(0xffffffffu, good, 0);
          __syncwarp();
          if (!good) ok = false;
        }
        if (ok) {
          float* dst = a.dq_acc + (vec_off + r) * D;
#pragma unroll
          for (int hf = 0; hf < D / 64; ++hf) {
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
              uint32_t v[32];
              tmem_ld32(t_row + L::col_dq(hf) + c2 * 32, v);
              float4* d4 = reinterpret_cast<float4*>(dst + hf * 64 + c2 * 32);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                atomicAdd(d4 + e, make_float4(u2f(v[4 * e]), u2f(v[4 * e + 1]), u2f(v[4 * e + 2]),
                                              u2f(v[4 * e + 3])));
            }
          }
          if (a.deterministic) {
            __threadfence();
            __syncwarp();
            if (lane == 0) atomicAdd(sem, 1);
          }
        }
        tc_fence_before();
        mbar_arrive(bar(L::kBarDQEmpty));
        if (!ok) break;
      }
      if (!ok) break;
      // ---- dK, dV epilogue for key row kv
      if (!warp_wait_b(bar(L::kBarDKVFull), unit & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const bool row_ok = kv < a.Sk;
      const size_t out_off = ((size_t)bhk * a.Sk + (row_ok ? kv : 0)) * D;
      __nv_bfloat16* dk_row = reinterpret_cast<__nv_bfloat16*>(a.dk) + out_off;
      __nv_bfloat16* dv_row = reinterpret_cast<__nv_bfloat16*>(a.dv) + out_off;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t vk[32], vv[32];
        __syncwarp();  // reconverge after the per-row stores before the warp-wide loads
        if (n_it > 0) {
          tmem_ld32(t_row + L::kColDK + c * 32, vk);
          tmem_ld32(t_row + L::kColDV + c * 32, vv);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) vk[e] = vv[e] = 0u;
        }
        if (row_ok) {
          uint32_t wk[16], wv[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            wk[e] = pack_bf16x2(u2f(vk[2 * e]) * a.scale, u2f(vk[2 * e + 1]) * a.scale);
            wv[e] = pack_bf16x2(u2f(vv[2 * e]), u2f(vv[2 * e + 1]));
          }
          uint4* dk4 = reinterpret_cast<uint4*>(dk_row + c * 32);
          uint4* dv4 = reinterpret_cast<uint4*>(dv_row + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            dk4[e] = make_uint4(wk[4 * e], wk[4 * e + 1], wk[4 * e + 2], wk[4 * e + 3]);
            dv4[e] = make_uint4(wv[4 * e], wv[4 * e + 1], wv[4 * e + 2], wv[4 * e + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar(L::kBarDKVEmpty));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(a.status, (int)FA_ERR_TIMEOUT);
}

// ------------------------------------------------------------------ dQ convert

template <int D>
__global__ void bwd_dq_convert(const BwdArgs a) {
  // 8 elements per thread
  const long long total = (long long)a.B * a.Hq * a.Sq * (D / 8);
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < total;
       x += (long long)gridDim.x * blockDim.x) {
    const long long row = x / (D / 8);
    const int c8 = (int)(x - row * (D / 8));
    const long long bh = row / a.Sq;
    const int i = (int)(row - bh * a.Sq);
    const float4* src =
        reinterpret_cast<const float4*>(a.dq_acc + ((size_t)bh * a.Sq_pad + i) * D + c8 * 8);
    const float4 x0 = src[0], x1 = src[1];
    uint4 w;
    w.x = pack_bf16x2(x0.x * a.scale, x0.y * a.scale);
    w.y = pack_bf16x2(x0.z * a.scale, x0.w * a.scale);
    w.z = pack_bf16x2(x1.x * a.scale, x1.y * a.scale);
    w.w = pack_bf16x2(x1.z * a.scale, x1.w * a.scale);
    reinterpret_cast<uint4*>(a.dq)[x] = w;
  }
}

template <int D>
static int launch_bwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream) {
  using L = BwdLayoutSmem<D>;
  int dev;
  DeviceInfo info;
  if (!current_device(&dev, &info)) return FA_ERR_CUDA;
  static bool attr_done[64] = {};
  if (dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(bwd_main<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::kAllocBytes) != cudaSuccess)
      return FA_ERR_CUDA;
    attr_done[dev] = true;
  }
  const int sms = info.sm_count;
  // 1. preprocess
  {
    const long long rows = (long long)a.B * a.Hq * a.Sq_pad;
    long long blocks = (rows + 7) / 8;  // 8 warps per block
    if (blocks > 8LL * sms) blocks = 8LL * sms;
    if (blocks < 1) blocks = 1;
    bwd_preprocess<D><<<(int)blocks, 256, 0, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  }
  // 2. main: one CTA per SM (all resident, which the deterministic mode's
  //    in-order semaphore chain relies on)
  {
    const int grid = a.n_units < sms ? a.n_units : sms;
    record_timing(false, stream);
    if (a.deterministic) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(grid);
      cfg.blockDim = dim3(192);
      cfg.dynamicSmemBytes = L::kAllocBytes;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeCooperative;
      attr[0].val.cooperative = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaLaunchKernelEx(&cfg, bwd_main<D>, tq, tk, tv, tdo, a) != cudaSuccess)
        return FA_ERR_CUDA;
    } else {
      bwd_main<D><<<grid, 192, L::kAllocBytes, stream>>>(tq, tk, tv, tdo, a);
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
    bwd_dq_convert<D><<<(int)blocks, 256, 0, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    ++launches;
  }
  note_launches(launches);
  return FA_OK;
}

int launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream) {
  if (a.D == 128) return launch_bwd_d<128>(tq, tk, tv, tdo, a, stream);
  if (a.D == 64) return launch_bwd_d<64>(tq, tk, tv, tdo, a, stream);
  return FA_ERR_UNSUPPORTED;
}

}  // namespace fa

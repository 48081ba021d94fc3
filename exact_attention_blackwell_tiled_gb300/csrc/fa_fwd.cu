// fa_fwd.cu -- forward attention kernel for sm_103a.
//
// One persistent CTA per SM walks a list of (batch*head, 128-row Q tile) work
// units.  For each unit it streams the 128-row K/V tiles of the matching kv head
// and keeps the online-softmax state of its 128 query rows (FlashAttention-4
// pages: the three per-tile phases GEMM 1 -> softmax -> GEMM 2, the pipeline
// "Softmax(S_k) || GEMM 2(P_k V_k) || GEMM 1(Q K_{k+1}^T)", 128x128 tiles,
// accumulators in tensor memory, conditional rescale with threshold
// log2(256) = 8.0).
//
// Warp roles (192 threads):
//   warps 0-3  softmax: thread r owns query row r (= TMEM lane r).  Reads S from
//              TMEM, masks, updates the running max / sum, writes P (bf16) back
//              into TMEM over the S columns, rescales O in TMEM when the running
//              max moved by more than 8 (log2 units), and writes O / LSE at the
//              end of the unit.
//   warp 4     TMA producer: Q tile per unit into a 2-stage ring, K and V tiles
//              into a shared ring in the order the MMA issuer consumes them.
//   warp 5     TMEM allocator and single-thread tcgen05.mma issuer:
//              S[g%2] = Q K_g^T (SS MMA), then O += P_{g-1} V_{g-1} (TS MMA,
//              P read from TMEM), so GEMM 1 of tile g overlaps the softmax of
//              tile g-1 and GEMM 2 of tile g-1 overlaps the softmax of tile g.
//
// TMEM columns: S/P buffer 0 [0,128), S/P buffer 1 [128,256), O [256, 256+D).
// Scores are handled in base 2: t = s * scale * log2(e), P = 2^(t - m).
#include <cuda_bf16.h>

#include "exp2.cuh"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

__device__ int g_fwd_status = 0;

template <int D>
struct FwdLayout {
  static constexpr int kColBlocks = D / 64;         // 64-element (128-byte) column blocks
  static constexpr int kBlockBytes = kTile * 128;   // one 128-row x 64-col block
  static constexpr int kTileBytes = kTile * D * 2;  // a Q, K or V tile
  static constexpr int kQStages = 2;
  static constexpr int kKVStages = (D == 128) ? 4 : 8;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kQStages * kTileBytes;
  static constexpr int kOffBar = kOffKV + kKVStages * kTileBytes;
  static constexpr int kBarQFull = 0;
  static constexpr int kBarQEmpty = kBarQFull + kQStages;
  static constexpr int kBarKVFull = kBarQEmpty + kQStages;
  static constexpr int kBarKVEmpty = kBarKVFull + kKVStages;
  static constexpr int kBarSFull = kBarKVEmpty + kKVStages;  // 2
  static constexpr int kBarPFull = kBarSFull + 2;            // 2
  static constexpr int kBarO = kBarPFull + 2;                // GEMM 2 completions
  static constexpr int kBarOFree = kBarO + 1;                // epilogue done with O
  static constexpr int kBarDrain = kBarOFree + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // TMEM base slot, abort flag
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAllocBytes = kBytes + 1024;  // slack for 1024-byte alignment
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;
};

struct UnitRange {
  int first, stride, end;
};

__device__ __forceinline__ UnitRange cta_units(const FwdArgs& a) {
  UnitRange r;
  if (a.chunk > 0) {
    r.first = blockIdx.x * a.chunk;
    r.stride = 1;
    r.end = min(a.n_units, r.first + a.chunk);
  } else {
    r.first = blockIdx.x;
    r.stride = gridDim.x;
    r.end = a.n_units;
  }
  return r;
}

// Unit u -> (flat batch*head index, q tile).  Units are head-major so that the
// CTAs running at the same time share the K/V of few heads in L2.  Causal
// units alternate longest / shortest inside a head so contiguous chunks carry
// near-equal work.
__device__ __forceinline__ void unit_coords(const FwdArgs& a, int u, int& bh, int& qt) {
  const int nq = a.n_qtiles;
  bh = u / nq;
  const int r = u - bh * nq;
  qt = a.causal ? ((r & 1) ? (r >> 1) : (nq - 1 - (r >> 1))) : r;
}

__device__ __forceinline__ int unit_kv_tiles(const FwdArgs& a, int qt) {
  int kv_len = a.Sk;
  if (a.causal) kv_len = min(a.Sk, min(a.Sq, (qt + 1) * kTile));
  return (kv_len + kTile - 1) / kTile;
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

template <int D>
__global__ void __launch_bounds__(192, 1)
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
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kBarSFull + s), 1);
      mbar_init(bar(L::kBarPFull + s), 128);
    }
    mbar_init(bar(L::kBarO), 1);
    mbar_init(bar(L::kBarOFree), 128);
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const UnitRange ur = cta_units(a);
  const int group = a.Hq / a.Hkv;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t kv_it = 0, q_it = 0;
      bool ok = true;
      bool have_v = false;
      int v_bhk = 0, v_j = 0;
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
      for (int u = ur.first; ok && u < ur.end; u += ur.stride) {
        int bh, qt;
        unit_coords(a, u, bh, qt);
        const int b = bh / a.Hq, h = bh - (bh / a.Hq) * a.Hq;
        const int bhk = b * a.Hkv + h / group;
        const int n_kv = unit_kv_tiles(a, qt);
        const uint32_t qs = q_it % L::kQStages;
        if (!mbar_wait(bar(L::kBarQEmpty + qs), ((q_it / L::kQStages) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(L::kBarQFull + qs), L::kTileBytes);
#pragma unroll
        for (int cb = 0; cb < L::kColBlocks; ++cb)
          tma_load_3d(sbase + L::kOffQ + qs * L::kTileBytes + cb * L::kBlockBytes, &tm_q,
                      bar(L::kBarQFull + qs), cb * 64, qt * kTile, bh);
        ++q_it;
        for (int j = 0; j < n_kv; ++j) {
          if (!load_kv(&tm_k, bhk, j)) { ok = false; break; }
          if (have_v && !load_kv(&tm_v, v_bhk, v_j)) { ok = false; break; }
          have_v = true;
          v_bhk = bhk;
          v_j = j;
        }
      }
      if (ok && have_v) load_kv(&tm_v, v_bhk, v_j);
      // Let every issued copy land before the CTA can exit.
      for (uint32_t n = (kv_it > (uint32_t)L::kKVStages ? kv_it - L::kKVStages : 0); n < kv_it; ++n)
        drain_wait(bar(L::kBarKVFull + n % L::kKVStages), (n / L::kKVStages) & 1);
      for (uint32_t n = (q_it > (uint32_t)L::kQStages ? q_it - L::kQStages : 0); n < q_it; ++n)
        drain_wait(bar(L::kBarQFull + n % L::kQStages), (n / L::kQStages) & 1);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kTile, kTile, false, false);
      constexpr uint32_t kIdescO = idesc_bf16_f32(kTile, D, false, true);
      uint32_t kv_it = 0, q_it = 0, g = 0, tile = 0;
      bool ok = true;
      bool have_prev = false, prev_first = false;
      uint32_t prev_g = 0, prev_tile = 0;
      auto gemm2 = [&](uint32_t pg, bool first, uint32_t ptile) -> bool {
        const uint32_t sb = pg & 1;
        if (!mbar_wait(bar(L::kBarPFull + sb), (pg >> 1) & 1, abort_flag)) return false;
        if (first && ptile > 0 && !mbar_wait(bar(L::kBarOFree), (ptile - 1) & 1, abort_flag))
          return false;
        const uint32_t st = kv_it % L::kKVStages;
        if (!mbar_wait(bar(L::kBarKVFull + st), (kv_it / L::kKVStages) & 1, abort_flag))
          return false;
        tc_fence_after();
        const uint32_t v_base = sbase + L::kOffKV + st * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          // V as the MN-major B operand: 16 kv rows per step; 64-column blocks
          // of V are kBlockBytes apart.
          const uint64_t bdesc = sdesc_sw128(v_base + kk * 16 * 128, L::kBlockBytes, 1024);
          umma_ts(tmem + L::kColO, tmem + sb * 128 + kk * 8, bdesc, kIdescO,
                  (kk > 0 || !first) ? 1u : 0u);
        }
        umma_commit(bar(L::kBarKVEmpty + st));
        ++kv_it;
        umma_commit(bar(L::kBarO));
        return true;
      };
      for (int u = ur.first; ok && u < ur.end; u += ur.stride) {
        int bh, qt;
        unit_coords(a, u, bh, qt);
        const int n_kv = unit_kv_tiles(a, qt);
        const uint32_t qs = q_it % L::kQStages;
        if (!mbar_wait(bar(L::kBarQFull + qs), (q_it / L::kQStages) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t q_base = sbase + L::kOffQ + qs * L::kTileBytes;
        for (int j = 0; j < n_kv; ++j) {
          const uint32_t st = kv_it % L::kKVStages;
          if (!mbar_wait(bar(L::kBarKVFull + st), (kv_it / L::kKVStages) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t k_base = sbase + L::kOffKV + st * L::kTileBytes;
          const uint32_t sb = g & 1;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // Q and K as K-major operands: 16 head-dim columns per step.
            const uint32_t off = (kk >> 2) * L::kBlockBytes + (kk & 3) * 32;
            umma_ss(tmem + sb * 128, sdesc_sw128(q_base + off, 16, 1024),
                    sdesc_sw128(k_base + off, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
          }
          umma_commit(bar(L::kBarKVEmpty + st));
          ++kv_it;
          umma_commit(bar(L::kBarSFull + sb));
          if (j == n_kv - 1) umma_commit(bar(L::kBarQEmpty + qs));
          if (have_prev && !gemm2(prev_g, prev_first, prev_tile)) {
            ok = false;
            break;
          }
          have_prev = true;
          prev_first = (j == 0);
          prev_g = g;
          prev_tile = tile;
          ++g;
        }
        ++q_it;
        ++tile;
      }
      if (ok && have_prev) gemm2(prev_g, prev_first, prev_tile);
      // Every issued MMA must complete before TMEM is released.
      umma_commit(bar(L::kBarDrain));
      drain_wait(bar(L::kBarDrain), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int row = threadIdx.x;  // query row inside the tile == TMEM lane
    const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16);
    uint32_t g = 0, o_seen = 0;
    bool ok = true;
    for (int u = ur.first; ok && u < ur.end; u += ur.stride) {
      int bh, qt;
      unit_coords(a, u, bh, qt);
      const int n_kv = unit_kv_tiles(a, qt);
      const int q_row = qt * kTile + row;
      const int lim = a.causal ? min(a.Sk, q_row + 1) : a.Sk;  // keys [0, lim) visible
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < n_kv; ++j) {
        const uint32_t sb = g & 1;
        if (!warp_wait(bar(L::kBarSFull + sb), (g >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        float t[kTile];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(t_row + sb * 128 + c * 32, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) t[c * 32 + i] = u2f(r[i]) * a.scale_log2;
        }
        const int kv0 = j * kTile;
        if (kv0 + kTile > lim) {
#pragma unroll
          for (int c = 0; c < kTile; ++c)
            if (kv0 + c >= lim) t[c] = -INFINITY;
        }
        float tmax = t[0];
#pragma unroll
        for (int c = 1; c < kTile; ++c) tmax = fmaxf(tmax, t[c]);
        // Conditional rescale: keep a stale running max unless the new max
        // exceeds it by more than 8 (P then stays <= 2^8).
        float alpha = 1.f;
        bool rescale = false;
        if (j == 0) {
          m_run = tmax;
        } else if (tmax > m_run + 8.0f) {
          alpha = ex2_mufu(m_run - tmax);
          m_run = tmax;
          rescale = true;
        }
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        uint32_t p[kTile / 2];
        float sum = 0.f;
#pragma unroll
        for (int c = 0; c < kTile / 2; ++c) {
          const float p0 = ex2_mufu(t[2 * c] - m_use);
          const float p1 = ex2_mufu(t[2 * c + 1] - m_use);
          sum += p0 + p1;
          p[c] = pack_bf16x2(p0, p1);
        }
        l_run = l_run * alpha + sum;
        // GEMM 2 of the previous tile must be done before O is touched or the
        // next P is published (keeps one GEMM 2 phase outstanding at most).
        while (o_seen < g) {
          if (!warp_wait(bar(L::kBarO), o_seen & 1, abort_flag)) { ok = false; break; }
          ++o_seen;
        }
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(t_row + L::kColO + c * 32, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(u2f(r[i]) * alpha);
            tmem_st32(t_row + L::kColO + c * 32, r);
          }
        }
        __syncwarp();
        tmem_st32(t_row + sb * 128, *reinterpret_cast<const uint32_t(*)[32]>(&p[0]));
        tmem_st32(t_row + sb * 128 + 32, *reinterpret_cast<const uint32_t(*)[32]>(&p[32]));
        tc_fence_before();
        mbar_arrive(bar(L::kBarPFull + sb));
        ++g;
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16, LSE = ln2 * (m + log2 l)
      while (o_seen < g) {
        if (!warp_wait(bar(L::kBarO), o_seen & 1, abort_flag)) { ok = false; break; }
        ++o_seen;
      }
      if (!ok) break;
      tc_fence_after();
      const float inv_l = 1.0f / l_run;
      const bool row_ok = q_row < a.Sq;
      __nv_bfloat16* orow =
          reinterpret_cast<__nv_bfloat16*>(a.o) + ((size_t)bh * a.Sq + (row_ok ? q_row : 0)) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        __syncwarp();  // reconverge after the per-row store before the warp-wide load
        tmem_ld32(t_row + L::kColO + c * 32, r);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(u2f(r[2 * i]) * inv_l, u2f(r[2 * i + 1]) * inv_l);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (row_ok) a.lse[(size_t)bh * a.Sq + q_row] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
      tc_fence_before();
      mbar_arrive(bar(L::kBarOFree));
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

template <int D>
static int launch_fwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        FwdArgs a, cudaStream_t stream) {
  using L = FwdLayout<D>;
  int dev;
  DeviceInfo info;
  if (!current_device(&dev, &info)) return FA_ERR_CUDA;
  static bool attr_done[64] = {};
  if (dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::kAllocBytes) != cudaSuccess)
      return FA_ERR_CUDA;
    attr_done[dev] = true;
  }
  int* status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_fwd_status) != cudaSuccess)
    return FA_ERR_CUDA;
  a.status = status;
  const int sms = info.sm_count;
  int grid;
  if (a.causal) {
    // contiguous chunks of an even number of units: a long and a short q tile
    // of the same head pair up, so chunks carry near-equal work
    int chunk = (a.n_units + sms - 1) / sms;
    if (chunk > 1 && (chunk & 1)) ++chunk;
    a.chunk = chunk;
    grid = (a.n_units + chunk - 1) / chunk;
  } else {
    a.chunk = 0;
    grid = a.n_units < sms ? a.n_units : sms;
  }
  record_timing(false, stream);
  fwd_kernel<D><<<grid, 192, L::kAllocBytes, stream>>>(tq, tk, tv, a);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
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
    y[i] = which ? ex2_poly(x[i]) : ex2_mufu(x[i]);
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

// fa_merge.cu -- log-sum-exp merge of attention parts over disjoint key sets.
//
// FlashAttention-4 pages: the three phases of "The Asymmetric Hardware Scaling
// Wall on NVIDIA Blackwell" rescale a running output whenever the running max
// moves; the same identity combines whole parts.  For parts c with normalised
// output O_c and log-sum-exp LSE_c (natural log; -inf for a part that saw no
// key), per row:
//
//     M = max_c LSE_c,  LSE = M + ln sum_c e^(LSE_c - M),  O = sum_c e^(LSE_c - LSE) O_c
//
// A row whose parts are all empty gets O = 0 and LSE = -inf.  The pages name
// sequence parallelism ("Production Deployment Guide") without a mechanism;
// this merge is its one exchange step, and the split-KV forward uses it on one
// GPU.
//
// HBM-bound: per row it reads n * (4 * D + 4) bytes and writes 2 * D + 4.  One
// warp per row; the part LSEs are read lane-strided and reduced with shuffles,
// and lane l owns the D/32 contiguous elements [l * D/32, ...) of every part
// row (16-byte loads at D = 128).  With at most eight parts every part row is
// loaded together with the LSEs; with at most 32, lane c computes part c's
// weight once and the weighted part rows are loaded eight at a time, so a
// warp keeps eight independent loads in flight instead of one.
#include <cuda_bf16.h>

#include <cmath>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kMergeWarps = 8;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Lane l's D/32 elements of part c's row, scaled by w (0 for an empty part,
// whose row is not read).
template <int kV>
struct Vec {
  float e[kV];
};

template <int D>
__device__ __forceinline__ Vec<D / 32> load_part(const MergeArgs& m, int c, long long row,
                                                 int lane, bool live) {
  constexpr int kV = D / 32;
  Vec<kV> x;
#pragma unroll
  for (int e = 0; e < kV; ++e) x.e[e] = 0.f;
  if (live) {
    const float* src = m.o_part + ((size_t)c * m.rows + row) * D + lane * kV;
    if (kV == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      x.e[0] = v.x, x.e[1] = v.y, x.e[2] = v.z, x.e[3] = v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2*>(src);
      x.e[0] = v.x, x.e[1] = v.y;
    }
  }
  return x;
}

// Lane l's D/32 merged elements of a row as bf16, and the row's LSE.
template <int D>
__device__ __forceinline__ void store_row(const MergeArgs& m, long long row, int lane,
                                          const float* acc, float lse) {
  constexpr int kV = D / 32;
  __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(m.o) + (size_t)row * D + lane * kV;
  if (kV == 4) {
    const __nv_bfloat162 p0 = __floats2bfloat162_rn(acc[0], acc[1]);
    const __nv_bfloat162 p1 = __floats2bfloat162_rn(acc[2], acc[3]);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t*>(&p0);
    w.y = *reinterpret_cast<const uint32_t*>(&p1);
    *reinterpret_cast<uint2*>(dst) = w;
  } else {
    *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(acc[0], acc[1]);
  }
  if (lane == 0) m.lse[row] = lse;
}

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32, 4)
    merge_kernel(const MergeArgs m) {
  constexpr int kV = D / 32;  // elements per lane
  constexpr int kBatch = 8;   // part rows in flight per warp
  grid_dep_wait();            // the parts come from the kernel before this one
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * kMergeWarps;
  for (long long row = (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5); row < m.rows;
       row += warps) {
    if (m.n <= kBatch) {
      // up to eight parts: the part rows are loaded together with the LSEs (one
      // round trip per row instead of two); an empty part's row, which its
      // split did not write, is loaded but given no weight
      const float l0 = lane < m.n ? m.lse_part[(size_t)lane * m.rows + row] : -INFINITY;
      Vec<kV> x[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) x[u] = load_part<D>(m, u, row, lane, u < m.n);
      const float M = warp_max(l0);
      float acc[kV];
#pragma unroll
      for (int e = 0; e < kV; ++e) acc[e] = 0.f;
      float lse = -INFINITY;
      if (M != -INFINITY) {
        const float p = expf(l0 - M);  // 0 for an empty part
        const float z = warp_sum(p);
        lse = M + logf(z);
        const float wl = p / z;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const float w = __shfl_sync(0xffffffffu, wl, u);
          if (u < m.n && w != 0.f) {
#pragma unroll
            for (int e = 0; e < kV; ++e) acc[e] = fmaf(w, x[u].e[e], acc[e]);
          }
        }
      }
      store_row<D>(m, row, lane, acc, lse);
      continue;
    }
    // part LSEs, lane-strided; lane c keeps part c's (the common n <= 32 case)
    const float l0 = lane < m.n ? m.lse_part[(size_t)lane * m.rows + row] : -INFINITY;
    float M = l0;
    for (int c = lane + 32; c < m.n; c += 32) M = fmaxf(M, m.lse_part[(size_t)c * m.rows + row]);
    M = warp_max(M);
    float acc[kV];
#pragma unroll
    for (int e = 0; e < kV; ++e) acc[e] = 0.f;
    float lse = -INFINITY;
    if (M != -INFINITY) {
      float z = expf(l0 - M);  // 0 for an empty part
      for (int c = lane + 32; c < m.n; c += 32) z += expf(m.lse_part[(size_t)c * m.rows + row] - M);
      z = warp_sum(z);
      lse = M + logf(z);
      const float inv_z = 1.0f / z;
      if (m.n <= 32) {
        // weights e^(LSE_c - M) / z held by lane c; the part rows of a batch
        // are loaded together so their latencies overlap
        const float wl = expf(l0 - M) * inv_z;
        for (int c0 = 0; c0 < m.n; c0 += kBatch) {
          float w[kBatch];
          Vec<kV> x[kBatch];
#pragma unroll
          for (int u = 0; u < kBatch; ++u) {
            w[u] = __shfl_sync(0xffffffffu, wl, (c0 + u) & 31);
            if (c0 + u >= m.n) w[u] = 0.f;
            x[u] = load_part<D>(m, c0 + u, row, lane, w[u] != 0.f);
          }
#pragma unroll
          for (int u = 0; u < kBatch; ++u)
#pragma unroll
            for (int e = 0; e < kV; ++e) acc[e] = fmaf(w[u], x[u].e[e], acc[e]);
        }
      } else {
        for (int c = 0; c < m.n; ++c) {
          const float lc = m.lse_part[(size_t)c * m.rows + row];
          const float w = expf(lc - M) * inv_z;
          const Vec<kV> x = load_part<D>(m, c, row, lane, lc != -INFINITY);
#pragma unroll
          for (int e = 0; e < kV; ++e) acc[e] = fmaf(w, x.e[e], acc[e]);
        }
      }
    }
    store_row<D>(m, row, lane, acc, lse);
  }
}

}  // namespace

int launch_merge(const MergeArgs& m, int D, cudaStream_t stream) {
  if (m.rows == 0) return FA_OK;
  int dev;
  DeviceInfo info;
  if (!current_device(&dev, &info)) return FA_ERR_CUDA;
  const long long blocks = (m.rows + kMergeWarps - 1) / kMergeWarps;
  const long long cap = 16LL * info.sm_count;
  const int grid = (int)(blocks < cap ? blocks : cap);
  cudaError_t e;
  if (D == 128)
    e = launch_pdl(merge_kernel<128>, dim3(grid), dim3(kMergeWarps * 32), 0, stream, m);
  else if (D == 64)
    e = launch_pdl(merge_kernel<64>, dim3(grid), dim3(kMergeWarps * 32), 0, stream, m);
  else
    return FA_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return FA_ERR_CUDA;
  note_launches(1);
  return FA_OK;
}

}  // namespace fa

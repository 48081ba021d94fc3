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
// warp per row; lane l owns the D/32 contiguous elements [l * D/32, ...) of
// every part row (16-byte loads at D = 128), and the part LSEs are read
// lane-strided and reduced with shuffles.
#include <cuda_bf16.h>

#include <cmath>

#include "fa_internal.h"

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

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32)
    merge_kernel(const MergeArgs m) {
  constexpr int kV = D / 32;  // elements per lane
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * kMergeWarps;
  for (long long row = (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5); row < m.rows;
       row += warps) {
    float M = -INFINITY;
    for (int c = lane; c < m.n; c += 32) M = fmaxf(M, m.lse_part[(size_t)c * m.rows + row]);
    M = warp_max(M);
    float acc[kV];
#pragma unroll
    for (int e = 0; e < kV; ++e) acc[e] = 0.f;
    float lse = -INFINITY;
    if (M != -INFINITY) {
      float z = 0.f;
      for (int c = lane; c < m.n; c += 32) z += expf(m.lse_part[(size_t)c * m.rows + row] - M);
      lse = M + logf(warp_sum(z));
      for (int c = 0; c < m.n; ++c) {
        const float lc = m.lse_part[(size_t)c * m.rows + row];
        if (lc == -INFINITY) continue;  // an empty part: its O was never written
        const float w = expf(lc - lse);
        const float* src = m.o_part + ((size_t)c * m.rows + row) * D + lane * kV;
        if (kV == 4) {
          const float4 x = *reinterpret_cast<const float4*>(src);
          acc[0] = fmaf(w, x.x, acc[0]);
          acc[1] = fmaf(w, x.y, acc[1]);
          acc[2] = fmaf(w, x.z, acc[2]);
          acc[3] = fmaf(w, x.w, acc[3]);
        } else {
          const float2 x = *reinterpret_cast<const float2*>(src);
          acc[0] = fmaf(w, x.x, acc[0]);
          acc[1] = fmaf(w, x.y, acc[1]);
        }
      }
    }
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
  if (D == 128)
    merge_kernel<128><<<grid, kMergeWarps * 32, 0, stream>>>(m);
  else if (D == 64)
    merge_kernel<64><<<grid, kMergeWarps * 32, 0, stream>>>(m);
  else
    return FA_ERR_UNSUPPORTED;
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  note_launches(1);
  return FA_OK;
}

}  // namespace fa

// fa_noalloc.cu -- a backward entry point for callers that cannot allocate.
//
// fa_bwd needs a caller-provided device workspace (an fp32 dQ accumulator, the
// per-row Delta / LSE vectors, semaphores and a status word).  Some callers
// have no way to obtain one: code running where cudaMalloc is forbidden or
// unavailable (inside a custom allocator's own callbacks, in a process whose
// memory is entirely owned by another framework's pool, in plugins that may
// only touch the buffers they are handed).  fa_bwd_noalloc serves them by
// using a fixed scratch array that lives in this library's own device image,
// so the call itself allocates nothing.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes.  Every
// GPU on which the library is loaded keeps that memory until the process exits.
// Host code cannot use the array's name as a device pointer: on the host it only
// stands for the symbol.  The device address is therefore looked up once per
// device with cudaGetSymbolAddress (on the first call made with that device
// current) and cached.  The cache is not refreshed: after cudaDeviceReset the
// device's context is a new one and the cached address is stale, so these
// entry points must not be used across a reset of the device.
#include <cuda_runtime.h>

#include <mutex>

#include "fa_internal.h"

namespace fa {

// 32 MiB: the backward workspace takes about (4*D + 8) bytes per query row
// (rows counted as B * Hq * Sq rounded up to 128), so this covers about 64,000
// rows at D = 128 and about 127,000 at D = 64.
constexpr size_t kNoAllocScratchBytes = 32ull << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// Device address of g_noalloc_scratch for the current device, or nullptr.
void* scratch_address() {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace
}  // namespace fa

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const void* dO, const float* lse, void* dq, void* dk, void* dv,
                              int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal,
                              float scale, int deterministic, fa_stream_t stream) {
  const size_t need = fa_bwd_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, deterministic);
  if (need == 0) return FA_ERR_INVALID_ARG;  // the sizes themselves are invalid
  if (need > fa::kNoAllocScratchBytes) return FA_ERR_WORKSPACE;
  void* scratch = fa::scratch_address();
  if (scratch == nullptr) return FA_ERR_CUDA;
  // fa_bwd clears every part of the workspace that must start at zero (dQ
  // accumulator, semaphores, status word) before using it, so what an earlier
  // call left in the scratch does not matter.
  return fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Sq, Sk, D, causal, scale, scratch,
                fa::kNoAllocScratchBytes, deterministic, stream);
}

// The status word sits at the start of the scratch, where fa_bwd keeps it in
// any workspace; reading it is a small device-to-host copy into a local
// variable, which allocates nothing either.
extern "C" int fa_bwd_noalloc_status(fa_stream_t stream) {
  void* scratch = fa::scratch_address();
  if (scratch == nullptr) return FA_ERR_CUDA;
  return fa_bwd_status(scratch, stream);
}

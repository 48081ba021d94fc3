// fa_api.cu -- the extern "C" boundary of libfa.so: argument validation, tensor
// maps, workspace layout and dispatch to the kernels.  See include/fa.h for the
// contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include "fa_internal.h"

namespace fa {

namespace {

thread_local int t_launches = 0;
thread_local cudaEvent_t t_ev_start = nullptr;
thread_local cudaEvent_t t_ev_stop = nullptr;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape rules shared by the forward and backward entry points.
int check_shape(int B, int Hq, int Hkv, int Sq, int Sk, int D, float scale) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 0 || Sk < 1) return FA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  // TMA coordinates and element counts are 32-bit signed in the kernels.
  const long long bh = (long long)B * Hq;
  if (bh > (1LL << 30) || (long long)Sq > (1LL << 30) || (long long)Sk > (1LL << 30))
    return FA_ERR_INVALID_ARG;
  // Row indices over all heads (q rows padded to 128) are 32-bit in the kernels.
  const long long q_rows = bh * (((long long)Sq + 127) / 128 * 128);
  const long long kv_rows = (long long)B * Hkv * Sk;
  if (q_rows > INT32_MAX || kv_rows > INT32_MAX) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// A call's visibility window, relative-position bias and key lengths
// (fa_score_mod).
struct ModArgs {
  int wl, wr;
  const float* alibi;
  const int* seqlens_k;
};

ModArgs plain_mod(int causal) { return ModArgs{-1, causal ? 0 : -1, nullptr, nullptr}; }

ModArgs read_mod(const fa_score_mod* m) {
  if (!m) return plain_mod(0);
  return ModArgs{m->window_left < 0 ? -1 : m->window_left,
                 m->window_right < 0 ? -1 : m->window_right, m->alibi_slopes, m->seqlens_k};
}

// The device arrays a modification reads are 4-byte aligned.  (A row that sees
// no key is allowed: O = 0, LSE = -inf.)
int check_mod(const ModArgs& m) {
  if (m.alibi && (reinterpret_cast<uintptr_t>(m.alibi) & 3)) return FA_ERR_MISALIGNED;
  if (m.seqlens_k && (reinterpret_cast<uintptr_t>(m.seqlens_k) & 3)) return FA_ERR_MISALIGNED;
  return FA_OK;
}

// The exact causal window keeps the causal schedules (longest units first).
int is_causal(const ModArgs& m) { return (m.wl < 0 && m.wr == 0) ? 1 : 0; }

int check_device() {
  int dev;
  DeviceInfo info;
  if (!current_device(&dev, &info)) return FA_ERR_CUDA;
  if (info.cc_major != 10 || info.cc_minor != 3) return FA_ERR_UNSUPPORTED;
  // The tensor maps are encoded through the driver API, which needs a context
  // current on the calling thread.  The runtime binds its primary context to a
  // thread lazily (at the first call that needs it), so on a thread that has
  // made no such call yet -- a framework's worker thread whose allocations were
  // all served from a cache, say -- the encoder failed with
  // CUDA_ERROR_INVALID_CONTEXT.  Selecting the current device again binds it.
  if (cudaSetDevice(dev) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

}  // namespace

void note_launches(int n) { t_launches += n; }

void record_timing(bool stop, cudaStream_t stream) {
  if (!t_ev_start || !t_ev_stop) return;
  if (!stop) {
    cudaEventRecord(t_ev_start, stream);
  } else {
    cudaEventRecord(t_ev_stop, stream);
    t_ev_start = t_ev_stop = nullptr;
  }
}

bool current_device(int* dev, DeviceInfo* out) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool have[64] = {};
  int d;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (!have[d]) {
    DeviceInfo info;
    int v = 0;
    if (cudaDeviceGetAttribute(&info.sm_count, cudaDevAttrMultiProcessorCount, d) != cudaSuccess)
      return false;
    cudaDeviceGetAttribute(&info.cc_major, cudaDevAttrComputeCapabilityMajor, d);
    cudaDeviceGetAttribute(&info.cc_minor, cudaDevAttrComputeCapabilityMinor, d);
    cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
    info.smem_optin = (size_t)v;
    cache[d] = info;
    have[d] = true;
  }
  *dev = d;
  *out = cache[d];
  return true;
}

bool make_tmap_bsd(CUtensorMap* map, const void* base, int BH, int S, int D, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)S * D * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool bwd_layout(int B, int Hq, int Sq, int D, int groups, BwdLayout* L) {
  // A 256-byte header holding the status word comes first, so fa_bwd_status can
  // find it without knowing the sizes.
  const size_t nq = (size_t)((Sq + kTile - 1) / kTile);
  const size_t rows = (size_t)B * Hq * nq * kTile;
  L->off_status = 0;
  L->off_dq_acc = 256;
  L->off_delta = align256(L->off_dq_acc + (size_t)groups * rows * D * sizeof(float));
  L->off_lse2 = align256(L->off_delta + rows * sizeof(float));
  L->off_sem = align256(L->off_lse2 + rows * sizeof(float));
  L->total = align256(L->off_sem +
                      (size_t)groups * B * Hq * (2 * nq > 0 ? 2 * nq : 1) * sizeof(int));
  return true;
}

}  // namespace fa

using namespace fa;

extern "C" {

const char* fa_status_string(int s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    default: return "FA_ERR_UNKNOWN";
  }
}

int fa_last_launch_count(void) { return t_launches; }

int fa_set_bwd_kernel(int kind, int* previous) {
  if (kind != FA_BWD_KERNEL_AUTO && kind != FA_BWD_KERNEL_ONE_SM && kind != FA_BWD_KERNEL_PAIR)
    return FA_ERR_INVALID_ARG;
  const int was = fa::g_bwd_kernel.exchange(kind);
  if (previous) *previous = was;
  return FA_OK;
}

int fa_set_timing_events(void* start_event, void* stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr)) return FA_ERR_INVALID_ARG;
  t_ev_start = static_cast<cudaEvent_t>(start_event);
  t_ev_stop = static_cast<cudaEvent_t>(stop_event);
  return FA_OK;
}

}  // extern "C"

namespace fa {
namespace {

// Validation, tensor maps and the forward arguments shared by the plain and
// split entry points.  *nothing = true when Sq == 0 (valid, no work).
int fwd_setup(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
              int Hkv, int Sq, int Sk, int D, const ModArgs& m, float scale, CUtensorMap* tq,
              CUtensorMap* tk, CUtensorMap* tv, FwdArgs* a, bool* nothing) {
  *nothing = false;
  int rc = check_shape(B, Hq, Hkv, Sq, Sk, D, scale);
  if (rc) return rc;
  if ((rc = check_mod(m))) return rc;
  if (Sq == 0) {  // nothing to read or write; q, o, lse may be null
    *nothing = true;
    return FA_OK;
  }
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_MISALIGNED;
  if ((rc = check_device())) return rc;
  if (!make_tmap_bsd(tq, q, B * Hq, Sq, D) || !make_tmap_bsd(tk, k, B * Hkv, Sk, D) ||
      !make_tmap_bsd(tv, v, B * Hkv, Sk, D))
    return FA_ERR_CUDA;
  *a = FwdArgs{};
  a->o = o;
  a->lse = lse;
  a->B = B;
  a->Hq = Hq;
  a->Hkv = Hkv;
  a->Sq = Sq;
  a->Sk = Sk;
  a->causal = is_causal(m);
  a->wl = m.wl;
  a->wr = m.wr;
  a->alibi = m.alibi;
  a->seqlens_k = m.seqlens_k;
  a->scale_log2 = scale * 1.4426950408889634f;
  a->n_qtiles = (Sq + kTile - 1) / kTile;
  a->n_pairs = (a->n_qtiles + 1) / 2;
  a->n_units = B * Hq * a->n_pairs;
  a->n_split = 1;
  a->split_tiles = 0;
  return FA_OK;
}

int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int Sq, int Sk, int D, const ModArgs& m, float scale, fa_stream_t stream) {
  t_launches = 0;
  CUtensorMap tq, tk, tv;
  FwdArgs a;
  bool nothing;
  const int rc = fwd_setup(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, m, scale, &tq, &tk, &tv, &a,
                           &nothing);
  if (rc || nothing) return rc;
  return launch_fwd(tq, tk, tv, a, D, static_cast<cudaStream_t>(stream));
}

constexpr int kMaxAutoSplits = 64;
constexpr int kSplitUnitOverhead = 3;  // fixed cost of a unit, in kv tiles (Q load, epilogue)

// Split plan: the effective split count for a request and the kv tiles per
// split.  A request of 0 picks, when the units are fewer than the SMs, the
// count that minimises (waves of units) x (kv tiles per split + the fixed
// cost of a unit), ties to the smaller count.  0 on invalid sizes.
int split_plan(int B, int Hq, int Sq, int Sk, int n_req, int sms, int* tiles_per_split) {
  if (B < 1 || Hq < 1 || Sq < 0 || Sk < 1 || n_req < 0) return 0;
  const long long n_kv = ((long long)Sk + kTile - 1) / kTile;
  const long long pairs = (((long long)Sq + kTile - 1) / kTile + 1) / 2;
  const long long units = (long long)B * Hq * (pairs > 0 ? pairs : 1);
  auto effective = [&](long long n, long long* per) {
    if (n > n_kv) n = n_kv;
    if (n < 1) n = 1;
    *per = (n_kv + n - 1) / n;
    return (n_kv + *per - 1) / *per;  // no empty split
  };
  long long per = 0, n = 0;
  if (n_req > 0) {
    n = effective(n_req, &per);
  } else {
    if (sms < 1) return 0;
    n = effective(1, &per);
    if (units < sms) {
      long long best = -1;
      for (long long c = 1; c <= kMaxAutoSplits && c <= n_kv; ++c) {
        long long pc;
        const long long nc = effective(c, &pc);
        const long long waves = (nc * units + sms - 1) / sms;
        const long long cost = waves * (pc + kSplitUnitOverhead);
        if (best < 0 || cost < best) {
          best = cost;
          n = nc;
          per = pc;
        }
      }
    }
  }
  if (tiles_per_split) *tiles_per_split = (int)per;
  return (int)n;
}

int current_sm_count() {
  int dev;
  DeviceInfo info;
  if (!current_device(&dev, &info)) return 0;
  return info.sm_count;
}

// fp32 parts of O [n, rows, D], then (256-byte aligned) of LSE [n, rows].
size_t split_o_bytes(int n, long long rows, int D) {
  return ((size_t)n * (size_t)rows * D * sizeof(float) + 255) & ~(size_t)255;
}
size_t split_ws_bytes(int n, long long rows, int D) {
  return split_o_bytes(n, rows, D) + (size_t)n * (size_t)rows * sizeof(float);
}

}  // namespace
}  // namespace fa

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
           int Hkv, int Sq, int Sk, int D, int causal, float scale, fa_stream_t stream) {
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, plain_mod(causal), scale, stream);
}

int fa_fwd_mod(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
               int Hkv, int Sq, int Sk, int D, const fa_score_mod* mod, float scale,
               fa_stream_t stream) {
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, read_mod(mod), scale, stream);
}

int fa_fwd_status(fa_stream_t stream) { return fwd_status_take(static_cast<cudaStream_t>(stream)); }

int fa_fwd_split_count(int B, int Hq, int Sq, int Sk, int sm_count) {
  const int sms = sm_count > 0 ? sm_count : current_sm_count();
  return split_plan(B, Hq, Sq, Sk, 0, sms, nullptr);
}

size_t fa_fwd_split_workspace_bytes(int B, int Hq, int Sq, int Sk, int D, int n_splits) {
  if (D != 64 && D != 128) return 0;
  const int n = split_plan(B, Hq, Sq, Sk, n_splits, n_splits == 0 ? current_sm_count() : 1,
                           nullptr);
  if (n <= 1) return 0;
  return split_ws_bytes(n, (long long)B * Hq * Sq, D);
}

int fa_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                 int Hkv, int Sq, int Sk, int D, const fa_score_mod* mod, float scale,
                 int n_splits, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  t_launches = 0;
  if (n_splits < 0) return FA_ERR_INVALID_ARG;
  const ModArgs m = read_mod(mod);
  CUtensorMap tq, tk, tv;
  FwdArgs a;
  bool nothing;
  int rc = fwd_setup(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, m, scale, &tq, &tk, &tv, &a,
                     &nothing);
  if (rc || nothing) return rc;
  int per = 0;
  const int n = split_plan(B, Hq, Sq, Sk, n_splits, n_splits == 0 ? current_sm_count() : 1, &per);
  if (n < 1) return FA_ERR_INVALID_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (n == 1) return launch_fwd(tq, tk, tv, a, D, st);
  const long long rows = (long long)B * Hq * Sq;
  if (!workspace || !aligned16(workspace) || workspace_bytes < split_ws_bytes(n, rows, D))
    return FA_ERR_WORKSPACE;
  if ((long long)B * Hq * a.n_pairs * n > INT32_MAX) return FA_ERR_INVALID_ARG;
  a.n_split = n;
  a.split_tiles = per;
  a.n_units = B * Hq * a.n_pairs * n;
  a.o_part = static_cast<float*>(workspace);
  a.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + split_o_bytes(n, rows, D));
  if ((rc = launch_fwd(tq, tk, tv, a, D, st))) return rc;
  MergeArgs mg{a.o_part, a.lse_part, n, rows, o, lse};
  return launch_merge(mg, D, st);
}

int fa_lse_merge(const float* o_parts, const float* lse_parts, int n_parts, void* o, float* lse,
                 int64_t rows, int D, fa_stream_t stream) {
  t_launches = 0;
  if (n_parts < 1 || rows < 0) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (rows == 0) return FA_OK;
  if (!o_parts || !lse_parts || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(o_parts) || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse_parts) & 3) ||
      (reinterpret_cast<uintptr_t>(lse) & 3))
    return FA_ERR_MISALIGNED;
  int rc;
  if ((rc = check_device())) return rc;
  MergeArgs mg{o_parts, lse_parts, n_parts, (long long)rows, o, lse};
  return launch_merge(mg, D, static_cast<cudaStream_t>(stream));
}

size_t fa_bwd_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D, int deterministic) {
  if (check_shape(B, Hq, Hkv, Sq, Sk, D, 1.0f) != FA_OK) return 0;
  BwdLayout L;
  bwd_layout(B, Hq, Sq, D, dq_group_count(Sk, deterministic), &L);
  return L.total;
}

}  // extern "C"

namespace fa {
namespace {

int bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dO,
             const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq,
             int Sk, int D, const ModArgs& m, float scale, void* workspace,
             size_t workspace_bytes, int deterministic, fa_stream_t stream) {
  t_launches = 0;
  int rc = check_shape(B, Hq, Hkv, Sq, Sk, D, scale);
  if (rc) return rc;
  if ((rc = check_mod(m))) return rc;
  // With Sq == 0 the query-side tensors are empty and may be null; dk and dv
  // are still written (as zeros).
  const bool has_q = Sq > 0;
  if (!k || !v || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (has_q && (!q || !o || !dO || !lse || !dq)) return FA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_MISALIGNED;
  if (has_q && (!aligned16(q) || !aligned16(o) || !aligned16(dO) || !aligned16(lse) ||
                !aligned16(dq)))
    return FA_ERR_MISALIGNED;
  BwdLayout L;
  const int groups = dq_group_count(Sk, deterministic);
  bwd_layout(B, Hq, Sq, D, groups, &L);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < L.total)
    return FA_ERR_WORKSPACE;
  if ((rc = check_device())) return rc;
  BwdMaps maps;
  // Sq == 0 still needs dk = dv = 0: the kernels handle it with zero q tiles.
  // With no q tiles the q / dO maps are never used; they are built over k.
  const void* q_map = has_q ? q : k;
  const void* do_map = has_q ? dO : k;
  const int bh_map = has_q ? B * Hq : B * Hkv;
  const int sq_map = has_q ? Sq : Sk;
  // q and dO move in blocks of bwd_qblk_rows rows in the backward pass
  const int qrows = bwd_qblk_rows(D, deterministic);
  if (!make_tmap_bsd(&maps.q, q_map, bh_map, sq_map, D, qrows) ||
      !make_tmap_bsd(&maps.k, k, B * Hkv, Sk, D) || !make_tmap_bsd(&maps.v, v, B * Hkv, Sk, D) ||
      !make_tmap_bsd(&maps.dO, do_map, bh_map, sq_map, D, qrows) ||
      !make_tmap_bsd(&maps.q_half, q_map, bh_map, sq_map, D, 32) ||
      !make_tmap_bsd(&maps.dO_half, do_map, bh_map, sq_map, D, 32))
    return FA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  BwdArgs a{};
  a.o = o;
  a.dO = dO;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dq_acc = reinterpret_cast<float*>(ws + L.off_dq_acc);
  a.delta = reinterpret_cast<float*>(ws + L.off_delta);
  a.lse2 = reinterpret_cast<float*>(ws + L.off_lse2);
  a.sem = reinterpret_cast<int*>(ws + L.off_sem);
  a.status = reinterpret_cast<int*>(ws + L.off_status);
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Sq = Sq;
  a.Sk = Sk;
  a.D = D;
  a.n_qtiles = (Sq + kTile - 1) / kTile;
  a.n_qblk = (Sq + 63) / 64;
  a.Sq_pad = a.n_qtiles * kTile;
  a.n_ktiles = (Sk + kTile - 1) / kTile;
  a.n_units = B * Hkv * a.n_ktiles;
  a.causal = is_causal(m);
  a.wl = m.wl;
  a.wr = m.wr;
  a.alibi = has_q ? m.alibi : nullptr;
  a.seqlens_k = has_q ? m.seqlens_k : nullptr;  // with no queries dK = dV = 0 anyway
  // causal: longest-first snake over all heads.  Also when q and dO exceed L2:
  // measured on GB300 against head-major dealing at B2 H16 S8192 (q, dO 128
  // MiB), the main kernel ran 1,011 -> 1,189 TFLOP/s with atomic dQ and
  // 594 -> 664 in the deterministic mode
  a.snake = a.causal ? 1 : 0;
  a.deterministic = deterministic ? 1 : 0;
  // Head-major dealing (non-causal and windowed calls) with the deterministic
  // mode: each head's tiles are dealt highest first and the chain adds a
  // block's contributions in that order.  The snake keeps ascending order and
  // an ascending chain: reversed, it would deal the shortest units first and
  // leave a tail.
  a.desc = (a.deterministic && !a.snake) ? 1 : 0;
  a.unit_counter = reinterpret_cast<int*>(ws + L.off_status + 128);  // header, own line
  {
    // kv heads per group of the dynamic dealing: q, dO (bf16) and the dQ
    // accumulators (fp32, one per group) of the kv head's q heads, plus K, V
    const double per_kv_head = (double)(Hq / Hkv) * Sq * D * (4.0 + 4.0 * groups) +
                               (double)Sk * D * 4.0;
    int hg = (int)(kBwdGroupBytes / (per_kv_head > 1.0 ? per_kv_head : 1.0));
    if (hg > B * Hkv) hg = B * Hkv;
    a.head_group = hg < 1 ? 1 : hg;
  }
  a.dq_groups = groups;
  a.dq_group_stride = (size_t)B * Hq * a.Sq_pad * D;
  a.sem_group_stride = B * Hq * a.n_qblk;
  a.qblk_rows = qrows;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  return launch_bwd(maps, a, static_cast<cudaStream_t>(stream));
}

}  // namespace
}  // namespace fa

extern "C" {

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
           const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq,
           int Sk, int D, int causal, float scale, void* workspace, size_t workspace_bytes,
           int deterministic, fa_stream_t stream) {
  return bwd_impl(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Sq, Sk, D, plain_mod(causal),
                  scale, workspace, workspace_bytes, deterministic, stream);
}

int fa_bwd_mod(const void* q, const void* k, const void* v, const void* o, const void* dO,
               const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq,
               int Sk, int D, const fa_score_mod* mod, float scale, void* workspace,
               size_t workspace_bytes, int deterministic, fa_stream_t stream) {
  return bwd_impl(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Sq, Sk, D, read_mod(mod), scale,
                  workspace, workspace_bytes, deterministic, stream);
}

int fa_bwd_status(const void* workspace, fa_stream_t stream) {
  if (!workspace) return FA_ERR_WORKSPACE;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FA_ERR_CUDA;
  return v == 0 ? FA_OK : v;
}

int fa_wait_test(const int* flag, int which, int* status, fa_stream_t stream) {
  t_launches = 0;
  if (which < 0 || which > 1 || !status || (which == 0 && !flag)) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(status) & 3) || (flag && (reinterpret_cast<uintptr_t>(flag) & 3)))
    return FA_ERR_MISALIGNED;
  int rc = check_device();
  if (rc) return rc;
  return launch_wait_test(flag, which, status, static_cast<cudaStream_t>(stream));
}

int fa_exp2_test(const float* x, float* y, int64_t n, int which, fa_stream_t stream) {
  t_launches = 0;
  if (n < 0 || which < 0 || which > 2) return FA_ERR_INVALID_ARG;
  if (n > 0 && (!x || !y)) return FA_ERR_INVALID_ARG;
  if (n == 0) return FA_OK;
  int rc = check_device();
  if (rc) return rc;
  return launch_exp2_test(x, y, n, which, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

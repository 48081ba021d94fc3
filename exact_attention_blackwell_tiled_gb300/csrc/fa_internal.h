// fa_internal.h -- declarations shared by the host-side translation units of
// libfa.so (argument structs, per-device cache, kernel launchers).
#pragma once

#include <atomic>

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "fa.h"

namespace fa {

constexpr int kTile = 128;  // rows of a Q tile and of a K/V tile

struct DeviceInfo {
  int sm_count = 0;
  int cc_major = 0;
  int cc_minor = 0;
  size_t smem_optin = 0;
};

// Cached attributes of the current device; false if no device is usable.
bool current_device(int* dev, DeviceInfo* info);

// Encodes a 3-D tensor map over a [BH, S, D] bf16 tensor with box_rows-row x
// 64-column boxes and the 128-byte swizzle.  Returns false on failure.
bool make_tmap_bsd(CUtensorMap* map, const void* base, int BH, int S, int D,
                   int box_rows = kTile);

struct FwdArgs {
  void* o;
  float* lse;
  int* status;
  int B, Hq, Hkv, Sq, Sk;
  int causal;
  // visibility: key j is seen by query i iff (wl < 0 || j >= i - wl) and
  // (wr < 0 || j <= i + wr); causal is wl = -1, wr = 0
  int wl, wr;
  const float* alibi;  // [Hq] slopes of the relative-position bias, or null
  // [B] keys per batch (key padding mask: keys j >= seqlens_k[b] are hidden;
  // clamped to [0, Sk]), or null
  const int* seqlens_k;
  float scale_log2;  // scale * log2(e)
  int n_qtiles;
  int n_pairs;  // pairs of 128-row query tiles, the forward's unit of work
  int n_units;
  int sched;  // 0: round robin over head-major units; 2: longest-first snake
              // over all heads (causal); 3: split-KV, units (head, split, pair)
              // round robin
  int chunk;  // unused (0)
  // split-KV: split s holds kv tiles [s * split_tiles, (s + 1) * split_tiles);
  // each (query tile, split) writes its own normalised O and LSE to the parts
  int n_split;
  int split_tiles;
  float* o_part;    // [n_split, B * Hq, Sq, D]
  float* lse_part;  // [n_split, B * Hq, Sq], natural log, -inf: no visible key
};

int launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const FwdArgs& a, int D, cudaStream_t stream);

// The D = 64 forward with a ring of score buffers per query tile, for no mask or
// the causal one, a positive scale and no split (mode 0 of the forward: no
// window, bias or key counts).  `a` comes filled in by the forward's launcher
// (schedule, status pointer); `grid` CTAs.
bool fwd_ring64_eligible(const FwdArgs& a, int D, int mode);
int launch_fwd_ring64(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const FwdArgs& a, int grid, cudaStream_t stream);


// Log-sum-exp merge of n attention parts over disjoint key sets.
struct MergeArgs {
  const float* o_part;    // [n, rows, D] fp32, normalised per part
  const float* lse_part;  // [n, rows], natural log, -inf = empty part
  int n;
  long long rows;
  void* o;     // [rows, D] bf16
  float* lse;  // [rows]
};
int launch_merge(const MergeArgs& m, int D, cudaStream_t stream);
int fwd_status_take(cudaStream_t stream);
int launch_exp2_test(const float* x, float* y, int64_t n, int which, cudaStream_t stream);
int launch_wait_test(const int* flag, int which, int* status, cudaStream_t stream);

struct BwdArgs {
  const void* o;
  const void* dO;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  float* dq_acc;   // dq_groups x [B, Hq, Sq_pad, D]
  float* delta;    // [B, Hq, Sq_pad]
  float* lse2;     // [B, Hq, Sq_pad]
  int* sem;        // dq_groups x [B, Hq, n_qblk]
  int* status;     // [1]
  int B, Hq, Hkv, Sq, Sk, D;
  int Sq_pad;
  int causal;
  // visibility window, relative-position bias and key lengths, as in FwdArgs
  int wl, wr;
  const float* alibi;
  const int* seqlens_k;
  int deterministic;
  float scale;
  float scale_log2;
  int n_qtiles;  // 128-row tiles of Sq
  int n_qblk;    // 64-row query blocks of Sq (the backward's q step)
  int n_ktiles;  // 128-row kv tiles of Sk
  int n_units;
  int snake;     // 1: units dealt longest-first (ascending kv tile) in a snake
  int desc;      // 1: each head's kv tiles dealt in descending order (deterministic mode)
  // Dynamic dealing (bwd_main with the snake order): a CTA takes its next unit
  // from an atomic counter, in an order that runs over groups of head_group kv
  // heads, each group's longest units (lowest kv tile) first, so that the
  // q / dO / dQ-accumulator lines of the heads in flight stay in L2
  int dyn;
  int head_group;
  int* unit_counter;  // in the workspace header; cleared by the preprocess kernel
  // dQ accumulators: 1 in the atomic mode; in the deterministic mode kv tile j
  // adds into accumulator j % dq_groups, chained only behind tile j - dq_groups
  int dq_groups;
  size_t dq_group_stride;  // floats from one accumulator to the next
  int sem_group_stride;    // semaphores from one group to the next
  int qblk_rows;           // query rows per block of the main kernel (64 or 128):
                           // semaphore i of a head counts the writers of block i
};

constexpr int kDetGroups = 4;       // deterministic-mode accumulators (at most)
// L2 bytes the backward's dynamic dealing gives one group of kv heads (their
// q, dO and dQ accumulators and K / V): about two groups are in flight at once
constexpr double kBwdGroupBytes = 96.0 * (1 << 20);
constexpr int kDetGroupsLong = 2;   // ... from kDetLongTiles kv tiles on
constexpr int kDetLongTiles = 32;

// Accumulators of a backward call: 1 atomic, else min(G, kv tiles) with G = 4,
// or 2 from 32 kv tiles on.  Measured on GB300 (main kernel + the convert that
// sums the accumulators): at B2 H16 S8192 (64 kv tiles) 1 / 2 / 4 / 8 groups
// took 1.95 / 1.92 / 2.08 / 1.94 ms of main kernel, the convert growing with
// the count; at B4 H16 S2048 (16 tiles) 0.31 / 0.30 / 0.26 / 0.24 ms, where 4
// gives the shortest total.
inline int dq_group_count(int Sk, int deterministic) {
  const int n_ktiles = (Sk + kTile - 1) / kTile;
  if (!deterministic) return 1;
  const int g = n_ktiles >= kDetLongTiles ? kDetGroupsLong : kDetGroups;
  return n_ktiles < g ? (n_ktiles > 0 ? n_ktiles : 1) : g;
}

struct BwdLayout {
  size_t off_dq_acc, off_delta, off_lse2, off_sem, off_status, total;
};
bool bwd_layout(int B, int Hq, int Sq, int D, int groups, BwdLayout* L);

// Tensor maps of a backward call: q and dO in boxes of bwd_qblk_rows rows, k
// and v in 128-row boxes, and q_half / dO_half in 32-row boxes (the CTA-pair
// kernel: each CTA of a pair reads its 32 queries of a 64-row block).
struct BwdMaps {
  CUtensorMap q, k, v, dO, q_half, dO_half;
};

int launch_bwd(const BwdMaps& m, const BwdArgs& a, cudaStream_t stream);

// The CTA-pair main kernel (D = 128, atomic dQ, no score modification), and
// the process-wide kernel choice fa_set_bwd_kernel sets.
extern std::atomic<int> g_bwd_kernel;
bool bwd_pair_eligible(const BwdArgs& a, bool mod);
int launch_bwd_main_pair(const BwdMaps& m, const BwdArgs& a, cudaStream_t stream);

// The backward's query rows per block: 128 (bwd_main_q128) for the
// deterministic mode at D = 128, 64 (bwd_main) otherwise.  The q and dO tensor
// maps use boxes of this many rows.  Measured on GB300: with atomic dQ adds
// both kernels are bound by the fp32 reduction traffic into L2 (4.4 GB per
// backward at B2 H16 S8192 causal, 3.4-3.6 TB/s either way), where the 64-row
// kernel's adds interfere less with its softmax warps; the deterministic mode,
// which stores a quarter of its contributions, runs 1.2-1.45x faster with
// 128-row blocks.
inline int bwd_qblk_rows(int D, int deterministic) {
  return (D == 128 && deterministic) ? 128 : 64;
}

// Main kernel of the 128-row-block backward (D = 128 only).
int launch_bwd_main_q128(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const BwdArgs& a, bool mod, int grid,
                         cudaStream_t stream);

void note_launches(int n);

// Launch with programmatic stream serialisation: the kernel may be scheduled
// while the previous kernel in the stream is still running, so it must call
// grid_dep_wait before touching memory that kernel may write.
template <typename Kernel, typename... Args>
inline cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Events requested by fa_set_timing_events for the next main-kernel launch on
// this thread; record_timing(true/false) records start/stop and clears after stop.
void record_timing(bool stop, cudaStream_t stream);

}  // namespace fa

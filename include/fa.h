/*
 * fa.h -- C ABI of the GB300 (sm_103a) fused exact-attention library libfa.so.
 *
 * The operation is exact scaled-dot-product attention as the FlashAttention-4
 * pages state it (blog page "FlashAttention-4 Guide", section "The Asymmetric
 * Hardware Scaling Wall on NVIDIA Blackwell": GEMM 1  S = QK^T * scale, the
 * softmax  P = exp(S - m)/l,  GEMM 2  O = PV; the simulator's signature in
 * "End-to-End Implementation" takes q, k, v, a causal flag and a scale).  The
 * log-sum-exp output and the backward pass are the plain mathematics of that
 * definition:
 *
 *   s_ij = scale * q_i . k_j   (causal: only j <= i, top-left)
 *   LSE_i = ln sum_j exp(s_ij),  P_ij = exp(s_ij - LSE_i),  O_i = sum_j P_ij v_j
 *   dV_j = sum_i P_ij dO_i,  dS_ij = P_ij (dO_i . v_j - dO_i . O_i),
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i
 *
 * Layout: every tensor is dense row-major [B, H, S, D] (the simulator's
 * docstring layout); H = Hq for q, o, dO, dq and H = Hkv for k, v, dk, dv.
 * q/k/v/o/dO/dq/dk/dv are bf16 (raw 16-bit storage), lse is fp32 [B, Hq, Sq] in
 * natural log.  Grouped heads: Hq % Hkv == 0 and q head h reads kv head
 * floor(h * Hkv / Hq).  D must be 64 or 128.
 *
 * Ownership: the caller owns every buffer (all device pointers), including the
 * backward workspace.  The library never allocates device memory; it keeps a
 * small host-side cache of per-device attributes.  All calls are asynchronous
 * on `stream` (0 = legacy default stream); results are valid after the stream
 * is synchronised.
 *
 * Threads: any host thread may call, on the device current for that thread
 * (the runtime's cudaGetDevice).  Each call makes that device's primary context
 * current on the calling thread before it builds its tensor maps, so a thread
 * that has made no CUDA call of its own yet is served as well.
 *
 * Errors: arguments are validated on the host before anything is launched; on
 * a validation error nothing is written and a status code is returned.  Launch
 * failures return FA_ERR_CUDA.  Device-side waits carry an iteration/time cap;
 * one that runs out records FA_ERR_TIMEOUT in a status word and the kernel
 * returns early (fa_fwd_status / fa_bwd_status report it).
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, Hq % Hkv != 0, non-finite scale,
                             or more than 2^31 - 1 rows over all heads (B * Hq * Sq with Sq
                             rounded up to 128, or B * Hkv * Sk) */
  FA_ERR_UNSUPPORTED = 2, /* head dimension other than 64 / 128, or a device that is not sm_103 */
  FA_ERR_MISALIGNED = 3,  /* a tensor pointer not 16-byte aligned (TMA requirement) */
  FA_ERR_WORKSPACE = 4,   /* backward workspace missing, misaligned or too small */
  FA_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed */
  FA_ERR_TIMEOUT = 6      /* a device-side wait ran out (reported by the status calls) */
} fa_status;

/* An opaque CUDA stream (cudaStream_t). */
typedef void* fa_stream_t;

/*
 * Forward pass: o = softmax(scale * q k^T [causal]) v and lse.
 *   q   [B, Hq,  Sq, D] bf16      k, v [B, Hkv, Sk, D] bf16
 *   o   [B, Hq,  Sq, D] bf16 out  lse  [B, Hq, Sq] fp32 out (natural log)
 * Sizes: B, Hq, Hkv, Sk >= 1; Sq >= 0 (Sq == 0 is a no-op); D in {64, 128};
 * B * Hq * Sq (Sq rounded up to 128) and B * Hkv * Sk below 2^31; scale finite.  causal != 0 applies the top-left mask q_idx >= kv_idx, which
 * leaves no row empty when Sk >= 1.  Pointers must be non-null and 16-byte
 * aligned (when Sq == 0 nothing is checked, read or written).  Output rows are
 * written exactly once; nothing outside them is touched.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
           int Hkv, int Sq, int Sk, int D, int causal, float scale, fa_stream_t stream);

/*
 * Score modification: a sliding-window mask, a key padding mask and a linear
 * relative-position bias (FlashAttention-4 pages, "CuTe-DSL Implementation and
 * Rapid JIT Compilation": the FlexAttention integration's score modifications,
 * relative position biases and custom masks, which the pages name without
 * defining).  Key kv_idx of batch b is visible to query q_idx iff
 *   (window_left  < 0 || kv_idx >= q_idx - window_left) &&
 *   (window_right < 0 || kv_idx <= q_idx + window_right) &&
 *   (seqlens_k == NULL || kv_idx < seqlens_k[b]),
 * so {-1, 0, NULL} is fa_fwd's causal mask and {-1, -1, NULL} no mask.
 * seqlens_k is null or a device array of B int32 key counts (4-byte aligned,
 * else FA_ERR_MISALIGNED; each clamped to [0, Sk]).  The keys past a batch's
 * count are still read from k and v (with weight 0), so they must hold finite
 * values.  A query row that sees no key gets O = 0 and LSE = -inf, and the
 * backward gives it dQ = 0; keys no row sees get dK = dV = 0.
 * alibi_slopes is null or a device array of Hq fp32 slopes (4-byte aligned,
 * else FA_ERR_MISALIGNED); the score of (q_idx, kv_idx) in query head h becomes
 * scale * q.k + alibi_slopes[h] * (kv_idx - q_idx).  Neither array is read when
 * Sq == 0.
 */
typedef struct {
  int window_left;
  int window_right;
  const float* alibi_slopes;
  const int* seqlens_k;
} fa_score_mod;

/*
 * fa_fwd with a score modification; mod == NULL is fa_fwd without the causal
 * mask.  Same tensors, sizes, pointer rules and errors as fa_fwd.
 */
int fa_fwd_mod(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
               int Hkv, int Sq, int Sk, int D, const fa_score_mod* mod, float scale,
               fa_stream_t stream);

/*
 * Synchronises `stream`, returns FA_OK or FA_ERR_TIMEOUT if any forward launch on
 * this device since the previous call recorded a timed-out wait, and clears the
 * record.  FA_ERR_CUDA if the synchronisation itself fails.
 */
int fa_fwd_status(fa_stream_t stream);

/*
 * Bytes of device workspace fa_bwd needs for these sizes (0 on bad sizes).  The
 * workspace holds fp32 dQ accumulators [B, Hq, ceil(Sq/128)*128, D] (one in the
 * atomic mode; in the deterministic mode G = min(4, ceil(Sk/128)), or
 * min(2, ceil(Sk/128)) from 32 kv tiles (Sk > 3968) on, kv tile j adding into
 * accumulator j % G in its own ordered chain, the accumulators summed in fixed
 * order at the end), the per-row dot products D_i = dO_i . O_i and
 * LSE*log2(e) (fp32 [B, Hq, padded Sq]), the deterministic mode's per-(group,
 * b, h, query block) semaphores and a status word.  The deterministic
 * size is at least the atomic one.  It needs no initialisation: fa_bwd clears
 * or overwrites what it uses.
 */
size_t fa_bwd_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D, int deterministic);

/*
 * Backward pass: dq, dk, dv of L with dL/dO = dO, given the forward's o and lse.
 *   q, o, dO, dq [B, Hq, Sq, D] bf16;  k, v, dk, dv [B, Hkv, Sk, D] bf16;
 *   lse [B, Hq, Sq] fp32 (natural log, as written by fa_fwd).
 * dq, dk, dv are overwritten (not accumulated); dk and dv sum over the q heads
 * of a group.  workspace: device memory of at least
 * fa_bwd_workspace_bytes(...) bytes, 256-byte aligned.  deterministic != 0
 * serialises the dQ accumulation in a fixed kv-tile order through semaphores,
 * so repeated runs give identical bits; otherwise dQ partials are added with
 * fp32 atomics (the last bits may differ between runs).  Same size and
 * pointer rules as fa_fwd, except that Sq == 0 is not a no-op: dk and dv are
 * then zero (q, o, dO, lse and dq may be null).
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
           const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq,
           int Sk, int D, int causal, float scale, void* workspace, size_t workspace_bytes,
           int deterministic, fa_stream_t stream);

/*
 * fa_bwd with a score modification (see fa_score_mod); o and lse must come from
 * fa_fwd_mod with the same modification.  mod == NULL is fa_bwd without the
 * causal mask.  Same tensors, workspace, sizes, pointer rules and errors as
 * fa_bwd.
 */
int fa_bwd_mod(const void* q, const void* k, const void* v, const void* o, const void* dO,
               const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq,
               int Sk, int D, const fa_score_mod* mod, float scale, void* workspace,
               size_t workspace_bytes, int deterministic, fa_stream_t stream);

/*
 * Synchronises `stream` and returns the status the last fa_bwd recorded in
 * `workspace` (FA_OK or FA_ERR_TIMEOUT); FA_ERR_CUDA if the sync fails.
 */
int fa_bwd_status(const void* workspace, fa_stream_t stream);

/*
 * Backward main kernel for the calls it applies to: head dim 128, atomic dQ
 * (deterministic == 0) and no score modification beyond the causal mask.
 *   FA_BWD_KERNEL_AUTO (0, the default): the one-SM kernel.
 *   FA_BWD_KERNEL_ONE_SM (1): one CTA per kv tile (128 keys), 64-query blocks.
 *   FA_BWD_KERNEL_PAIR (2): clusters of two CTAs on kv tile pairs (256 keys),
 *     every product in the 2-CTA MMA mode, the dQ reduction over 256 keys
 *     before the global fp32 adds (half the adds of the one-SM kernel).
 *     FlashAttention-4 pages, key contribution #3.  Measured slower than the
 *     one-SM kernel on GB300, hence not the default.
 * Other calls ignore the setting.  Process-wide; takes effect at the next
 * fa_bwd / fa_bwd_mod / fa_bwd_noalloc launch.  Writes the previous setting to
 * *previous unless it is null.  Returns FA_OK, or FA_ERR_INVALID_ARG (and
 * changes nothing) for another value of kind.
 */
#define FA_BWD_KERNEL_AUTO 0
#define FA_BWD_KERNEL_ONE_SM 1
#define FA_BWD_KERNEL_PAIR 2
int fa_set_bwd_kernel(int kind, int* previous);

/*
 * Split-KV forward: the kv tiles (128 keys each) are cut into n contiguous
 * splits, every (128-row query tile, split) is an independent unit of work, and
 * the splits' partial results are merged by log-sum-exp (fa_lse_merge below).
 * This fills the GPU when B * Hq * ceil(Sq / 256) units are fewer than its SMs
 * (short query blocks against a long context).  The pages name sequence
 * parallelism ("Production Deployment Guide": distributed sequence parallelism
 * configurations) without a mechanism; this is its single-GPU form.
 *
 * fa_fwd_split_count: the number of splits fa_fwd_split uses when asked for
 * n_splits = 0.  With units = B * Hq * ceil(ceil(Sq / 128) / 2): 1 when
 * units >= sm_count; otherwise the n in 1..64 (and at most the kv tiles
 * ceil(Sk / 128)) that minimises ceil(n * units / sm_count) * (tiles + 3),
 * where tiles = ceil(kv tiles / n) is the length of a split and 3 the fixed
 * cost of a unit in kv tiles; ties go to the smaller n, and n is reduced so
 * that no split is empty.  sm_count <= 0 uses the current device's count.
 * Returns 0 on invalid sizes or when no device can be queried.
 */
int fa_fwd_split_count(int B, int Hq, int Sq, int Sk, int sm_count);

/*
 * Workspace bytes fa_fwd_split needs for n_splits (0: the automatic count on
 * the current device): fp32 parts of O [n, B, Hq, Sq, D] and of LSE
 * [n, B, Hq, Sq] for the effective split count n (a request above the kv tile
 * count, or one that would leave a split empty, is reduced).  0 when the
 * effective count is 1 (no workspace needed) or on invalid sizes.
 */
size_t fa_fwd_split_workspace_bytes(int B, int Hq, int Sq, int Sk, int D, int n_splits);

/*
 * fa_fwd_mod computed as n_splits key splits and a merge (two kernels).  Same
 * tensors, sizes, score modification and errors as fa_fwd_mod; mod == NULL is
 * no mask.  n_splits >= 0 (0: automatic, see fa_fwd_split_count); an effective
 * count of 1 runs fa_fwd_mod itself and ignores the workspace.  Otherwise the
 * workspace is a caller-owned device buffer of at least
 * fa_fwd_split_workspace_bytes(B, Hq, Sq, Sk, D, n_splits) bytes, 16-byte
 * aligned (else FA_ERR_WORKSPACE); it is scratch, its contents on return are
 * unspecified.  The result matches fa_fwd_mod up to the rounding of the
 * merge (O passes through fp32 parts, then one bf16 rounding).
 */
int fa_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                 int Hkv, int Sq, int Sk, int D, const fa_score_mod* mod, float scale,
                 int n_splits, void* workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Log-sum-exp merge of n_parts attention results over disjoint key sets of the
 * same queries (the identity behind the online softmax, "The Asymmetric
 * Hardware Scaling Wall" phases: rescale by the exponential of the change in
 * the max).  Per row r:
 *   M = max_c lse_parts[c][r],  lse[r] = M + ln sum_c exp(lse_parts[c][r] - M),
 *   o[r] = sum_c exp(lse_parts[c][r] - lse[r]) * o_parts[c][r]
 *   o_parts   [n_parts, rows, D] fp32, each part normalised by its own sum
 *   lse_parts [n_parts, rows] fp32, natural log; -inf marks an empty part,
 *             whose o_parts row is not read
 *   o [rows, D] bf16 out, lse [rows] fp32 out
 * A row whose parts are all empty gets o = 0 and lse = -inf.  rows >= 0
 * (0 is a no-op), n_parts >= 1, D in {64, 128}; o_parts and o 16-byte
 * aligned, lse_parts and lse 4-byte aligned (else FA_ERR_MISALIGNED).
 */
int fa_lse_merge(const float* o_parts, const float* lse_parts, int n_parts, void* o, float* lse,
                 int64_t rows, int D, fa_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* fa_status_string(int status);

/*
 * Test hook for the exponential split of the forward softmax (FlashAttention-4
 * pages, key contribution #2: a degree-3 polynomial on the FMA units run beside
 * the MUFU exp2).  Writes y[i] = 2^x[i] computed the way the kernel does:
 * which = 0 the hardware ex2.approx path, which = 1 the polynomial path,
 * which = 2 the same polynomial on the packed two-lane fp32 pipe (the form the
 * forward softmax runs; even elements go through lane 0, odd through lane 1).
 * x, y: device fp32 arrays of n elements.  Inputs below -125 give 2^-125 on the
 * polynomial path (the kernel's clamp), values above 64 are not supported.
 */
int fa_exp2_test(const float* x, float* y, int64_t n, int which, fa_stream_t stream);

/*
 * Test hook for the kernels' bounded waits.  One device thread runs one of the
 * waits the kernels use, with the same time limit (2 s of the GPU's global
 * timer), and writes FA_OK or FA_ERR_TIMEOUT to the device int *status:
 *   which = 0: the deterministic backward's semaphore spin, until the device
 *              int *flag reaches 1;
 *   which = 1: an mbarrier wait on a phase that nothing completes (always
 *              FA_ERR_TIMEOUT; flag is unused and may be null).
 * Returns FA_ERR_INVALID_ARG for another `which` or a null pointer it needs,
 * FA_ERR_MISALIGNED for pointers not 4-byte aligned; otherwise the launch
 * status.  The wait running out leaves the CUDA context usable.
 */
int fa_wait_test(const int* flag, int which, int* status, fa_stream_t stream);

/* Number of kernels the last forward, backward or merge call on this thread
 * launched. */
int fa_last_launch_count(void);

/*
 * Measurement hook.  Records two caller-owned CUDA events (cudaEvent_t, passed
 * as void*) on the call's stream immediately before and after the main kernel
 * of the NEXT fa_fwd or fa_bwd issued by this thread (the forward kernel, or
 * the backward's main kernel without its preprocess / convert kernels), then
 * forgets them.  Passing two nulls cancels a pending request.  Returns
 * FA_ERR_INVALID_ARG if exactly one of the two is null.
 */
int fa_set_timing_events(void* start_event, void* stop_event);

/*
 * Backward pass for callers that cannot allocate device memory.  The pages have
 * no counterpart: this exists for code that is not allowed to call cudaMalloc
 * or to own a workspace buffer (for example code running inside another
 * framework's allocator or memory pool, or a plugin limited to the buffers it
 * is handed).  It computes exactly what fa_bwd computes, with the same
 * arguments minus the workspace: the workspace is a fixed 32 MiB scratch array
 * compiled into this library, which every GPU that loads the library keeps
 * until the process exits.  No call allocates or frees memory.
 *   - Sizes whose workspace (fa_bwd_workspace_bytes) exceeds 32 MiB are
 *     rejected with FA_ERR_WORKSPACE (about 64,000 query rows B*Hq*Sq at
 *     D = 128, about 127,000 at D = 64; in the deterministic mode, which keeps up
 *     to four accumulators (two from 32 kv tiles on), about a quarter or a half
 *     of those); invalid sizes return
 *     FA_ERR_INVALID_ARG.
 *   - The first call on each device looks up the scratch's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - All calls share the one scratch array and it keeps the last call's
 *     contents; each call clears what it needs cleared.  Calls that overlap on
 *     the GPU (different streams, or different host threads without ordering)
 *     race on it and produce wrong gradients: serialise them.
 *   - A device-side wait that runs out is recorded in the scratch's status
 *     word; fa_bwd_noalloc_status reads it back.
 *   - The scratch's address is looked up once per device and kept, so the
 *     entry points must not be used across cudaDeviceReset of that device.
 */
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                   const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq,
                   int Sk, int D, int causal, float scale, int deterministic, fa_stream_t stream);

/*
 * Status of the last fa_bwd_noalloc on the current device (the pages have no
 * counterpart; this is the no-allocation form of fa_bwd_status).  Synchronises
 * `stream` (pass the stream of the fa_bwd_noalloc call), then returns FA_OK or
 * FA_ERR_TIMEOUT from the status word in the built-in scratch; FA_ERR_CUDA if
 * the synchronisation, the address lookup or the read fails.  Allocates
 * nothing.  Each fa_bwd_noalloc clears the word, so the status is that of the
 * latest call.
 */
int fa_bwd_noalloc_status(fa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */

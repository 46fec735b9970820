/*
 * capattn — soft-capped unified attention (forward and backward) on GB300.
 *
 * C ABI of the library libcapattn.so.  Plain pointers and sizes only.
 *
 * What the calls compute (pages "triton_kernels.py" and "mosaic_backward.py",
 * xrex_unified unified attention; notation per batch b and query head h, with
 * KV head g = h / q_heads_per_kv_head as in mosaic_backward.py
 * make_mosaic_backward_dq_kernel):
 *
 *   s_ij = sm_scale * <Q_i, K_j>                  (triton_kernels.py forward kernel)
 *   c_ij = cap(s_ij)                              (mosaic_backward.py _apply_cap_mosaic)
 *            none / cap <= 0 : s
 *            tanh            : cap * tanh(s / cap)
 *            soft_sign       : s / (1 + |s| / cap)
 *            alsc            : cap * (sig(a(s/cap + b)) - sig(ab)) / (sig(ab)(1 - sig(ab)) + 1e-12)
 *   t_ij = temp_i * c_ij                          (triton_kernels.py dQ kernel, temperature)
 *   live_ij = [seg_i == seg_j] and (!causal or i >= j) and
 *             (window_len == 0 or j > i - window_len) and ranker_ij
 *                                                 (triton_kernels.py forward kernel masks;
 *                                                  mosaic_backward.py ranker_mask_mosaic_kv_q)
 *   ranker_ij = (j in [hl,hu) and (i in [hl,hu) or i in [cl,cu)))
 *               or (i in [cl,cu) and i == j)
 *   LSE_i = log sum_{live j} exp(t_ij)   (natural log; -inf for a fully masked row)
 *   P_ij  = live_ij ? exp(t_ij - LSE_i) : 0,   O_i = sum_j P_ij V_j
 *
 * Backward (mosaic_backward.py backward kernels and delta pre-pass):
 *   delta_i = sum_d O_id dO_id
 *   dT_ij   = P_ij (dO_i . V_j - delta_i) + z_loss_weight * P_ij * LSE_i
 *   dX_ij   = sm_scale * cap'(s_ij) * temp_i * dT_ij   (cap' is the exact derivative of cap)
 *   dQ_i = sum_j dX_ij K_j;  dK_j = sum_{h in g} sum_i dX_ij Q_i;  dV_j = sum_{h in g} sum_i P_ij dO_i
 * which is the gradient of sum(O * dO) + (z_loss_weight / 2) * sum over live rows of LSE^2.
 *
 * Layouts (all contiguous, row-major), with L query rows and Lk keys:
 *   q, o, dO, dq : [B, L, Hq, D]      k, v, dk, dv : [B, Lk, Hkv, D]
 *   lse, m, l, delta : [B, Hq, L] float32
 *   temp : [B, L] float32 (NULL means 1)
 *   seg  : [B, L] int32 segment ids, non-decreasing along each batch row
 *          (packed documents); NULL means one segment.
 *   bounds : [B, 4] int32 (hl, hu, cl, cu) per batch row with
 *            0 <= hl <= hu <= L and 0 <= cl <= cu <= L; NULL disables the ranker mask.
 *   Query and key lengths may differ (mosaic_backward.py's orchestration reads
 *   q as (B, Q, H, D) and k as (B, KV, H_kv, D)): query i and key j positions
 *   are compared directly (causal keeps j <= i, the window j > i - window_len).
 *   seg and bounds describe one sequence and require Lk == L
 *   (CAPATTN_ERR_INVALID_ARG otherwise).
 *   Element type of q/k/v/o/dO/dq/dk/dv: bf16 (CAPATTN_BF16) or float32 (CAPATTN_FP32).
 *   Every tensor pointer must be 16-byte aligned.
 *
 * Ownership: the caller owns every buffer, including the workspace; the
 * library allocates no device memory on these calls.  All calls enqueue work on
 * `stream` and return without synchronising.  Argument errors are detected on
 * the host before anything is launched and returned synchronously.  Errors in
 * device-resident data (segment ids that decrease, ranker bounds out of range)
 * and bounded-wait timeouts inside kernels are recorded in a status word in the
 * workspace; read it with capattn_device_status.
 */
#ifndef CAPATTN_H_
#define CAPATTN_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum capattn_status {
  CAPATTN_OK = 0,
  CAPATTN_ERR_INVALID_ARG = 1,   /* bad shape, pointer, alignment or parameter */
  CAPATTN_ERR_UNSUPPORTED = 2,   /* valid but not implemented (head dim D other than 64 or 128) */
  CAPATTN_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
  CAPATTN_ERR_DEVICE_TIMEOUT = 4,/* a kernel gave up on a bounded wait (device status) */
  CAPATTN_ERR_WORKSPACE = 5,     /* workspace NULL or smaller than capattn_workspace_bytes */
  CAPATTN_ERR_DEVICE_DATA = 6,   /* device status: bad segment ids or ranker bounds */
  CAPATTN_ERR_TOO_LARGE = 7      /* problem needs more scratch than capattn_fwd_noalloc holds */
} capattn_status;

/* Cap methods (mosaic_backward.py _apply_cap_mosaic).  A cap <= 0 behaves as none. */
enum { CAPATTN_CAP_NONE = 0, CAPATTN_CAP_TANH = 1, CAPATTN_CAP_SOFT_SIGN = 2, CAPATTN_CAP_ALSC = 3 };

/* Element types of the attention tensors. */
enum { CAPATTN_BF16 = 0, CAPATTN_FP32 = 1 };

/* Which pass a workspace size or visit map refers to. */
enum { CAPATTN_PASS_FWD = 0, CAPATTN_PASS_BWD = 1, CAPATTN_PASS_BWD_NO_POOL = 2 };
enum { CAPATTN_VISIT_Q_TILES = 0, CAPATTN_VISIT_KV_TILES = 1 };
/* flags of capattn_bwd_ex */
enum { CAPATTN_BWD_REUSE_FWD_MAPS = 1 };

/*
 * Configuration (the pages' KernelConfig: cap method and parameters, sm_scale,
 * causal, window_len, z_loss_weight, and the GQA factor of
 * mosaic_attention_backward).  struct_size must be sizeof(capattn_config).
 */
typedef struct capattn_config {
  uint32_t struct_size;
  int32_t cap_method;          /* CAPATTN_CAP_* */
  float cap, alpha, beta;      /* cap > 0 activates the method; alpha, beta for ALSC */
  float sm_scale;              /* multiplies Q.K before the cap */
  int32_t causal;              /* nonzero: key j visible only if j <= i */
  int32_t window_len;          /* > 0: key j visible only if j > i - window_len; 0: off */
  float z_loss_weight;         /* >= 0; adds z * P * LSE to dT */
  int32_t q_heads_per_kv_head; /* G = Hq / Hkv */
  int32_t B, L, Hq, Hkv, D;    /* batch, sequence length, heads, head dim */
  int32_t dtype;               /* CAPATTN_BF16 or CAPATTN_FP32 */
  int32_t Lk;                  /* key / value length; 0 means Lk = L */
} capattn_config;

/* Human-readable name of a status code (static string). */
const char* capattn_status_string(capattn_status s);

/* Checks a configuration without touching any pointer (same rules as the compute calls). */
capattn_status capattn_validate_config(const capattn_config* cfg);

/*
 * Bytes of device workspace needed by capattn_fwd (pass CAPATTN_PASS_FWD) or
 * capattn_bwd / capattn_bwd_dtemp / capattn_bwd_ex (CAPATTN_PASS_BWD) for this
 * configuration; 0 if cfg is invalid.  The backward needs more: it also holds
 * the per-(head, row) partial sums of the temperature gradient (8 bytes per
 * (b, query head, row)) and, for bf16, a pool for the stored-dX backward:
 * 32 KB per (b, query head, query tile, key tile of the tile's band), the band
 * being the key tiles the causal / window masks of cfg leave a query tile
 * (all of them without those masks).  The pool is left out, and that backward
 * not used, when it would exceed 16 GiB.  CAPATTN_PASS_BWD_NO_POOL gives the
 * backward's size without the pool (the smallest workspace a backward takes;
 * it then recomputes dX for dQ).  A workspace sized for the backward serves
 * both passes.  The workspace must be 256-byte aligned.  Its first word is the
 * device status.
 */
size_t capattn_workspace_bytes(const capattn_config* cfg, int pass);

/*
 * Tile sizes the kernels use for this configuration (the granularity of the
 * visit maps): bf16 uses 128 x 128 tiles, fp32 64 x 64.
 */
capattn_status capattn_tile_sizes(const capattn_config* cfg, int32_t* block_q, int32_t* block_kv);

/*
 * Forward (triton_kernels.py make_triton_forward_kernel, with its residuals).
 * Inputs q, k, v, temp (nullable), seg (nullable), bounds (nullable): device.
 * k, v: [B,Lk,Hkv,D].  Outputs (device): o [B,L,Hq,D] in the input element type; lse [B,Hq,L]
 * natural-log log-sum-exp; m and l [B,Hq,L] (nullable): row max of t and
 * sum of exp(t - m), so that lse = m + log(l).  A fully masked row gives
 * o = 0, lse = m = -inf, l = 0.
 * workspace: device, >= capattn_workspace_bytes(cfg, CAPATTN_PASS_FWD).
 */
capattn_status capattn_fwd(const capattn_config* cfg, const void* q, const void* k, const void* v,
                           const float* temp, const int32_t* seg, const int32_t* bounds, void* o,
                           float* lse, float* m, float* l, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/*
 * Backward (mosaic_backward.py make_preprocess_backward_kernel,
 * make_mosaic_backward_dkv_kernel, make_mosaic_backward_dq_kernel and the
 * mosaic_attention_backward orchestration, with the group sum over query heads
 * done inside the dK/dV kernel).
 * Inputs (device): q, k, v, temp, seg, bounds as in capattn_fwd; o and lse as
 * written by capattn_fwd; dO [B,L,Hq,D] upstream gradient.
 * Outputs (device): dq [B,L,Hq,D], dk and dv [B,Lk,Hkv,D] (input element type,
 * fully overwritten); delta [B,Hq,L] float32 = rowsum(o * dO).
 * workspace: device, >= capattn_workspace_bytes(cfg, CAPATTN_PASS_BWD).
 * bf16 takes one of two kernel sequences.  With the dX pool (the workspace
 * holds it) and no temperature gradient: delta, then dK/dV, which also writes
 * each visited tile's dX to the pool, then dQ as a GEMM over the stored tiles
 * (the scores and dX are computed once per tile pair).  Otherwise (a smaller
 * workspace, or a temperature gradient): a dQ
 * kernel that recomputes the scores and dX and also writes delta, then dK/dV.
 * capattn_workspace_bytes(cfg, CAPATTN_PASS_BWD_NO_POOL) is the size without the pool.
 * The two agree to rounding (delta and dQ are summed in different orders).
 */
capattn_status capattn_bwd(const capattn_config* cfg, const void* q, const void* k, const void* v,
                           const float* temp, const int32_t* seg, const int32_t* bounds,
                           const void* o, const float* lse, const void* dO, void* dq, void* dk,
                           void* dv, float* delta, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/*
 * capattn_bwd plus the gradient of the per-query temperature, which the pages'
 * backward returns as zeros (mosaic_attention_backward): the forward
 * (triton_kernels.py make_triton_forward_kernel) multiplies the capped score
 * c = cap(sm_scale * q.k) by temp, so dtemp[b, i] = sum over query heads h and
 * keys j of dT[b,h,i,j] * c[b,h,i,j], with dT = P (dP - delta + z LSE) the
 * gradient of the tempered logit (0 for masked pairs).
 * temp and dtemp [B,L] float32 (device) are required (CAPATTN_ERR_INVALID_ARG
 * if either is null); dtemp is overwritten.  The dQ kernels leave per-(head,
 * row) partial sums in the workspace and a final pass adds them over the heads
 * in a fixed order, so dtemp is the same bit for bit on every run.  Everything
 * else is as in capattn_bwd.
 */
capattn_status capattn_bwd_dtemp(const capattn_config* cfg, const void* q, const void* k,
                                 const void* v, const float* temp, const int32_t* seg,
                                 const int32_t* bounds, const void* o, const float* lse,
                                 const void* dO, void* dq, void* dk, void* dv, float* delta,
                                 float* dtemp, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/*
 * The backward with every optional input and output; capattn_bwd is this call
 * with dlse = dtemp = NULL and flags = 0, capattn_bwd_dtemp with dlse = NULL
 * and flags = 0.
 * dlse [B,Hq,L] float32 (device, nullable): an upstream gradient of the lse
 * that capattn_fwd returns.  Since d lse_i / d t_ij = P_ij, it adds
 * dlse_i * P_ij to dT (the same form as the z-loss term of
 * mosaic_backward.py's backward kernels), so a caller whose own loss uses lse
 * gets that part of the gradient in dq, dk, dv (and dtemp).  Rows that are
 * fully masked ignore it.  dtemp [B,L] float32 (nullable) as in
 * capattn_bwd_dtemp; it needs temp (CAPATTN_ERR_INVALID_ARG otherwise).
 * flags: 0 or CAPATTN_BWD_REUSE_FWD_MAPS (other bits: CAPATTN_ERR_INVALID_ARG).
 * With CAPATTN_BWD_REUSE_FWD_MAPS the backward does not rebuild the per-row
 * live spans and the block visit maps: it uses the ones capattn_fwd left in
 * this workspace.  The caller guarantees that the last capattn_fwd on this
 * workspace ran with the same cfg, seg and bounds (same contents), and that
 * nothing but backward calls with those same arguments has used the workspace
 * since (they leave the maps as they were).  A call that breaks this gets wrong gradients,
 * not an error.  It also skips the device checks of seg and bounds, which
 * that capattn_fwd already reported in the status word.
 * Everything else is as in capattn_bwd.
 */
capattn_status capattn_bwd_ex(const capattn_config* cfg, const void* q, const void* k, const void* v,
                              const float* temp, const int32_t* seg, const int32_t* bounds,
                              const void* o, const float* lse, const void* dO, const float* dlse,
                              void* dq, void* dk, void* dv, float* delta, float* dtemp,
                              uint32_t flags, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream);

/*
 * Synchronises `stream`, reads and clears the device status word at the start
 * of `workspace`.  Returns CAPATTN_OK, CAPATTN_ERR_DEVICE_TIMEOUT or
 * CAPATTN_ERR_DEVICE_DATA; *raw_bits (nullable) receives the raw bits
 * (1 = wait timeout, 2 = decreasing segment ids, 4 = ranker bounds out of range,
 * 8 = history / candidate ids not contiguous, from capattn_ranker_bounds_from_ids,
 * 16 = a visited (query tile, key tile) pair outside the causal / window band of
 * the configuration, which the stored-dX backward has no slot for: an internal
 * inconsistency, never expected).
 */
capattn_status capattn_device_status(void* workspace, cudaStream_t stream, uint32_t* raw_bits);

/*
 * Self-check of the kernels' bounded waits (the pages have no counterpart:
 * this library bounds every mbarrier wait of its tcgen05 kernels instead of
 * waiting forever, and this call exercises that protocol).  Launches one CTA
 * per SM, each shaped like the attention kernels: it allocates all 512 TMEM
 * columns, one warp waits on an mbarrier that nothing arrives on for limit_ns
 * nanoseconds of the global timer (1 .. 100,000,000), gives up, records the
 * timeout bit (1) in the status word at the start of `workspace` and raises the
 * CTA's abort flag; the other waiting warps leave on the flag; TMEM is freed.
 * Afterwards capattn_device_status returns CAPATTN_ERR_DEVICE_TIMEOUT, and the
 * attention kernels run normally (a leaked TMEM allocation would stall them).
 * workspace: device, 256-byte aligned, at least 256 bytes.  Async on `stream`.
 * CAPATTN_ERR_WORKSPACE for a null or misaligned workspace,
 * CAPATTN_ERR_INVALID_ARG for a limit outside the range.
 */
capattn_status capattn_check_bounded_wait(void* workspace, uint64_t limit_ns, cudaStream_t stream);

/*
 * Ranker bounds from history / candidate segment ids (mosaic_backward.py's
 * test marks a row's history positions with HISTORY_SEGMENT_ID and its
 * candidates with CANDIDATE_SEGMENT_ID; the mapping to SegmentBounds is not
 * shown, so this is a stated reading): per batch row, history = [first, last +
 * 1) of the positions whose id is history_id, candidates likewise for
 * candidate_id, (0, 0) when an id is absent.
 * seg [B,L] int32 (device, 4-byte aligned); bounds [B,4] int32 (device, output,
 * (hl, hu, cl, cu) as the ranker mask of capattn_fwd / capattn_bwd reads them).
 * workspace (nullable; a capattn workspace): when given, a row whose history
 * or candidate positions have gaps sets status bit 8 (capattn_device_status
 * then returns CAPATTN_ERR_DEVICE_DATA); its bounds are still the hull.
 * Async on `stream`.  CAPATTN_ERR_INVALID_ARG for null arrays, B or L < 1, equal
 * ids or misaligned pointers.
 */
capattn_status capattn_ranker_bounds_from_ids(const int32_t* seg, int32_t B, int32_t L,
                                              int32_t history_id, int32_t candidate_id,
                                              int32_t* bounds, void* workspace, cudaStream_t stream);

/*
 * Visit maps (host computation).  For which = CAPATTN_VISIT_Q_TILES, out holds
 * for every (b, query tile) a bitmap over KV tiles: bit t of word
 * out[(b * n_q_tiles + qt) * words_kv + t / 32] is set iff the tile pair
 * holds at least one live (i, j); words_kv = ceil(n_kv_tiles / 32).  For
 * CAPATTN_VISIT_KV_TILES, the transpose: per (b, KV tile) a bitmap over query
 * tiles.  Tile sizes as capattn_tile_sizes.  seg and bounds: host, nullable.
 * out_words must be at least the map size; *n_words receives it.
 */
capattn_status capattn_visit_map_host(const capattn_config* cfg, const int32_t* seg,
                                      const int32_t* bounds, int which, uint32_t* out,
                                      size_t out_words, size_t* n_words);

/*
 * The same maps built by the device pre-pass that capattn_fwd / capattn_bwd
 * run, copied to the device buffer out (same format).  seg, bounds: device.
 * Uses `workspace` (>= capattn_workspace_bytes(cfg, CAPATTN_PASS_BWD)).
 */
capattn_status capattn_visit_map_device(const capattn_config* cfg, const int32_t* seg,
                                        const int32_t* bounds, int which, uint32_t* out,
                                        size_t out_words, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream);

/*
 * Live-pair bit matrix of batch row b (host computation with the same per-row
 * rule the kernels use): bit j of word bits[i * ceil(Lk/64) + j / 64] is set iff
 * pair (i, j) is live (i < L, j < Lk).  seg and bounds: host, nullable (full [B, L] / [B, 4]).
 */
capattn_status capattn_mask_bits_host(const capattn_config* cfg, const int32_t* seg,
                                      const int32_t* bounds, int32_t b, uint64_t* bits,
                                      size_t n_words);

/*
 * The polynomial the kernels use for the ALSC cap on the FMA pipe (a
 * restatement of mosaic_backward.py _apply_cap_mosaic's sigmoid, for speed):
 * sigma(alpha / cap * sm_scale * X + alpha * beta) - sigma(alpha * beta)
 *   = X * (coeffs[0] + coeffs[1] X + ... + coeffs[6] X^6)
 * for a raw score X (q . k, before sm_scale) with |X| <= *xmax; outside that
 * range (decided per warp and step) the kernels evaluate the sigmoid itself.
 * coeffs: host, 7 floats; xmax: host.  CAPATTN_ERR_INVALID_ARG unless the
 * config is valid with cap_method CAPATTN_CAP_ALSC and cap > 0.
 */
capattn_status capattn_debug_alsc_poly(const capattn_config* cfg, float* coeffs, float* xmax);

/*
 * Forward without any allocation or workspace argument (the pages have no
 * counterpart; this is an addition for callers that cannot allocate, such as
 * plugins inside a framework that owns all device memory and gives them no
 * scratch, or services held to a fixed memory budget).  Same inputs, outputs
 * and results as capattn_fwd, but the scratch lives in a fixed 8 MiB device
 * array inside the library (held by every GPU that loads it until exit).
 *  - Returns CAPATTN_ERR_TOO_LARGE, before launching anything, when
 *    capattn_workspace_bytes(cfg, CAPATTN_PASS_FWD) exceeds 8 MiB (roughly
 *    B * L above 500,000).
 *  - Calls no cudaMalloc, cudaFree or other allocating routine.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress with that device current); make that first call
 *    before any stream capture.  The address is kept for the life of the
 *    process: after cudaDeviceReset (or anything else that tears down the
 *    device's primary context) it is stale, so do not call this entry point on
 *    that device again.
 *  - All calls on a device share the one array: calls that may overlap on the
 *    GPU (different streams, or concurrent host threads) race on it and must be
 *    serialised by the caller.  Each call clears the array's status word first;
 *    read the bits that call left (wait timeouts, bad segment ids or ranker
 *    bounds) with capattn_noalloc_status before the next call.
 */
capattn_status capattn_fwd_noalloc(const capattn_config* cfg, const void* q, const void* k,
                                   const void* v, const float* temp, const int32_t* seg,
                                   const int32_t* bounds, void* o, float* lse, float* m, float* l,
                                   cudaStream_t stream);

/*
 * Device status left by the last capattn_fwd_noalloc call on the current
 * device (no counterpart on the pages; the companion of that entry point).
 * Synchronises `stream`, copies the status word of the fixed array into a host
 * word, clears it, and returns as capattn_device_status does (CAPATTN_OK,
 * CAPATTN_ERR_DEVICE_TIMEOUT or CAPATTN_ERR_DEVICE_DATA, raw bits in *raw_bits,
 * nullable).  Allocates no device memory.
 */
capattn_status capattn_noalloc_status(cudaStream_t stream, uint32_t* raw_bits);

/*
 * Per-kernel timing.  While enabled, every kernel the library launches whose
 * kind is selected (all kinds by default) is bracketed by CUDA events recorded
 * on the caller's stream (library-owned events; a small fixed pool), and the
 * launches of every kind are counted.  capattn_profile_read synchronises those
 * events and returns, per kernel kind (CAPATTN_KERNEL_*), the summed
 * milliseconds (0 for unselected kinds) and launch counts since the last reset
 * (reset = nonzero clears after reading).  Each recorded event costs the stream
 * a few microseconds, so a timing run selects only the kernel it times.
 * capattn_profile_select takes a bit mask of kinds (bit k = kind k; 0 selects
 * none) and returns CAPATTN_ERR_INVALID_ARG for bits beyond the known kinds.
 * Not thread-safe; meant for benchmarking.  Disabled by default.
 */
enum { CAPATTN_KERNEL_PREPASS = 0, CAPATTN_KERNEL_FWD = 1, CAPATTN_KERNEL_DELTA = 2,
       CAPATTN_KERNEL_DKV = 3, CAPATTN_KERNEL_DQ = 4, CAPATTN_KERNEL_KINDS = 5 };
capattn_status capattn_profile_enable(int on);
capattn_status capattn_profile_select(unsigned int kind_mask);
capattn_status capattn_profile_read(double* ms, int64_t* launches, int n_kinds, int reset);
const char* capattn_kernel_name(int kind);

#ifdef __cplusplus
}
#endif

#endif /* CAPATTN_H_ */

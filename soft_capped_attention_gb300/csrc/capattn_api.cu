// C-ABI entry points: argument validation, workspace layout, cap constants,
// host-side visit maps and mask bits, and the launch sequence of each pass.
#include <math.h>
#include <string.h>

#include <vector>

#include "capattn_internal.h"
#include "row_span.h"

namespace capattn {

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static int tile_q(const capattn_config& c) { return c.dtype == CAPATTN_BF16 ? 128 : 64; }
static int tile_kv(const capattn_config& c) { return c.dtype == CAPATTN_BF16 ? 128 : 64; }
// Key / value length (0 in the config means equal to the query length).
static int key_len(const capattn_config& c) { return c.Lk > 0 ? c.Lk : c.L; }

WorkspaceLayout workspace_layout(const capattn_config& c, int bq, int bk) {
  WorkspaceLayout w;
  const size_t nq = (c.L + bq - 1) / bq, nk = (key_len(c) + bk - 1) / bk;
  const size_t wq = (nq + 31) / 32, wk = (nk + 31) / 32;
  w.status_off = 0;
  w.rowinfo_off = 256;
  w.qmap_off = align256(w.rowinfo_off + sizeof(int4) * (size_t)c.B * c.L);
  w.kmap_off = align256(w.qmap_off + sizeof(uint32_t) * (size_t)c.B * nq * wk);
  w.qfull_off = align256(w.kmap_off + sizeof(uint32_t) * (size_t)c.B * nk * wq);
  w.total = align256(w.qfull_off + sizeof(int2) * (size_t)c.B * nq);
  w.dtemp_part_off = w.total;
  w.total_bwd = align256(w.dtemp_part_off + sizeof(float) * 2 * (size_t)c.B * c.Hq * c.L);
  // dX pool of the stored-dX backward (bf16 only): per (batch, query head,
  // query tile) a slot for every key tile of the tile's causal / window band
  // [kt_lo, kt_hi]; the data-dependent masks only ever remove tiles from it.
  w.dx_off = w.total_dx = w.total_bwd;
  w.dx_wmax = 0;
  w.dx_c = c.window_len > 0 ? (c.window_len - 1 + bk - 1) / bk : -1;
  if (c.dtype == CAPATTN_BF16 && bq == bk) {
    int64_t wmax = 0;
    for (int64_t qt = 0; qt < (int64_t)nq; ++qt) {
      const int64_t lo = w.dx_c >= 0 ? (qt - w.dx_c > 0 ? qt - w.dx_c : 0) : 0;
      const int64_t hi = c.causal ? (qt < (int64_t)nk - 1 ? qt : (int64_t)nk - 1) : (int64_t)nk - 1;
      if (hi - lo + 1 > wmax) wmax = hi - lo + 1;
    }
    const double pool = (double)c.B * c.Hq * (double)nq * (double)wmax * (double)kDxTileBytes;
    if (wmax > 0 && pool <= (double)kDxPoolMaxBytes) {
      w.dx_wmax = (int32_t)wmax;
      w.dx_off = (w.total_bwd + 1023) & ~size_t(1023);
      w.total_dx = w.dx_off + (size_t)pool;
    }
  }
  return w;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Segment ids and ranker bounds describe positions of one sequence: they need
// equal query and key lengths.
static capattn_status check_masks(const capattn_config& c, const void* seg, const void* bounds) {
  return (key_len(c) != c.L && (seg || bounds)) ? CAPATTN_ERR_INVALID_ARG : CAPATTN_OK;
}

static capattn_status validate(const capattn_config* c) {
  if (!c) return CAPATTN_ERR_INVALID_ARG;
  if (c->struct_size != sizeof(capattn_config)) return CAPATTN_ERR_INVALID_ARG;
  if (c->B < 1 || c->L < 1 || c->Lk < 0 || c->Hq < 1 || c->Hkv < 1 || c->D < 1)
    return CAPATTN_ERR_INVALID_ARG;
  if (c->q_heads_per_kv_head < 1 || c->Hkv * c->q_heads_per_kv_head != c->Hq)
    return CAPATTN_ERR_INVALID_ARG;
  if (c->dtype != CAPATTN_BF16 && c->dtype != CAPATTN_FP32) return CAPATTN_ERR_INVALID_ARG;
  if (c->cap_method < CAPATTN_CAP_NONE || c->cap_method > CAPATTN_CAP_ALSC)
    return CAPATTN_ERR_INVALID_ARG;
  if (!(isfinite(c->sm_scale)) || !(isfinite(c->cap)) || !(isfinite(c->alpha)) ||
      !(isfinite(c->beta)) || !(isfinite(c->z_loss_weight)) || c->z_loss_weight < 0.f)
    return CAPATTN_ERR_INVALID_ARG;
  if (c->window_len < 0) return CAPATTN_ERR_INVALID_ARG;
  // Index arithmetic in the kernels is 32-bit per (batch, head) plane and
  // 64-bit across planes; keep one plane comfortably inside int32.
  if ((int64_t)c->L * c->Hq * c->D >= (1ll << 31)) return CAPATTN_ERR_UNSUPPORTED;
  if ((int64_t)key_len(*c) * c->Hkv * c->D >= (1ll << 31)) return CAPATTN_ERR_UNSUPPORTED;
  if (c->D != 64 && c->D != 128) return CAPATTN_ERR_UNSUPPORTED;
  return CAPATTN_OK;
}

// sigma(b + d) - sigma(b) = d * g(d) for |d| <= kAlscPolyD: g interpolated at
// the 7 Chebyshev nodes of [-kAlscPolyD, kAlscPolyD] (degree 6, error ~1e-8
// against g's values of 0.1 .. 0.25), then written in the raw score X = d / u:
// sigma - sigma(b) = X * sum_k gu[k] X^k with gu[k] = g_k u^(k + 1).
static constexpr double kAlscPolyD = 0.5;
static void alsc_poly_fit(double b, double sb, double u, float gu[7], float* xmax) {
  const double pi = 3.14159265358979323846;
  double a[7][8];  // Vandermonde rows in t = d / D, with the values g(d) appended
  for (int j = 0; j < 7; ++j) {
    const double t = cos((2.0 * j + 1.0) * pi / 14.0);
    const double d = kAlscPolyD * t;
    const double g = fabs(d) < 1e-9 ? sb * (1.0 - sb) : (1.0 / (1.0 + exp(-(b + d))) - sb) / d;
    double tk = 1.0;
    for (int k = 0; k < 7; ++k) {
      a[j][k] = tk;
      tk *= t;
    }
    a[j][7] = g;
  }
  // Gaussian elimination with partial pivoting
  for (int c = 0; c < 7; ++c) {
    int piv = c;
    for (int r = c + 1; r < 7; ++r)
      if (fabs(a[r][c]) > fabs(a[piv][c])) piv = r;
    for (int k = 0; k < 8; ++k) std::swap(a[c][k], a[piv][k]);
    for (int r = 0; r < 7; ++r) {
      if (r == c) continue;
      const double f = a[r][c] / a[c][c];
      for (int k = c; k < 8; ++k) a[r][k] -= f * a[c][k];
    }
  }
  double up = u;       // u^(k + 1)
  double dk = 1.0;     // D^k
  for (int k = 0; k < 7; ++k) {
    gu[k] = (float)(a[k][7] / a[k][k] / dk * up);
    up *= u;
    dk *= kAlscPolyD;
  }
  *xmax = u > 0.0 ? (float)(kAlscPolyD / u) : 0.f;
}

static CapConsts make_cap(const capattn_config& c) {
  CapConsts k;
  memset(&k, 0, sizeof(k));
  k.method = (c.cap > 0.f) ? c.cap_method : CAPATTN_CAP_NONE;
  const double cap = c.cap > 0.f ? (double)c.cap : 1.0;
  k.cap = (float)cap;
  k.inv_cap = (float)(1.0 / cap);
  if (k.method == CAPATTN_CAP_ALSC) {
    const double ab = (double)c.alpha * (double)c.beta;
    const double sb = 1.0 / (1.0 + exp(-ab));
    const double denom = sb * (1.0 - sb) + 1e-12;
    k.alsc_a = (float)((double)c.alpha / cap);
    k.alsc_b = (float)ab;
    k.alsc_out = (float)(cap / denom);
    k.alsc_sb = (float)sb;
    k.alsc_dout = (float)((double)c.alpha / denom);
    alsc_poly_fit(ab, sb, (double)c.sm_scale * (double)c.alpha / cap, k.alsc_gu, &k.alsc_xmax);
  }
  return k;
}

static void fill_params(Params& p, const capattn_config& c, void* ws) {
  memset(&p, 0, sizeof(p));
  p.B = c.B; p.L = c.L; p.Lk = key_len(c); p.Hq = c.Hq; p.Hkv = c.Hkv; p.D = c.D;
  p.G = c.q_heads_per_kv_head;
  p.block_q = tile_q(c);
  p.block_kv = tile_kv(c);
  p.nq = (c.L + p.block_q - 1) / p.block_q;
  p.nk = (p.Lk + p.block_kv - 1) / p.block_kv;
  p.wq = (p.nq + 31) / 32;
  p.wk = (p.nk + 31) / 32;
  p.sm_scale = c.sm_scale;
  p.causal = c.causal ? 1 : 0;
  p.window_len = c.window_len;
  p.z_loss_weight = c.z_loss_weight;
  p.cap = make_cap(c);
  WorkspaceLayout w = workspace_layout(c, p.block_q, p.block_kv);
  char* base = static_cast<char*>(ws);
  p.status = reinterpret_cast<uint32_t*>(base + w.status_off);
  p.dq_work = reinterpret_cast<uint32_t*>(base + w.status_off + 128);  // in the status block
  p.fwd_work = reinterpret_cast<uint32_t*>(base + w.status_off + 192);
  p.rowinfo = reinterpret_cast<int4*>(base + w.rowinfo_off);
  p.qmap = reinterpret_cast<uint32_t*>(base + w.qmap_off);
  p.kmap = reinterpret_cast<uint32_t*>(base + w.kmap_off);
  p.qfull = reinterpret_cast<int2*>(base + w.qfull_off);
  p.dtemp_part = reinterpret_cast<float*>(base + w.dtemp_part_off);  // backward workspace only
  p.dx_pool = nullptr;  // set by a backward that takes the stored-dX path
  p.dx_wmax = w.dx_wmax;
  p.dx_c = w.dx_c;
}

static capattn_status check_ws(const capattn_config& c, void* ws, size_t bytes, int pass) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return CAPATTN_ERR_WORKSPACE;
  const WorkspaceLayout w = workspace_layout(c, tile_q(c), tile_kv(c));
  if (bytes < (pass == CAPATTN_PASS_BWD ? w.total_bwd : w.total)) return CAPATTN_ERR_WORKSPACE;
  return CAPATTN_OK;
}

// Whether a backward takes the stored-dX path: bf16, no temperature gradient
// (the dQ kernel's per-row sums provide it), and a workspace that holds the pool.
static bool use_dx_pool(const capattn_config& c, size_t bytes, bool dtemp) {
  if (c.dtype != CAPATTN_BF16 || dtemp) return false;
  const WorkspaceLayout w = workspace_layout(c, tile_q(c), tile_kv(c));
  return w.dx_wmax > 0 && bytes >= w.total_dx;
}

static capattn_status cuda_status(cudaError_t e) {
  return e == cudaSuccess ? CAPATTN_OK : CAPATTN_ERR_CUDA;
}

// Host restatement of the pre-pass, for the debug exports.
static void host_spans(const capattn_config& c, const int32_t* seg, const int32_t* bounds, int b,
                       std::vector<RowSpan>& spans) {
  spans.resize(c.L);
  const int32_t* srow = seg ? seg + (size_t)b * c.L : nullptr;
  int32_t hl = 0, hu = 0, cl = 0, cu = 0;
  if (bounds) {
    hl = imin32(imax32(bounds[4 * b + 0], 0), c.L);
    hu = imin32(imax32(bounds[4 * b + 1], 0), c.L);
    cl = imin32(imax32(bounds[4 * b + 2], 0), c.L);
    cu = imin32(imax32(bounds[4 * b + 3], 0), c.L);
  }
  const int32_t Lk = key_len(c);
  for (int i = 0; i < c.L; ++i) {
    int32_t first = 0, last1 = Lk;
    if (srow) {
      first = lower_bound_i32(srow, c.L, srow[i]);
      last1 = upper_bound_i32(srow, c.L, srow[i]);
    }
    spans[i] = row_span(i, Lk, c.causal ? 1 : 0, c.window_len, first, last1, bounds ? 1 : 0, hl,
                        hu, cl, cu);
  }
}

}  // namespace capattn

using namespace capattn;

// Backward with the optional LSE gradient and temperature gradient.
static capattn_status bwd_impl(const capattn_config* cfg, const void* q, const void* k, const void* v,
                               const float* temp, const int32_t* seg, const int32_t* bounds,
                               const void* o, const float* lse, const void* dO, const float* dlse,
                               void* dq, void* dk, void* dv, float* delta, float* dtemp,
                               uint32_t flags, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
  capattn_status st = validate(cfg);
  if (st != CAPATTN_OK) return st;
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv || !delta)
    return CAPATTN_ERR_INVALID_ARG;
  if (flags & ~(uint32_t)CAPATTN_BWD_REUSE_FWD_MAPS) return CAPATTN_ERR_INVALID_ARG;
  st = check_masks(*cfg, seg, bounds);
  if (st != CAPATTN_OK) return st;
  if (dtemp && !temp) return CAPATTN_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv, delta, temp, seg, bounds, dtemp, dlse};
  for (const void* ptr : ptrs)
    if (ptr && !aligned16(ptr)) return CAPATTN_ERR_INVALID_ARG;
  st = check_ws(*cfg, workspace, workspace_bytes, CAPATTN_PASS_BWD);
  if (st != CAPATTN_OK) return st;
  Params p;
  fill_params(p, *cfg, workspace);
  p.q = q; p.k = k; p.v = v; p.temp = temp; p.seg = seg; p.bounds = bounds;
  p.o = const_cast<void*>(o); p.lse = const_cast<float*>(lse);
  p.dO = dO; p.dq = dq; p.dk = dk; p.dv = dv; p.delta = delta; p.dtemp = dtemp; p.dlse = dlse;
  if (use_dx_pool(*cfg, workspace_bytes, dtemp != nullptr))
    p.dx_pool = static_cast<char*>(workspace) + workspace_layout(*cfg, p.block_q, p.block_kv).dx_off;
  // Spans and query-tile maps: from the forward (same workspace, same inputs)
  // or rebuilt.  Key-tile map: on the bf16 paths the dQ kernel or the delta
  // kernel ORs it together from the query-tile maps into the words
  // rowmap_kernel cleared; fp32 runs kmap_kernel.
  const bool reuse = (flags & CAPATTN_BWD_REUSE_FWD_MAPS) != 0;
  cudaError_t e = launch_prepass(p, !reuse, cfg->dtype != CAPATTN_BF16, stream);
  if (e != cudaSuccess) return cuda_status(e);
  // bf16: the dQ kernel computes delta itself; fp32: a separate pass
  if (cfg->dtype != CAPATTN_BF16) {
    e = launch_delta_fp32(p, stream);
    if (e != cudaSuccess) return cuda_status(e);
  }
  e = (cfg->dtype == CAPATTN_BF16) ? launch_bwd_bf16(p, stream) : launch_bwd_fp32(p, stream);
  if (e != cudaSuccess) return cuda_status(e);
  // dtemp: the dQ kernels leave per-(head, row) partial sums; they are added in
  // a fixed order, so the result does not depend on scheduling
  if (dtemp) e = launch_dtemp_reduce(p, stream);
  return cuda_status(e);
}

extern "C" {

capattn_status capattn_debug_alsc_poly(const capattn_config* cfg, float* coeffs, float* xmax) {
  const capattn_status st = validate(cfg);
  if (st != CAPATTN_OK) return st;
  if (!coeffs || !xmax || cfg->cap_method != CAPATTN_CAP_ALSC || !(cfg->cap > 0.f)) return CAPATTN_ERR_INVALID_ARG;
  const CapConsts k = make_cap(*cfg);
  for (int i = 0; i < 7; ++i) coeffs[i] = k.alsc_gu[i];
  *xmax = k.alsc_xmax;
  return CAPATTN_OK;
}


const char* capattn_status_string(capattn_status s) {
  switch (s) {
    case CAPATTN_OK: return "ok";
    case CAPATTN_ERR_INVALID_ARG: return "invalid argument";
    case CAPATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case CAPATTN_ERR_CUDA: return "CUDA error";
    case CAPATTN_ERR_DEVICE_TIMEOUT: return "a kernel gave up on a bounded wait";
    case CAPATTN_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case CAPATTN_ERR_DEVICE_DATA: return "invalid device data (segment ids or ranker bounds)";
    case CAPATTN_ERR_TOO_LARGE: return "problem exceeds the fixed scratch of capattn_fwd_noalloc";
  }
  return "unknown status";
}

capattn_status capattn_validate_config(const capattn_config* cfg) { return validate(cfg); }

size_t capattn_workspace_bytes(const capattn_config* cfg, int pass) {
  if (validate(cfg) != CAPATTN_OK) return 0;
  const WorkspaceLayout w = workspace_layout(*cfg, tile_q(*cfg), tile_kv(*cfg));
  switch (pass) {
    case CAPATTN_PASS_FWD: return w.total;
    case CAPATTN_PASS_BWD: return w.total_dx;
    case CAPATTN_PASS_BWD_NO_POOL: return w.total_bwd;
  }
  return 0;
}

capattn_status capattn_tile_sizes(const capattn_config* cfg, int32_t* block_q, int32_t* block_kv) {
  capattn_status st = validate(cfg);
  if (st != CAPATTN_OK) return st;
  if (block_q) *block_q = tile_q(*cfg);
  if (block_kv) *block_kv = tile_kv(*cfg);
  return CAPATTN_OK;
}

capattn_status capattn_fwd(const capattn_config* cfg, const void* q, const void* k, const void* v,
                           const float* temp, const int32_t* seg, const int32_t* bounds, void* o,
                           float* lse, float* m, float* l, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
  capattn_status st = validate(cfg);
  if (st != CAPATTN_OK) return st;
  if (!q || !k || !v || !o || !lse) return CAPATTN_ERR_INVALID_ARG;
  st = check_masks(*cfg, seg, bounds);
  if (st != CAPATTN_OK) return st;
  const void* ptrs[] = {q, k, v, o, lse, temp, seg, bounds, m, l};
  for (const void* ptr : ptrs)
    if (ptr && !aligned16(ptr)) return CAPATTN_ERR_INVALID_ARG;
  st = check_ws(*cfg, workspace, workspace_bytes, CAPATTN_PASS_FWD);
  if (st != CAPATTN_OK) return st;
  Params p;
  fill_params(p, *cfg, workspace);
  p.q = q; p.k = k; p.v = v; p.temp = temp; p.seg = seg; p.bounds = bounds;
  p.o = o; p.lse = lse; p.m = m; p.l = l;
  cudaError_t e = launch_prepass(p, true, false, stream);
  if (e != cudaSuccess) return cuda_status(e);
  e = (cfg->dtype == CAPATTN_BF16) ? launch_fwd_bf16(p, stream) : launch_fwd_fp32(p, stream);
  return cuda_status(e);
}

capattn_status capattn_bwd(const capattn_config* cfg, const void* q, const void* k, const void* v,
                           const float* temp, const int32_t* seg, const int32_t* bounds,
                           const void* o, const float* lse, const void* dO, void* dq, void* dk,
                           void* dv, float* delta, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
  return bwd_impl(cfg, q, k, v, temp, seg, bounds, o, lse, dO, nullptr, dq, dk, dv, delta, nullptr,
                  0u, workspace, workspace_bytes, stream);
}

capattn_status capattn_bwd_ex(const capattn_config* cfg, const void* q, const void* k, const void* v,
                              const float* temp, const int32_t* seg, const int32_t* bounds,
                              const void* o, const float* lse, const void* dO, const float* dlse,
                              void* dq, void* dk, void* dv, float* delta, float* dtemp,
                              uint32_t flags, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
  return bwd_impl(cfg, q, k, v, temp, seg, bounds, o, lse, dO, dlse, dq, dk, dv, delta, dtemp,
                  flags, workspace, workspace_bytes, stream);
}

capattn_status capattn_bwd_dtemp(const capattn_config* cfg, const void* q, const void* k,
                                 const void* v, const float* temp, const int32_t* seg,
                                 const int32_t* bounds, const void* o, const float* lse,
                                 const void* dO, void* dq, void* dk, void* dv, float* delta,
                                 float* dtemp, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream) {
  if (!temp || !dtemp) return CAPATTN_ERR_INVALID_ARG;
  return bwd_impl(cfg, q, k, v, temp, seg, bounds, o, lse, dO, nullptr, dq, dk, dv, delta, dtemp,
                  0u, workspace, workspace_bytes, stream);
}

capattn_status capattn_ranker_bounds_from_ids(const int32_t* seg, int32_t B, int32_t L,
                                              int32_t history_id, int32_t candidate_id,
                                              int32_t* bounds, void* workspace, cudaStream_t stream) {
  if (!seg || !bounds || B < 1 || L < 1 || history_id == candidate_id) return CAPATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(seg) & 3u) || (reinterpret_cast<uintptr_t>(bounds) & 3u) ||
      (workspace && !aligned16(workspace)))
    return CAPATTN_ERR_INVALID_ARG;
  return cuda_status(launch_ranker_bounds(seg, B, L, history_id, candidate_id, bounds,
                                          static_cast<uint32_t*>(workspace), stream));
}

capattn_status capattn_device_status(void* workspace, cudaStream_t stream, uint32_t* raw_bits) {
  if (!workspace) return CAPATTN_ERR_WORKSPACE;
  uint32_t bits = 0;
  if (cudaMemcpyAsync(&bits, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    return CAPATTN_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return CAPATTN_ERR_CUDA;
  if (bits && cudaMemsetAsync(workspace, 0, sizeof(uint32_t), stream) != cudaSuccess)
    return CAPATTN_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return CAPATTN_ERR_CUDA;
  if (raw_bits) *raw_bits = bits;
  if (bits & kStatusTimeoutBit) return CAPATTN_ERR_DEVICE_TIMEOUT;
  if (bits) return CAPATTN_ERR_DEVICE_DATA;
  return CAPATTN_OK;
}

capattn_status capattn_check_bounded_wait(void* workspace, uint64_t limit_ns, cudaStream_t stream) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return CAPATTN_ERR_WORKSPACE;
  if (limit_ns < 1 || limit_ns > 100000000ull) return CAPATTN_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return CAPATTN_ERR_CUDA;
  return cuda_status(launch_wait_check(static_cast<uint32_t*>(workspace), limit_ns, sms, stream));
}

capattn_status capattn_visit_map_host(const capattn_config* cfg, const int32_t* seg,
                                      const int32_t* bounds, int which, uint32_t* out,
                                      size_t out_words, size_t* n_words) {
  capattn_status st = validate(cfg);
  if (st != CAPATTN_OK) return st;
  if (which != CAPATTN_VISIT_Q_TILES && which != CAPATTN_VISIT_KV_TILES)
    return CAPATTN_ERR_INVALID_ARG;
  st = check_masks(*cfg, seg, bounds);
  if (st != CAPATTN_OK) return st;
  const int bq = tile_q(*cfg), bk = tile_kv(*cfg);
  const int nq = (cfg->L + bq - 1) / bq, nk = (key_len(*cfg) + bk - 1) / bk;
  const int wq = (nq + 31) / 32, wk = (nk + 31) / 32;
  const size_t need = which == CAPATTN_VISIT_Q_TILES ? (size_t)cfg->B * nq * wk
                                                     : (size_t)cfg->B * nk * wq;
  if (n_words) *n_words = need;
  if (!out) return out_words == 0 ? CAPATTN_OK : CAPATTN_ERR_INVALID_ARG;
  if (out_words < need) return CAPATTN_ERR_INVALID_ARG;
  memset(out, 0, need * sizeof(uint32_t));
  std::vector<RowSpan> spans;
  for (int b = 0; b < cfg->B; ++b) {
    host_spans(*cfg, seg, bounds, b, spans);
    for (int i = 0; i < cfg->L; ++i) {
      const RowSpan& r = spans[i];
      const int qt = i / bq;
      auto mark = [&](int kt) {
        if (which == CAPATTN_VISIT_Q_TILES)
          out[((size_t)b * nq + qt) * wk + kt / 32] |= 1u << (kt % 32);
        else
          out[((size_t)b * nk + kt) * wq + qt / 32] |= 1u << (qt % 32);
      };
      if (r.hi > r.lo)
        for (int kt = r.lo / bk; kt <= (r.hi - 1) / bk; ++kt) mark(kt);
      if (r.e >= 0) mark(r.e / bk);
    }
  }
  return CAPATTN_OK;
}

capattn_status capattn_visit_map_device(const capattn_config* cfg, const int32_t* seg,
                                        const int32_t* bounds, int which, uint32_t* out,
                                        size_t out_words, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream) {
  capattn_status st = validate(cfg);
  if (st != CAPATTN_OK) return st;
  if (which != CAPATTN_VISIT_Q_TILES && which != CAPATTN_VISIT_KV_TILES)
    return CAPATTN_ERR_INVALID_ARG;
  st = check_masks(*cfg, seg, bounds);
  if (st != CAPATTN_OK) return st;
  st = check_ws(*cfg, workspace, workspace_bytes, CAPATTN_PASS_FWD);
  if (st != CAPATTN_OK) return st;
  Params p;
  fill_params(p, *cfg, workspace);
  p.seg = seg;
  p.bounds = bounds;
  const size_t need = which == CAPATTN_VISIT_Q_TILES ? (size_t)p.B * p.nq * p.wk
                                                     : (size_t)p.B * p.nk * p.wq;
  if (!out || out_words < need) return CAPATTN_ERR_INVALID_ARG;
  cudaError_t e = launch_prepass(p, true, true, stream);
  if (e != cudaSuccess) return cuda_status(e);
  e = cudaMemcpyAsync(out, which == CAPATTN_VISIT_Q_TILES ? p.qmap : p.kmap,
                      need * sizeof(uint32_t), cudaMemcpyDeviceToDevice, stream);
  return cuda_status(e);
}

capattn_status capattn_mask_bits_host(const capattn_config* cfg, const int32_t* seg,
                                      const int32_t* bounds, int32_t b, uint64_t* bits,
                                      size_t n_words) {
  capattn_status st = validate(cfg);
  if (st != CAPATTN_OK) return st;
  if (b < 0 || b >= cfg->B || !bits) return CAPATTN_ERR_INVALID_ARG;
  st = check_masks(*cfg, seg, bounds);
  if (st != CAPATTN_OK) return st;
  const int Lk = key_len(*cfg);
  const size_t wpr = (Lk + 63) / 64;
  if (n_words < wpr * cfg->L) return CAPATTN_ERR_INVALID_ARG;
  memset(bits, 0, wpr * cfg->L * sizeof(uint64_t));
  std::vector<RowSpan> spans;
  host_spans(*cfg, seg, bounds, b, spans);
  for (int i = 0; i < cfg->L; ++i)
    for (int j = 0; j < Lk; ++j)
      if (span_live(spans[i], j)) bits[i * wpr + j / 64] |= 1ull << (j % 64);
  return CAPATTN_OK;
}

}  // extern "C"

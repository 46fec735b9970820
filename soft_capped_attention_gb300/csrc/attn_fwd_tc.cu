// bf16 forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes: triton_kernels.py make_triton_forward_kernel (scores, cap,
// temperature, masks, online softmax with the l / m residuals), with the cap
// forms of mosaic_backward.py _apply_cap_mosaic, the ranker mask of
// ranker_mask_mosaic_kv_q (transposed) and an exp2-domain softmax as in the
// Mosaic kernels.
//
// One CTA owns two 128-row query tiles (Q0, Q1) of one (batch, head) and walks
// the union of their KV visit maps.  Warp roles (10 warps):
//   warp 0      TMA producer: Q0, Q1 once, then K_j / V_j into a 2-stage ring;
//   warp 1      TMEM allocator and MMA issuer (one thread), ping-ponging the
//               two tiles so that one tile's softmax overlaps the other tile's
//               MMAs:  S0_j S1_j | PV0_j S0_{j+1} | PV1_j S1_{j+1} | ...
//                 S_t = Q_t K_j^T  (SS MMA, M = N = 128)
//                 O_t += P_t V_j   (TS MMA: P_t read from TMEM as bf16)
//   warps 2..5  softmax of tile 0, warps 6..9 softmax of tile 1: one thread
//               per query row (its TMEM lane).  Pass 1 takes the row maximum of
//               the raw scores (every cap is increasing, so the logit maximum is
//               the transformed raw maximum); pass 2 applies sm_scale, cap,
//               temperature and the row's live span, writes P = 2^(x - m) as
//               packed bf16 over the first 64 columns of S, and accumulates l.
//               The running max is only moved (and O rescaled in TMEM) when it
//               grows by more than 2^8; otherwise P stays <= 256.
// A tile's S_{j+1} is issued after its PV_j, so when the softmax sees S_{j+1}
// complete, PV_j is complete too and O may be rescaled in place.
// TMEM: S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512).
#include <math.h>

#include "cap_math.cuh"
#include "capattn_internal.h"
#include "softmax_elem.cuh"
#include "tc_common.cuh"
#include "tma_maps.h"

namespace capattn {

namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int HD = 128;
constexpr int NSTAGE = 2;
constexpr int SLAB = 128 * 64 * 2;          // one [128][64] bf16 box
constexpr int TILE = 2 * SLAB;               // 128 x 128 bf16
constexpr int SMEM_BYTES = 2 * TILE + NSTAGE * 2 * TILE + 1024;
constexpr int NTHREADS = 320;
constexpr float kRescaleThreshold = 8.0f;    // log2 units

// Iterates the union of two rows of a visit bitmap, reporting per tile which
// of the two query tiles is live in it.
struct PairIter {
  const uint32_t* m0;
  const uint32_t* m1;  // null when the second tile does not exist
  int nwords, w;
  uint32_t b0, b1;
  __device__ PairIter(const uint32_t* a, const uint32_t* c, int n) : m0(a), m1(c), nwords(n), w(0) {
    b0 = n > 0 ? a[0] : 0u;
    b1 = (n > 0 && c) ? c[0] : 0u;
  }
  __device__ bool next(int& t, bool& a0, bool& a1) {
    while ((b0 | b1) == 0u) {
      if (++w >= nwords) return false;
      b0 = m0[w];
      b1 = m1 ? m1[w] : 0u;
    }
    const uint32_t u = b0 | b1;
    const int bit = __ffs(u) - 1;
    const uint32_t mask = 1u << bit;
    a0 = (b0 & mask) != 0u;
    a1 = (b1 & mask) != 0u;
    b0 &= ~mask;
    b1 &= ~mask;
    t = w * 32 + bit;
    return true;
  }
};

__device__ __forceinline__ int count_union(const uint32_t* a, const uint32_t* c, int n) {
  int s = 0;
  for (int w = 0; w < n; ++w) s += __popc(a[w] | (c ? c[w] : 0u));
  return s;
}

// S = Q K^T from the tiles' K-major descriptors.
__device__ __forceinline__ void issue_s(uint32_t d, uint64_t dQ, uint64_t dK) {
  constexpr uint32_t idesc = idesc_bf16(BM, BN, 0, 0);
#pragma unroll
  for (int ks = 0; ks < HD / 16; ++ks) {
    const uint32_t off = (ks >> 2) * SLAB + (ks & 3) * 32;
    mma_ss(d, desc_add(dQ, off), desc_add(dK, off), idesc, ks > 0 ? 1u : 0u);
  }
}

// O += P V with P (bf16) in TMEM and V's MN-major descriptor.
__device__ __forceinline__ void issue_pv(uint32_t d, uint32_t pt, uint64_t dV, uint32_t acc0) {
  constexpr uint32_t idesc = idesc_bf16(BM, HD, 0, 1);
#pragma unroll
  for (int ks = 0; ks < BN / 16; ++ks)
    mma_ts(d, pt + ks * 8, desc_add(dV, ks * 2048), idesc, (acc0 || ks > 0) ? 1u : 0u);
}

// Maximum and minimum raw score over the live columns k0 .. k0 + 127 of one row.
template <bool MASKED>
__device__ __forceinline__ void row_range(const uint32_t (&v)[128], int k0, int4 ri, float& vmax,
                                          float& vmin) {
  float a0 = -INFINITY, a1 = -INFINITY, b0 = INFINITY, b1 = INFINITY;
#pragma unroll
  for (int e = 0; e < 128; e += 2) {
    float x = __uint_as_float(v[e]), y = __uint_as_float(v[e + 1]);
    float xl = x, yl = y;
    if constexpr (MASKED) {
      const int j0 = k0 + e, j1 = k0 + e + 1;
      const bool l0 = (j0 >= ri.x && j0 < ri.y) || j0 == ri.z;
      const bool l1 = (j1 >= ri.x && j1 < ri.y) || j1 == ri.z;
      x = l0 ? x : -INFINITY;
      y = l1 ? y : -INFINITY;
      xl = l0 ? xl : INFINITY;
      yl = l1 ? yl : INFINITY;
    }
    a0 = fmaxf(a0, x);
    a1 = fmaxf(a1, y);
    b0 = fminf(b0, xl);
    b1 = fminf(b1, yl);
  }
  vmax = fmaxf(a0, a1);
  vmin = fminf(b0, b1);
}

// Maximum (and, with NEED_MIN, minimum) raw score of a fully live row of 128
// columns, with three-input max / min in two independent chains each.
template <bool NEED_MIN>
__device__ __forceinline__ void row_range_full(const uint32_t (&v)[128], float& vmax, float& vmin) {
  float a0 = -INFINITY, a1 = -INFINITY, b0 = INFINITY, b1 = INFINITY;
#pragma unroll
  for (int e = 0; e < 128; e += 4) {
    const float x0 = __uint_as_float(v[e]), x1 = __uint_as_float(v[e + 1]);
    const float x2 = __uint_as_float(v[e + 2]), x3 = __uint_as_float(v[e + 3]);
    a0 = fmax3(a0, x0, x1);
    a1 = fmax3(a1, x2, x3);
    if constexpr (NEED_MIN) {
      b0 = fmin3(b0, x0, x1);
      b1 = fmin3(b1, x2, x3);
    }
  }
  vmax = fmaxf(a0, a1);
  vmin = NEED_MIN ? fminf(b0, b1) : vmax;
}

// 32 columns of P for the tanh cap when every |X * in| of the warp is within
// the polynomial's range: the first POLY_PAIRS column pairs evaluate tanh on the
// FMA pipe, the rest with tanh.approx; packed fp32x2 arithmetic throughout.
template <bool MASKED, int POLY_PAIRS>
__device__ __forceinline__ float p_chunk_tanh_fast(const uint32_t (&v)[32], uint32_t (&pk)[16],
                                                   const Xf& xf, float mul, float addm, int j0,
                                                   int4 ri, bool any) {
  const F2 in2 = f2(xf.in, xf.in), mul2 = f2(mul, mul), add2 = f2(addm, addm);
  F2 acc = f2(0.f, 0.f);
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const F2 u = f2_mul(f2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), in2);
    F2 t;
    if (e < POLY_PAIRS) {
      t = tanh_poly2(u);
    } else {
      float a, b;
      f2_split(u, a, b);
      t = f2(tanh_approx(a), tanh_approx(b));
    }
    float x0, x1;
    f2_split(f2_fma(t, mul2, add2), x0, x1);
    float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
    if constexpr (MASKED) {
      const int ja = j0 + 2 * e, jb = ja + 1;
      if (!(any && ((ja >= ri.x && ja < ri.y) || ja == ri.z))) p0 = 0.f;
      if (!(any && ((jb >= ri.x && jb < ri.y) || jb == ri.z))) p1 = 0.f;
    }
    acc = f2_add(acc, f2(p0, p1));
    pk[e] = pack_bf16x2(p0, p1);
  }
  float s0, s1;
  f2_split(acc, s0, s1);
  return s0 + s1;
}

// 32 columns of P = 2^(mul * f(X) + addm), packed to bf16 into pk; returns
// their sum.  (No TMEM access here: callers branch per row, and the warp-wide
// tcgen05 store must run after the branch has reconverged.)
template <int METHOD, bool MASKED>
__device__ __forceinline__ float p_chunk(const uint32_t (&v)[32], uint32_t (&pk)[16], const Xf& xf,
                                         float mul, float addm, int j0, int4 ri, bool any) {
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    float p0 = ex2_approx(fmaf(mul, cap_f<METHOD>(__uint_as_float(v[2 * e]), xf), addm));
    float p1 = ex2_approx(fmaf(mul, cap_f<METHOD>(__uint_as_float(v[2 * e + 1]), xf), addm));
    if constexpr (MASKED) {
      const int ja = j0 + 2 * e, jb = ja + 1;
      if (!(any && ((ja >= ri.x && ja < ri.y) || ja == ri.z))) p0 = 0.f;
      if (!(any && ((jb >= ri.x && jb < ri.y) || jb == ri.z))) p1 = 0.f;
    }
    s0 += p0;
    s1 += p1;
    pk[e] = pack_bf16x2(p0, p1);
  }
  return s0 + s1;
}

constexpr int kPolyPairs = 10;  // of 16 column pairs per chunk: tanh on the FMA pipe

template <int METHOD>
__device__ __forceinline__ float p_dispatch(bool full_any, bool poly, const uint32_t (&v)[32],
                                           uint32_t (&pk)[16], const Xf& xf, float mul, float addm,
                                           int j0, int4 ri, bool any) {
  if constexpr (METHOD == CAPATTN_CAP_TANH) {
    if (poly) {
      return full_any ? p_chunk_tanh_fast<false, kPolyPairs>(v, pk, xf, mul, addm, j0, ri, any)
                      : p_chunk_tanh_fast<true, kPolyPairs>(v, pk, xf, mul, addm, j0, ri, any);
    }
  }
  return full_any ? p_chunk<METHOD, false>(v, pk, xf, mul, addm, j0, ri, any)
                  : p_chunk<METHOD, true>(v, pk, xf, mul, addm, j0, ri, any);
}

template <int METHOD>
__global__ void __launch_bounds__(NTHREADS, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[16];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int hb = blockIdx.x;
  const int h = hb % p.Hq, b = hb / p.Hq;
  const int npair = (p.nq + 1) >> 1;
  const int pr = npair - 1 - (int)blockIdx.y;  // heaviest (latest) query tiles first
  const int qt0 = 2 * pr;
  const bool has1 = qt0 + 1 < p.nq;
  const int g = h / p.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ0 = base, sQ1 = base + TILE;
  const uint32_t sKV = base + 2 * TILE;  // stage s: K at sKV + s*2*TILE, V at + TILE

  const uint32_t bar_q = smem_u32(&bars[0]);
  const uint32_t bar_kfull = smem_u32(&bars[1]);   // + s*8
  const uint32_t bar_vfull = smem_u32(&bars[3]);   // + s*8
  const uint32_t bar_empty = smem_u32(&bars[5]);   // + s*8
  const uint32_t bar_sfull = smem_u32(&bars[7]);   // + tile*8
  const uint32_t bar_pfull = smem_u32(&bars[9]);   // + tile*8
  const uint32_t bar_final = smem_u32(&bars[11]);

  const uint32_t* map0 = p.qmap + ((size_t)b * p.nq + qt0) * p.wk;
  const uint32_t* map1 = has1 ? map0 + p.wk : nullptr;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar_q, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar_kfull + 8 * s, 1);
      mbar_init(bar_vfull + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_sfull + 8 * t, 1);
      mbar_init(bar_pfull + 8 * t, 4);
    }
    mbar_init(bar_final, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int n = count_union(map0, map1, p.wk);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (n > 0) {
      const bool leader = elect_one_sync();
      if (leader) {
        tma_prefetch_desc(&mq);
        tma_prefetch_desc(&mk);
        tma_prefetch_desc(&mv);
        mbar_expect_tx(bar_q, 2 * TILE);
        tma_load_4d(sQ0, &mq, bar_q, 0, h, qt0 * BM, b);
        tma_load_4d(sQ0 + SLAB, &mq, bar_q, 64, h, qt0 * BM, b);
        tma_load_4d(sQ1, &mq, bar_q, 0, h, qt0 * BM + BM, b);
        tma_load_4d(sQ1 + SLAB, &mq, bar_q, 64, h, qt0 * BM + BM, b);
      }
      __syncwarp();
      PairIter it(map0, map1, p.wk);
      int t, j = 0;
      bool a0, a1;
      while (it.next(t, a0, a1)) {
        const int s = j % NSTAGE, u = j / NSTAGE;
        if (u > 0 && !mbar_wait_warp(bar_empty + 8 * s, (u - 1) & 1, p.status, &abort_flag)) break;
        if (leader) {
          const uint32_t sK = sKV + s * 2 * TILE, sV = sK + TILE;
          mbar_expect_tx(bar_kfull + 8 * s, TILE);
          tma_load_4d(sK, &mk, bar_kfull + 8 * s, 0, g, t * BN, b);
          tma_load_4d(sK + SLAB, &mk, bar_kfull + 8 * s, 64, g, t * BN, b);
          mbar_expect_tx(bar_vfull + 8 * s, TILE);
          tma_load_4d(sV, &mv, bar_vfull + 8 * s, 0, g, t * BN, b);
          tma_load_4d(sV + SLAB, &mv, bar_vfull + 8 * s, 64, g, t * BN, b);
        }
        __syncwarp();
        ++j;
      }
      if (leader) {
        drain_wait(bar_q, 0);
        for (int jj = (j > NSTAGE ? j - NSTAGE : 0); jj < j; ++jj) {
          drain_wait(bar_kfull + 8 * (jj % NSTAGE), (jj / NSTAGE) & 1);
          drain_wait(bar_vfull + 8 * (jj % NSTAGE), (jj / NSTAGE) & 1);
        }
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (n > 0) {
      const bool leader = elect_one_sync();
      const uint64_t dQ0 = smem_desc(sQ0, 16, 1024), dQ1 = smem_desc(sQ1, 16, 1024);
      const uint64_t dKV = smem_desc(sKV, 16, 1024);      // K / V stages, K-major
      const uint64_t dKVmn = smem_desc(sKV, SLAB, 1024);  // the same, MN-major
      bool ok = mbar_wait_warp(bar_q, 0, p.status, &abort_flag);
      tc_fence_after();
      PairIter it(map0, map1, p.wk);
      int t;
      bool c0 = false, c1 = false;  // activity of the current tile
      bool n0 = false, n1 = false;  // activity of the next tile
      it.next(t, c0, c1);
      int pc0 = 0, pc1 = 0;         // p_full phases consumed per query tile
      uint32_t started0 = 0, started1 = 0;
      if (ok) ok = mbar_wait_warp(bar_kfull, 0, p.status, &abort_flag);
      if (ok) {
        tc_fence_after();
        if (leader) {
          if (c0) { issue_s(tmem, dQ0, dKV); mma_commit(bar_sfull); }
          if (c1) { issue_s(tmem + 128u, dQ1, dKV); mma_commit(bar_sfull + 8); }
        }
        __syncwarp();
      }
      for (int j = 0; ok && j < n; ++j) {
        const int s = j % NSTAGE;
        const uint32_t vo = (uint32_t)(s * 2 * TILE + TILE);
        n0 = n1 = false;
        const bool more = (j + 1 < n) && it.next(t, n0, n1);
        const int s1 = (j + 1) % NSTAGE;
        const uint32_t ko = (uint32_t)(s1 * 2 * TILE);
        if (!mbar_wait_warp(bar_vfull + 8 * s, (j / NSTAGE) & 1, p.status, &abort_flag)) break;
        if (c0) {
          if (!mbar_wait_warp(bar_pfull, pc0 & 1, p.status, &abort_flag)) break;
          ++pc0;
          tc_fence_after();
          if (leader) issue_pv(tmem + 256u, tmem, desc_add(dKVmn, vo), started0);
          __syncwarp();
          started0 = 1;
        }
        if (more) {
          if (!mbar_wait_warp(bar_kfull + 8 * s1, ((j + 1) / NSTAGE) & 1, p.status, &abort_flag)) break;
          tc_fence_after();
          if (n0 && leader) { issue_s(tmem, dQ0, desc_add(dKV, ko)); mma_commit(bar_sfull); }
          __syncwarp();
        }
        if (c1) {
          if (!mbar_wait_warp(bar_pfull + 8, pc1 & 1, p.status, &abort_flag)) break;
          ++pc1;
          tc_fence_after();
          if (leader) issue_pv(tmem + 384u, tmem + 128u, desc_add(dKVmn, vo), started1);
          __syncwarp();
          started1 = 1;
        }
        if (leader) {
          mma_commit(bar_empty + 8 * s);
          if (more && n1) { issue_s(tmem + 128u, dQ1, desc_add(dKV, ko)); mma_commit(bar_sfull + 8); }
        }
        __syncwarp();
        c0 = n0;
        c1 = n1;
      }
      // The MMA thread does not wait for its own commit here: the consumer
      // warps wait for it, and warp 1 re-checks it before freeing TMEM.
      if (leader) mma_commit(bar_final);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int tsel = (warp - 2) >> 2;          // query tile 0 or 1
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int i = (qt0 + tsel) * BM + r;
    const bool valid = i < p.L;
    const uint32_t s_base = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)tsel * 128u;
    const uint32_t o_base = tmem + ((uint32_t)(quarter * 32) << 16) + 256u + (uint32_t)tsel * 128u;
    const uint32_t my_sfull = bar_sfull + 8 * tsel, my_pfull = bar_pfull + 8 * tsel;
    const int4 ri = valid ? p.rowinfo[(size_t)b * p.L + i] : make_int4(0, 0, -1, 0);
    const float temp = (p.temp && valid) ? p.temp[(size_t)b * p.L + i] : 1.f;
    const bool neg = temp < 0.f;
    // the row minimum is needed for a negative temperature and for the range
    // check of the tanh polynomial
    const bool need_min = (METHOD == CAPATTN_CAP_TANH) || __any_sync(0xFFFFFFFFu, neg);
    const Xf xf = make_xf<METHOD>(p.cap, p.sm_scale);
    float rmul, radd;
    row_consts<METHOD>(p.cap, p.sm_scale, temp, &rmul, &radd);
    float m_use = -INFINITY, m_true = -INFINITY, lsum = 0.f;
    int cnt = 0;
    bool aborted = false;
    PairIter it(map0, map1, p.wk);
    int t;
    bool a0, a1;
    while (it.next(t, a0, a1)) {
      if (!(tsel == 0 ? a0 : a1)) continue;
      const int k0 = t * BN;
      if (!mbar_wait_warp(my_sfull, cnt & 1, p.status, &abort_flag)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const bool full = (ri.x <= k0) && (ri.y >= k0 + BN);
      // ---- pass 1: range of the live raw scores (one batched TMEM read)
      float vmax, vmin;
      {
        uint32_t v[128];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(s_base + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[c * 32]));
        tmem_wait_ld();
        if (!full)
          row_range<true>(v, k0, ri, vmax, vmin);
        else if (need_min)
          row_range_full<true>(v, vmax, vmin);
        else
          row_range_full<false>(v, vmax, vmin);
      }
      // Every cap is increasing: the logit maximum is the transform of the raw
      // maximum (of the minimum for a negative temperature).
      const float xsel = neg ? vmin : vmax;
      const float x_max =
          (vmax == -INFINITY) ? -INFINITY : fmaf(rmul, cap_f<METHOD>(xsel, xf), radd);
      // tanh on the FMA pipe when the whole warp's arguments are in range
      bool poly = false;
      if constexpr (METHOD == CAPATTN_CAP_TANH)
        poly = __all_sync(0xFFFFFFFFu, fmaxf(vmax, -vmin) * fabsf(xf.in) <= kTanhPolyMaxU);
      m_true = fmaxf(m_true, x_max);
      const float m_new = fmaxf(m_use, x_max);
      const bool resc = m_new > m_use + kRescaleThreshold;
      float alpha = 1.f;
      if (resc) {
        alpha = ex2_approx(m_use - m_new);
        m_use = m_new;
      }
      // ---- O rescale (PV of the previous live tile is complete)
      if (cnt > 0 && __any_sync(0xFFFFFFFFu, resc)) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(o_base + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(o_base + c * 32, o);
        }
      }
      // ---- pass 2: P = 2^(x - m_use), packed bf16 over S columns [0, 64).
      // The next chunk's TMEM load is issued before the current chunk is computed.
      const bool any = m_use != -INFINITY;
      const float addm = radd - (any ? m_use : 0.f);
      const bool fast = full && any;
      float psum = 0.f;
      {
        uint32_t va[32], vb[32], pk[16];
        tmem_ld32(s_base, va);
        tmem_wait_ld();
#pragma unroll 1
        for (int c = 0; c < 4; c += 2) {
          tmem_ld32(s_base + (c + 1) * 32, vb);
          psum += p_dispatch<METHOD>(fast, poly, va, pk, xf, rmul, addm, k0 + c * 32, ri, any);
          __syncwarp();
          tmem_st16(s_base + c * 16, pk);
          tmem_wait_ld();
          if (c + 2 < 4) tmem_ld32(s_base + (c + 2) * 32, va);
          psum += p_dispatch<METHOD>(fast, poly, vb, pk, xf, rmul, addm, k0 + (c + 1) * 32, ri, any);
          __syncwarp();
          tmem_st16(s_base + (c + 1) * 16, pk);
          tmem_wait_ld();
        }
      }
      lsum = lsum * alpha + psum;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(my_pfull);
      ++cnt;
    }
    // ---------------------------------------------------------- epilogue
    bool have_o = false;
    if (cnt > 0 && !aborted) {
      have_o = mbar_wait_warp(bar_final, 0, p.status, &abort_flag);
      tc_fence_after();
    }
    const bool live = lsum > 0.f;
    const float inv = live ? 1.f / lsum : 0.f;
    __nv_bfloat16* og = static_cast<__nv_bfloat16*>(p.o) + ((size_t)(b * p.L + i) * p.Hq + h) * HD;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      if (have_o) {
        tmem_ld32(o_base + c * 32, o);
        tmem_wait_ld();
      }
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float a = (have_o && live) ? __uint_as_float(o[2 * e]) * inv : 0.f;
        const float bb = (have_o && live) ? __uint_as_float(o[2 * e + 1]) * inv : 0.f;
        pk[e] = pack_bf16x2(a, bb);
      }
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(og + c * 32);
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
      }
    }
    if (valid) {
      const size_t rr = ((size_t)b * p.Hq + h) * p.L + i;
      p.lse[rr] = live ? (m_use + log2f(lsum)) * kLn2 : -INFINITY;
      if (p.m) p.m[rr] = live ? m_true * kLn2 : -INFINITY;
      if (p.l) p.l[rr] = live ? lsum * ex2_approx(m_use - m_true) : 0.f;
    }
  }
  __syncwarp();  // warps 0 and 1 reach the CTA barrier converged
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    // Every MMA has completed before TMEM is released (normally already
    // observed by the consumer warps; bounded non-suspending poll).
    if (lane == 0 && n > 0) mbar_poll(bar_final, 0);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int METHOD>
struct FwdTcLaunch {
  static cudaError_t run(const Params& p, cudaStream_t s) {
    CUtensorMap mq, mk, mv;
    cudaError_t e = make_bhld_map(&mq, p.q, p.B, p.L, p.Hq, HD, BM);
    if (e == cudaSuccess) e = make_bhld_map(&mk, p.k, p.B, p.L, p.Hkv, HD, BN);
    if (e == cudaSuccess) e = make_bhld_map(&mv, p.v, p.B, p.L, p.Hkv, HD, BN);
    if (e != cudaSuccess) return e;
    auto kern = fwd_tc_kernel<METHOD>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    prof_begin(CAPATTN_KERNEL_FWD, s);
    prof_count(CAPATTN_KERNEL_FWD, 1);
    kern<<<dim3(p.Hq * p.B, (p.nq + 1) / 2), NTHREADS, SMEM_BYTES, s>>>(mq, mk, mv, p);
    prof_end(CAPATTN_KERNEL_FWD, s);
    return cudaGetLastError();
  }
};

}  // namespace

cudaError_t launch_fwd_bf16(const Params& p, cudaStream_t s) {
  return dispatch_cap<FwdTcLaunch>(p.cap.method, p, s);
}

}  // namespace capattn

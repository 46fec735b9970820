// Pieces shared by the bf16 forward kernels (attn_fwd_tc.cu: two query tiles
// per CTA; attn_fwd1_tc.cu: one query tile per CTA, two CTAs per SM;
// attn_fwd2_tc.cu: one query tile per CTA with two score buffers):
// tile constants, the score and PV MMA sequences, and the softmax's per-chunk
// arithmetic (triton_kernels.py make_triton_forward_kernel's cap, temperature,
// mask and exp2-domain softmax).
#pragma once

#include <math.h>

#include "cap_math.cuh"
#include "capattn_internal.h"
#include "softmax_elem.cuh"
#include "tc_common.cuh"

namespace capattn {
namespace fwdtc {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int SLAB = 128 * 64 * 2;          // one [128][64] bf16 box
// A 128-row tile of head dim HD (64 or 128) is HD / 64 slabs.
template <int HD>
constexpr int tile_bytes() { return (HD / 64) * SLAB; }
constexpr float kRescaleThreshold = 8.0f;    // log2 units
// of the 16 column pairs of a 32-column pass, those whose tanh runs on the FMA
// pipe (polynomial) when the range allows; the others use MUFU
constexpr int kFwdPolyPairs = 12;
// Capped logits of a row lie in a window [x_hi - W, x_hi] (log2 units) known
// before any score is seen: W = 2 |mul| for tanh and soft_sign (|f| < 1), |mul|
// for ALSC (0 < f < 1).  With the fixed reference
//   m = x_hi - min(max(0, W - kSpanLo), kTopMax)
// every exponent x - m lies in [-max(kSpanLo, W - kTopMax), min(W - kSpanLo,
// kTopMax)]: at most 2^100 (no overflow in fp32 even summed over a row of 2^20
// keys) and, while W <= kSpanMax, at least 2^-124 (inside ex2's normal range,
// which ends at 2^-126).  Windows up to kSpanLo + kTopMax put the bottom at
// -kSpanLo; wider ones trade bottom margin for the same top.
constexpr float kSpanLo = 120.0f;
constexpr float kTopMax = 100.0f;
constexpr float kSpanMax = 224.0f;
__device__ __forceinline__ float fixed_reference(float x_hi, float span) {
  return x_hi - fminf(fmaxf(0.f, span - kSpanLo), kTopMax);
}

// S = Q K^T from the tiles' K-major descriptors.
template <int HD>
__device__ __forceinline__ void issue_s(uint32_t d, uint64_t dQ, uint64_t dK) {
  constexpr uint32_t idesc = idesc_bf16(BM, BN, 0, 0);
#pragma unroll
  for (int ks = 0; ks < HD / 16; ++ks) {
    const uint32_t off = (ks >> 2) * SLAB + (ks & 3) * 32;
    mma_ss(d, desc_add(dQ, off), desc_add(dK, off), idesc, ks > 0 ? 1u : 0u);
  }
}

// O += P V with P (bf16) in TMEM (key columns [0, 64) packed at pt + [0, 32),
// [64, 128) at pt + [64, 96)) and V's MN-major descriptor (N = HD).
template <int HD>
__device__ __forceinline__ void issue_pv(uint32_t d, uint32_t pt, uint64_t dV, uint32_t acc0) {
  constexpr uint32_t idesc = idesc_bf16(BM, HD, 0, 1);
#pragma unroll
  for (int ks = 0; ks < BN / 16; ++ks)
    mma_ts(d, pt + (ks < 4 ? 8 * ks : 64 + 8 * (ks - 4)), desc_add(dV, ks * 2048), idesc,
           (acc0 || ks > 0) ? 1u : 0u);
}

// Maximum and minimum raw score over the live columns k0 .. k0 + NC - 1 of one row.
template <bool MASKED, int NC>
__device__ __forceinline__ void row_range(const uint32_t (&v)[NC], int k0, int4 ri, float& vmax,
                                          float& vmin) {
  float a0 = -INFINITY, a1 = -INFINITY, b0 = INFINITY, b1 = INFINITY;
#pragma unroll
  for (int e = 0; e < NC; e += 2) {
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

// Maximum (and, with NEED_MIN, minimum) raw score of NC fully live columns, with three-input max / min in two independent chains each.
template <bool NEED_MIN, int NC>
__device__ __forceinline__ void row_range_full(const uint32_t (&v)[NC], float& vmax, float& vmin) {
  float a0 = -INFINITY, a1 = -INFINITY, b0 = INFINITY, b1 = INFINITY;
#pragma unroll
  for (int e = 0; e < NC; e += 4) {
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

// NP column pairs of P for the tanh cap with the folded polynomial (every
// |X * in| of the warp within the polynomial's range): x = X Q(X^2) + addm on
// the FMA pipe, 2^x on MUFU.
template <bool MASKED, int NP>
__device__ __forceinline__ float p_chunk_tanh_fold(const uint32_t (&v)[2 * NP], uint32_t (&pk)[NP],
                                                   const TanhFold& tf, float addm, uint32_t live) {
  const F2 add2 = f2(addm, addm);
  F2 acc = f2(0.f, 0.f);
#pragma unroll
  for (int e = 0; e < NP; ++e) {
    float x0, x1;
    f2_split(tanh_fold_eval(f2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), tf, add2),
             x0, x1);
    float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
    if constexpr (MASKED) {
      if (!(live & (1u << (2 * e)))) p0 = 0.f;
      if (!(live & (2u << (2 * e)))) p1 = 0.f;
    }
    acc = f2_add(acc, f2(p0, p1));
    pk[e] = pack_bf16x2(p0, p1);
  }
  float s0, s1;
  f2_split(acc, s0, s1);
  return s0 + s1;
}

// The same with the tanh of the last NP - NPOLY column pairs on MUFU
// (tanh.approx) instead of the FMA pipe, balancing the two pipes.
template <bool MASKED, int NP, int NPOLY>
__device__ __forceinline__ float p_chunk_tanh_mixed(const uint32_t (&v)[2 * NP], uint32_t (&pk)[NP],
                                                    const TanhFold& tf, const Xf& xf, float mul, float addm,
                                                    uint32_t live) {
  const F2 add2 = f2(addm, addm);
  F2 acc = f2(0.f, 0.f);
#pragma unroll
  for (int e = 0; e < NP; ++e) {
    float p0, p1;
    if (e < NPOLY) {
      float x0, x1;
      f2_split(tanh_fold_eval(f2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), tf, add2), x0, x1);
      p0 = ex2_approx(x0);
      p1 = ex2_approx(x1);
    } else {
      p0 = ex2_approx(fmaf(mul, cap_f<CAPATTN_CAP_TANH>(__uint_as_float(v[2 * e]), xf), addm));
      p1 = ex2_approx(fmaf(mul, cap_f<CAPATTN_CAP_TANH>(__uint_as_float(v[2 * e + 1]), xf), addm));
    }
    if constexpr (MASKED) {
      if (!(live & (1u << (2 * e)))) p0 = 0.f;
      if (!(live & (2u << (2 * e)))) p1 = 0.f;
    }
    acc = f2_add(acc, f2(p0, p1));
    pk[e] = pack_bf16x2(p0, p1);
  }
  float s0, s1;
  f2_split(acc, s0, s1);
  return s0 + s1;
}

// ALSC with the sigmoid on the FMA pipe (alsc_poly2; every |X| <= alsc_xmax):
// NP column pairs of P = 2^(mul * (f(X) - sigma(alpha beta)) + addm0), packed
// to bf16 into pk; returns their sum.  (addm0 = addm - radd of the plain form.)
template <bool MASKED, int NP>
__device__ __forceinline__ float p_chunk_alsc(const uint32_t (&v)[2 * NP], uint32_t (&pk)[NP],
                                              const CapConsts& cap, float mul, float addm0, uint32_t live) {
  const F2 mul2 = f2(mul, mul), add2 = f2(addm0, addm0);
  F2 acc = f2(0.f, 0.f);
#pragma unroll
  for (int e = 0; e < NP; ++e) {
    float x0, x1;
    const F2 d = alsc_poly2(f2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), cap);
    f2_split(f2_fma(mul2, d, add2), x0, x1);
    float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
    if constexpr (MASKED) {
      if (!(live & (1u << (2 * e)))) p0 = 0.f;
      if (!(live & (2u << (2 * e)))) p1 = 0.f;
    }
    acc = f2_add(acc, f2(p0, p1));
    pk[e] = pack_bf16x2(p0, p1);
  }
  float s0, s1;
  f2_split(acc, s0, s1);
  return s0 + s1;
}

// Whether every raw score of the warp's 16 columns is within the ALSC
// polynomial's range (warp-wide vote).
__device__ __forceinline__ bool sub_alsc_poly(const uint32_t (&v)[16], float xmax) {
  float am = 0.f;
#pragma unroll
  for (int e = 0; e < 16; e += 2) am = fmax3_abs(am, __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
  return __all_sync(0xFFFFFFFFu, am <= xmax);
}

// Whether every raw score of the warp's 32 columns is within the ALSC
// polynomial's range (warp-wide vote).
__device__ __forceinline__ bool quarter_alsc_poly(const uint32_t (&v)[32], float xmax) {
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    a0 = fmax3_abs(a0, __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
    a1 = fmax3_abs(a1, __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
  }
  return __all_sync(0xFFFFFFFFu, fmaxf(a0, a1) <= xmax);
}

// NP column pairs of P = 2^(mul * f(X) + addm), packed to bf16 into pk; returns
// their sum.  With MASKED, bit k of `live` says whether column k is live.  (No
// TMEM access here: callers branch per row, and the warp-wide tcgen05 store
// must run after the branch has reconverged.)
template <int METHOD, bool MASKED, int NP>
__device__ __forceinline__ float p_chunk(const uint32_t (&v)[2 * NP], uint32_t (&pk)[NP], const Xf& xf,
                                         float mul, float addm, uint32_t live) {
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int e = 0; e < NP; ++e) {
    float p0 = ex2_approx(fmaf(mul, cap_f<METHOD>(__uint_as_float(v[2 * e]), xf), addm));
    float p1 = ex2_approx(fmaf(mul, cap_f<METHOD>(__uint_as_float(v[2 * e + 1]), xf), addm));
    if constexpr (MASKED) {
      if (!(live & (1u << (2 * e)))) p0 = 0.f;
      if (!(live & (2u << (2 * e)))) p1 = 0.f;
    }
    s0 += p0;
    s1 += p1;
    pk[e] = pack_bf16x2(p0, p1);
  }
  return s0 + s1;
}

// Whether no row of the warp has a live key among the 16 columns j0 .. j0 + 15
// (live span [ri.x, ri.y) plus the extra column ri.z).  A warp-wide vote: every
// lane of the warp must call it.
__device__ __forceinline__ bool sub_dead(int4 ri, int j0) {
  const bool live = (ri.x < j0 + 16 && ri.y > j0 && ri.x < ri.y) || (ri.z >= j0 && ri.z < j0 + 16);
  return __all_sync(0xFFFFFFFFu, !live);
}

// Whether the warp may take the folded tanh polynomial for 16 raw scores
// (every |X * in| within its range); always false for the other caps.
template <int METHOD>
__device__ __forceinline__ bool sub_poly(const uint32_t (&v)[16], const TanhFold& tf, const Xf& xf) {
  if constexpr (METHOD == CAPATTN_CAP_TANH) {
    float am = 0.f;
#pragma unroll
    for (int e = 0; e < 16; e += 2) am = fmax3_abs(am, __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
    return __all_sync(0xFFFFFFFFu, tf.ok && am * fabsf(xf.in) <= kTanhPolyMaxU);
  }
  return false;
}

// 16 columns of P (8 packed pairs): masked or not, FMA-pipe tanh or not.
template <int METHOD>
__device__ __forceinline__ float p_dispatch(bool full_any, bool poly, const uint32_t (&v)[16],
                                           uint32_t (&pk)[8], const Xf& xf, const TanhFold& tf,
                                           float mul, float addm, int j0, int4 ri, bool any,
                                           const CapConsts* cap = nullptr) {
  if constexpr (METHOD == CAPATTN_CAP_ALSC) {
    // the sigmoid on the FMA pipe (the caller voted the range)
    if (poly && cap) {
      const float addm0 = addm + mul * cap->alsc_sb;
      if (full_any) return p_chunk_alsc<false, 8>(v, pk, *cap, mul, addm0, 0xFFFFu);
      return p_chunk_alsc<true, 8>(v, pk, *cap, mul, addm0, any ? live_bits16(ri, j0) : 0u);
    }
  }
  if (full_any) {
    if constexpr (METHOD == CAPATTN_CAP_TANH) {
      if (poly) return p_chunk_tanh_fold<false, 8>(v, pk, tf, addm, 0xFFFFu);
    }
    return p_chunk<METHOD, false, 8>(v, pk, xf, mul, addm, 0xFFFFu);
  }
  const uint32_t live = any ? live_bits16(ri, j0) : 0u;
  if constexpr (METHOD == CAPATTN_CAP_TANH) {
    if (poly) return p_chunk_tanh_fold<true, 8>(v, pk, tf, addm, live);
  }
  return p_chunk<METHOD, true, 8>(v, pk, xf, mul, addm, live);
}

// Live-column bits of the 32 columns j0 .. j0 + 31 of a row (bit k: column
// j0 + k is in [ri.x, ri.y) or equals ri.z).
__device__ __forceinline__ uint32_t live_bits32(int4 ri, int j0) {
  const int lo = min(max(ri.x - j0, 0), 32);
  const int hi = min(max(ri.y - j0, 0), 32);
  const uint32_t below_hi = hi >= 32 ? 0xFFFFFFFFu : ((1u << hi) - 1u);
  const uint32_t below_lo = lo >= 32 ? 0xFFFFFFFFu : ((1u << lo) - 1u);
  uint32_t bits = hi > lo ? (below_hi & ~below_lo) : 0u;
  const uint32_t ez = (uint32_t)(ri.z - j0);
  if (ez < 32u) bits |= 1u << ez;
  return bits;
}

// sub_dead and sub_poly over 32 columns.
__device__ __forceinline__ bool quarter_dead(int4 ri, int j0) {
  const bool live = (ri.x < j0 + 32 && ri.y > j0 && ri.x < ri.y) || (ri.z >= j0 && ri.z < j0 + 32);
  return __all_sync(0xFFFFFFFFu, !live);
}
template <int METHOD>
__device__ __forceinline__ bool quarter_poly(const uint32_t (&v)[32], const TanhFold& tf, const Xf& xf) {
  if constexpr (METHOD == CAPATTN_CAP_TANH) {
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      a0 = fmax3_abs(a0, __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
      a1 = fmax3_abs(a1, __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
    }
    return __all_sync(0xFFFFFFFFu, tf.ok && fmaxf(a0, a1) * fabsf(xf.in) <= kTanhPolyMaxU);
  }
  return false;
}

// 32 columns of P (16 packed pairs): masked or not, FMA-pipe tanh or not.
template <int METHOD>
__device__ __forceinline__ float p_dispatch32(bool full_any, bool poly, const uint32_t (&v)[32],
                                             uint32_t (&pk)[16], const Xf& xf, const TanhFold& tf,
                                             float mul, float addm, int j0, int4 ri, bool any) {
  if (full_any) {
    if constexpr (METHOD == CAPATTN_CAP_TANH) {
      if (poly) return p_chunk_tanh_mixed<false, 16, kFwdPolyPairs>(v, pk, tf, xf, mul, addm, 0xFFFFFFFFu);
    }
    return p_chunk<METHOD, false, 16>(v, pk, xf, mul, addm, 0xFFFFFFFFu);
  }
  const uint32_t live = any ? live_bits32(ri, j0) : 0u;
  if constexpr (METHOD == CAPATTN_CAP_TANH) {
    if (poly) return p_chunk_tanh_mixed<true, 16, kFwdPolyPairs>(v, pk, tf, xf, mul, addm, live);
  }
  return p_chunk<METHOD, true, 16>(v, pk, xf, mul, addm, live);
}

}  // namespace fwdtc
}  // namespace capattn

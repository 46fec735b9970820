// Per-element score transforms shared by the tcgen05 kernels.
//
// The log2-domain logit of a raw score X = <Q_i, K_j> is
//     x = temp_i * cap(sm_scale * X) * log2(e)  =  mul_i * f(X * in + bias) + add_i
// with global constants (in, bias) and per-row constants (mul_i, add_i), where
// f is the shape of the cap (mosaic_backward.py _apply_cap_mosaic):
//   none      : f(u) = u                   in = 1,                      mul = sm_scale * temp * log2e
//   tanh      : f(u) = tanh(u)             in = sm_scale / cap,         mul = cap * temp * log2e
//   soft_sign : f(u) = u / (1 + |u|)       in = sm_scale / cap,         mul = cap * temp * log2e
//   alsc      : f(u) = 1 / (1 + 2^-u)      in = sm_scale * alpha / cap * log2e, bias = alpha * beta * log2e,
//                                          mul = temp * log2e * cap / denom, add = -mul * sigma(alpha beta)
// Every cap is increasing in X, so for temp_i >= 0 the row maximum of x is the
// transform of the row maximum of X (of the minimum for temp_i < 0): the
// forward finds the extreme raw score with one max pass.
//
// The derivative of the cap with respect to s = sm_scale * X, in terms of the
// same intermediate: none 1; tanh 1 - tanh^2; soft_sign 1 / (1 + |u|)^2;
// alsc (alpha / denom) * sigma (1 - sigma).  The backward folds the constant
// factor (alpha / denom for alsc) into dscale = sm_scale * temp * factor.
//
// tanh uses the tanh.approx instruction (max relative error measured ~1e-5 on
// GB300: an absolute logit error below cap * 1e-5); the others use ex2.approx
// and rcp.approx.
#pragma once

#include "capattn_internal.h"
#include "tc_common.cuh"

namespace capattn {

constexpr float kL2E = 1.4426950408889634f;

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Xf {  // global part of the transform
  float in, bias;
};

template <int METHOD>
__device__ __forceinline__ Xf make_xf(const CapConsts& k, float sm_scale) {
  Xf x;
  x.bias = 0.f;
  if constexpr (METHOD == CAPATTN_CAP_TANH || METHOD == CAPATTN_CAP_SOFT_SIGN) {
    x.in = sm_scale * k.inv_cap;
  } else if constexpr (METHOD == CAPATTN_CAP_ALSC) {
    x.in = sm_scale * k.alsc_a * kL2E;
    x.bias = k.alsc_b * kL2E;
  } else {
    x.in = 1.f;
  }
  return x;
}

// Per-row multiplier and offset of the transform.
template <int METHOD>
__device__ __forceinline__ void row_consts(const CapConsts& k, float sm_scale, float temp,
                                           float* mul, float* add) {
  if constexpr (METHOD == CAPATTN_CAP_TANH || METHOD == CAPATTN_CAP_SOFT_SIGN) {
    *mul = k.cap * temp * kL2E;
    *add = 0.f;
  } else if constexpr (METHOD == CAPATTN_CAP_ALSC) {
    *mul = temp * kL2E * k.alsc_out;
    *add = -(*mul) * k.alsc_sb;
  } else {
    *mul = sm_scale * temp * kL2E;
    *add = 0.f;
  }
}

// sm_scale * temp * (constant factor of the cap derivative).
template <int METHOD>
__device__ __forceinline__ float row_dscale(const CapConsts& k, float sm_scale, float temp) {
  if constexpr (METHOD == CAPATTN_CAP_ALSC) return sm_scale * temp * k.alsc_dout;
  return sm_scale * temp;
}

// f(X * in + bias)
template <int METHOD>
__device__ __forceinline__ float cap_f(float X, const Xf& xf) {
  if constexpr (METHOD == CAPATTN_CAP_TANH) {
    return tanh_approx(X * xf.in);
  } else if constexpr (METHOD == CAPATTN_CAP_SOFT_SIGN) {
    const float u = X * xf.in;
    return u * rcp_approx(1.0f + fabsf(u));
  } else if constexpr (METHOD == CAPATTN_CAP_ALSC) {
    return rcp_approx(1.0f + ex2_approx(-fmaf(X, xf.in, xf.bias)));
  } else {
    return X;
  }
}

// f and the variable part of its derivative.
template <int METHOD>
__device__ __forceinline__ float cap_f_d(float X, const Xf& xf, float* d) {
  if constexpr (METHOD == CAPATTN_CAP_TANH) {
    const float t = tanh_approx(X * xf.in);
    *d = fmaf(-t, t, 1.0f);
    return t;
  } else if constexpr (METHOD == CAPATTN_CAP_SOFT_SIGN) {
    const float u = X * xf.in;
    const float r = rcp_approx(1.0f + fabsf(u));
    *d = r * r;
    return u * r;
  } else if constexpr (METHOD == CAPATTN_CAP_ALSC) {
    const float sg = rcp_approx(1.0f + ex2_approx(-fmaf(X, xf.in, xf.bias)));
    *d = sg - sg * sg;
    return sg;
  } else {
    *d = 1.0f;
    return X;
  }
}

// Which of the 16 columns j0 .. j0 + 15 are live for a row with live span
// [ri.x, ri.y) and extra live column ri.z, as bits 0 .. 15 (computed once per
// 16 columns, so that each element's mask test is a single bit test).
__device__ __forceinline__ uint32_t live_bits16(int4 ri, int j0) {
  const int lo = min(max(ri.x - j0, 0), 16);
  const int hi = min(max(ri.y - j0, 0), 16);
  uint32_t bits = hi > lo ? ((1u << hi) - 1u) & ~((1u << lo) - 1u) : 0u;
  const uint32_t ez = (uint32_t)(ri.z - j0);
  if (ez < 16u) bits |= 1u << ez;
  return bits;
}

// max(acc, |a|, |b|) with the three-input max instruction.
__device__ __forceinline__ float fmax3_abs(float acc, float a, float b) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(acc), "f"(fabsf(a)), "f"(fabsf(b)));
  return r;
}

// Three-input max / min.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// ---------------------------------------------------------------- packed fp32
// Two fp32 lanes in one 64-bit register pair (fma/mul/add .f32x2).
struct F2 {
  unsigned long long v;
};
__device__ __forceinline__ F2 f2(float a, float b) {
  F2 r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r.v) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_split(F2 x, float& a, float& b) {
  asm("mov.b64 {%0,%1}, %2;" : "=f"(a), "=f"(b) : "l"(x.v));
}
__device__ __forceinline__ F2 f2_mul(F2 a, F2 b) {
  F2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
  F2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ F2 f2_fma(F2 a, F2 b, F2 c) {
  F2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
  return r;
}

// ---------------------------------------------------------------- tanh on the FMA pipe
// tanh(u) = u + u^3 (c0 + w (c1 + w (c2 + w c3))), w = u^2, for |u| <= 0.5:
// coefficients from csrc/fit_tanh_poly.py (max |error| 2.5e-8 in fp32, below
// the tanh.approx instruction's error).  Kernels take this path only when a
// whole warp's arguments are inside the range, and then split each chunk
// between this FMA-pipe form and the MUFU instruction to balance the pipes.
constexpr float kTanhPolyMaxU = 0.5f;
constexpr float kTanhC0 = -0.333330512f;
constexpr float kTanhC1 = 0.133239388f;
constexpr float kTanhC2 = -0.0529243536f;
constexpr float kTanhC3 = 0.0170059651f;

// The same polynomial with the argument scale `in` and an output scale `mul`
// folded into its coefficients: mul * tanh(in * X) = X * Q(X^2), Q(z) = K0 + z (K1 + z (K2 + z (K3 + z K4))),
// K0 = mul in, K(k+1) = mul c_k in^(2k+3).  Evaluating Q in fp32 keeps the
// result within 2e-7 * mul of mul * tanh (tests/test_tanh_poly.py bounds
// it); the coefficients stay normal floats while |K4| >= 1e-30, which callers
// check before taking this form.
struct TanhFold {
  F2 k0, k1, k2, k3, k4;
  bool ok;  // coefficients usable (no underflow)
};
__device__ __forceinline__ TanhFold tanh_fold(float in, float mul) {
  const float w = in * in;
  const float a0 = mul * in;
  const float a1 = a0 * w * kTanhC0;
  const float a2 = a0 * w * w * kTanhC1;
  const float a3 = a0 * w * w * w * kTanhC2;
  const float a4 = a0 * w * w * w * w * kTanhC3;
  TanhFold t;
  t.k0 = f2(a0, a0);
  t.k1 = f2(a1, a1);
  t.k2 = f2(a2, a2);
  t.k3 = f2(a3, a3);
  t.k4 = f2(a4, a4);
  t.ok = (mul == 0.f) || (fabsf(a4) >= 1e-30f);
  return t;
}
// x = X * Q(X^2) + add for a pair of raw scores.
__device__ __forceinline__ F2 tanh_fold_eval(F2 X, const TanhFold& t, F2 add) {
  const F2 z = f2_mul(X, X);
  F2 q = f2_fma(t.k4, z, t.k3);
  q = f2_fma(q, z, t.k2);
  q = f2_fma(q, z, t.k1);
  q = f2_fma(q, z, t.k0);
  return f2_fma(X, q, add);
}

// ALSC's sigmoid on the FMA pipe for a pair of raw scores with |X| <= k.alsc_xmax:
// sigma(z) - sigma(alpha beta) = X * sum_j alsc_gu[j] X^j (host-fitted polynomial).
__device__ __forceinline__ F2 alsc_poly2(F2 X, const CapConsts& k) {
  F2 q = f2(k.alsc_gu[6], k.alsc_gu[6]);
  q = f2_fma(q, X, f2(k.alsc_gu[5], k.alsc_gu[5]));
  q = f2_fma(q, X, f2(k.alsc_gu[4], k.alsc_gu[4]));
  q = f2_fma(q, X, f2(k.alsc_gu[3], k.alsc_gu[3]));
  q = f2_fma(q, X, f2(k.alsc_gu[2], k.alsc_gu[2]));
  q = f2_fma(q, X, f2(k.alsc_gu[1], k.alsc_gu[1]));
  q = f2_fma(q, X, f2(k.alsc_gu[0], k.alsc_gu[0]));
  return f2_mul(X, q);
}

__device__ __forceinline__ F2 tanh_poly2(F2 u) {
  const F2 w = f2_mul(u, u);
  F2 p = f2_fma(f2(kTanhC3, kTanhC3), w, f2(kTanhC2, kTanhC2));
  p = f2_fma(p, w, f2(kTanhC1, kTanhC1));
  p = f2_fma(p, w, f2(kTanhC0, kTanhC0));
  return f2_fma(f2_mul(u, w), p, u);
}

}  // namespace capattn

// Logit caps and their derivatives in fp32 (mosaic_backward.py
// _apply_cap_mosaic for the forward of each method; the derivative is the exact
// derivative of that forward).
//
//   tanh      : c = cap * tanh(s / cap),            c' = 1 - tanh^2
//   soft_sign : c = s * r, r = 1 / (1 + |s| / cap), c' = r^2
//   alsc      : c = (cap / denom) * (sig(z) - sig(ab)), z = (alpha / cap) s + ab,
//               c' = (alpha / denom) * sig(z) (1 - sig(z))
//
// tanh and the logistic function are written through exp2 and a reciprocal:
// tanh(x) = sign(x) * (1 - 2 / (1 + e^{2|x|})), sig(z) = 1 / (1 + e^{-z}).  Both
// forms have an absolute error of a few fp32 ulps of 1, which the output scale
// (cap, or cap / denom) turns into an absolute logit error far below the
// tolerances; e^{2|x|} overflowing to +inf gives exactly 1.
#pragma once

#include "capattn_internal.h"
#include "tc_common.cuh"

namespace capattn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int METHOD>
__device__ __forceinline__ float cap_value(float s, const CapConsts& k) {
  if constexpr (METHOD == CAPATTN_CAP_TANH) {
    const float ax = fabsf(s) * k.inv_cap;
    const float e = ex2_approx(ax * (2.0f * kLog2e));
    const float t = 1.0f - 2.0f * rcp_approx(1.0f + e);
    return copysignf(k.cap * t, s);
  } else if constexpr (METHOD == CAPATTN_CAP_SOFT_SIGN) {
    const float r = rcp_approx(1.0f + fabsf(s) * k.inv_cap);
    return s * r;
  } else if constexpr (METHOD == CAPATTN_CAP_ALSC) {
    const float z = fmaf(s, k.alsc_a, k.alsc_b);
    const float sg = rcp_approx(1.0f + ex2_approx(-z * kLog2e));
    return k.alsc_out * (sg - k.alsc_sb);
  } else {
    return s;
  }
}

// Returns cap(s) and writes cap'(s) to *d.
template <int METHOD>
__device__ __forceinline__ float cap_value_grad(float s, const CapConsts& k, float* d) {
  if constexpr (METHOD == CAPATTN_CAP_TANH) {
    const float ax = fabsf(s) * k.inv_cap;
    const float e = ex2_approx(ax * (2.0f * kLog2e));
    const float t = 1.0f - 2.0f * rcp_approx(1.0f + e);
    *d = fmaf(-t, t, 1.0f);
    return copysignf(k.cap * t, s);
  } else if constexpr (METHOD == CAPATTN_CAP_SOFT_SIGN) {
    const float r = rcp_approx(1.0f + fabsf(s) * k.inv_cap);
    *d = r * r;
    return s * r;
  } else if constexpr (METHOD == CAPATTN_CAP_ALSC) {
    const float z = fmaf(s, k.alsc_a, k.alsc_b);
    const float sg = rcp_approx(1.0f + ex2_approx(-z * kLog2e));
    *d = k.alsc_dout * sg * (1.0f - sg);
    return k.alsc_out * (sg - k.alsc_sb);
  } else {
    *d = 1.0f;
    return s;
  }
}

// Dispatch a templated functor on the runtime cap method.
template <template <int> class F, typename... Args>
cudaError_t dispatch_cap(int method, Args&&... args) {
  switch (method) {
    case CAPATTN_CAP_TANH: return F<CAPATTN_CAP_TANH>::run(args...);
    case CAPATTN_CAP_SOFT_SIGN: return F<CAPATTN_CAP_SOFT_SIGN>::run(args...);
    case CAPATTN_CAP_ALSC: return F<CAPATTN_CAP_ALSC>::run(args...);
    default: return F<CAPATTN_CAP_NONE>::run(args...);
  }
}

}  // namespace capattn

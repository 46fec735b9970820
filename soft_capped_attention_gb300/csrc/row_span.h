// Per-query-row live key set, shared by the host visit-map code and the device
// pre-pass.
//
// For query row i the live keys j are those that pass every enabled mask
// (triton_kernels.py forward kernel: segment equality, causal i >= j, window
// j > i - window_len; mosaic_backward.py ranker_mask_mosaic_kv_q: history keys
// for history and candidate queries, plus the candidate query itself).  With
// segment ids non-decreasing along the row, that set is always one interval
// [lo, hi) plus at most one extra key e (the candidate's own position):
//   * causal gives j < i + 1, the window j >= i - window_len + 1, the segment
//     run of i gives [first, last + 1) of equal ids;
//   * the ranker restricts the interval to the history range [hl, hu) for rows
//     in history or candidates (empty for all other rows) and adds e = i for a
//     candidate row; e = i passes the causal, window and segment tests by
//     construction (i >= i, i > i - window_len for window_len > 0, seg_i == seg_i).
#pragma once

#ifdef __CUDACC__
#define CAPATTN_HD __host__ __device__ __forceinline__
#else
#define CAPATTN_HD inline
#endif

#include <stdint.h>

namespace capattn {

struct RowSpan {
  int32_t lo;  // first live key of the interval
  int32_t hi;  // one past the last live key (hi <= lo: empty interval)
  int32_t e;   // extra live key outside [lo, hi), or -1
};

CAPATTN_HD int32_t imax32(int32_t a, int32_t b) { return a > b ? a : b; }
CAPATTN_HD int32_t imin32(int32_t a, int32_t b) { return a < b ? a : b; }

// seg_first / seg_last1: the run of equal segment ids around i ([0, L) without segments).
// has_bounds: ranker mask on, with (hl, hu, cl, cu) already clamped to [0, L].
CAPATTN_HD RowSpan row_span(int32_t i, int32_t L, int32_t causal, int32_t window_len,
                            int32_t seg_first, int32_t seg_last1, int32_t has_bounds, int32_t hl,
                            int32_t hu, int32_t cl, int32_t cu) {
  int32_t lo = seg_first, hi = imin32(seg_last1, L);
  if (causal) hi = imin32(hi, i + 1);
  if (window_len > 0) lo = imax32(lo, i - window_len + 1);
  int32_t e = -1;
  if (has_bounds) {
    const bool in_h = (i >= hl) && (i < hu);
    const bool in_c = (i >= cl) && (i < cu);
    if (in_h || in_c) {
      lo = imax32(lo, hl);
      hi = imin32(hi, hu);
    } else {
      hi = lo;
    }
    if (in_c) e = i;
  }
  if (hi < lo) hi = lo;
  if (e >= lo && e < hi) e = -1;
  RowSpan r;
  r.lo = lo;
  r.hi = hi;
  r.e = e;
  return r;
}

CAPATTN_HD bool span_live(const RowSpan& r, int32_t j) {
  return (j >= r.lo && j < r.hi) || j == r.e;
}

// First index k in [0, n) with a[k] >= x (a non-decreasing).
CAPATTN_HD int32_t lower_bound_i32(const int32_t* a, int32_t n, int32_t x) {
  int32_t lo = 0, hi = n;
  while (lo < hi) {
    int32_t mid = (lo + hi) >> 1;
    if (a[mid] < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// First index k in [0, n) with a[k] > x (a non-decreasing).
CAPATTN_HD int32_t upper_bound_i32(const int32_t* a, int32_t n, int32_t x) {
  int32_t lo = 0, hi = n;
  while (lo < hi) {
    int32_t mid = (lo + hi) >> 1;
    if (a[mid] <= x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

}  // namespace capattn

// Pre-pass kernels: per-row live key spans, block visit maps, and the delta
// pre-pass of the backward (mosaic_backward.py make_preprocess_backward_kernel,
// with delta = rowsum(O * dO) on the normalised O and the unscaled dO).
#include <cuda_bf16.h>

#include "capattn_internal.h"
#include "row_span.h"

namespace capattn {

__device__ __forceinline__ void set_bit_range(uint32_t* bm, int a, int c) {
  for (int w = a >> 5; w <= (c >> 5); ++w) {
    const int lo = (w == (a >> 5)) ? (a & 31) : 0;
    const int hi = (w == (c >> 5)) ? (c & 31) : 31;
    const uint32_t upto = hi == 31 ? 0xFFFFFFFFu : ((1u << (hi + 1)) - 1u);
    atomicOr(&bm[w], upto & ~((1u << lo) - 1u));
  }
}

// One CTA per (query tile, b).  Per row i of the tile: the run of equal segment
// ids around i (binary search on a non-decreasing row), the clamped ranker
// bounds and the row's live key span, written to rowinfo.  Per tile: the OR of
// the KV tiles its rows touch, and the range of KV tiles every row covers
// completely (the tiles in which no pair needs a mask test); a tile with rows
// past L has no fully covered KV tile.
// The first CTA zeroes the work counter of the persistent forward.
// The CTA of every 32nd query tile also clears the word of the key-tile map
// that holds the bits of query tiles [qt, qt + 32), for every KV tile: the
// bf16 dQ kernel ORs each query tile's bits into that map later (kmap_kernel
// instead writes whole words).
__global__ void rowmap_kernel(Params p) {
  extern __shared__ uint32_t bm[];
  __shared__ int full_lo, full_hi;
  pdl_trigger();
  pdl_wait();
  const int qt = blockIdx.x, b = blockIdx.y;
  if ((qt | b | threadIdx.x) == 0) *p.fwd_work = 0u;  // the persistent forward's work counter
  for (int w = threadIdx.x; w < p.wk; w += blockDim.x) bm[w] = 0u;
  if ((qt & 31) == 0)
    for (int kt = threadIdx.x; kt < p.nk; kt += blockDim.x)
      p.kmap[((size_t)b * p.nk + kt) * p.wq + (qt >> 5)] = 0u;
  if (threadIdx.x == 0) {
    full_lo = 0;
    full_hi = p.nk;
  }
  int32_t hl = 0, hu = 0, cl = 0, cu = 0;
  if (p.bounds) {
    const int4 bd = reinterpret_cast<const int4*>(p.bounds)[b];
    if (qt == 0 && threadIdx.x == 0 &&
        !(bd.x >= 0 && bd.x <= bd.y && bd.y <= p.L && bd.z >= 0 && bd.z <= bd.w && bd.w <= p.L))
      atomicOr(p.status, kStatusBadBoundsBit);
    hl = imin32(imax32(bd.x, 0), p.L);
    hu = imin32(imax32(bd.y, 0), p.L);
    cl = imin32(imax32(bd.z, 0), p.L);
    cu = imin32(imax32(bd.w, 0), p.L);
  }
  __syncthreads();
  for (int t = threadIdx.x; t < p.block_q; t += blockDim.x) {
    const int i = qt * p.block_q + t;
    int fa = 1, fb = 0;  // empty
    if (i < p.L) {
      int32_t first = 0, last1 = p.Lk;
      if (p.seg) {
        const int32_t* srow = p.seg + (size_t)b * p.L;
        const int32_t x = srow[i];
        if (i > 0 && srow[i - 1] > x) atomicOr(p.status, kStatusBadSegmentsBit);
        first = lower_bound_i32(srow, p.L, x);
        last1 = upper_bound_i32(srow, p.L, x);
      }
      const RowSpan r = row_span(i, p.Lk, p.causal, p.window_len, first, last1, p.bounds ? 1 : 0, hl,
                                 hu, cl, cu);
      p.rowinfo[(size_t)b * p.L + i] = make_int4(r.lo, r.hi, r.e, 0);
      if (r.hi > r.lo) {
        set_bit_range(bm, r.lo / p.block_kv, (r.hi - 1) / p.block_kv);
        fa = (r.lo + p.block_kv - 1) / p.block_kv;
        fb = r.hi / p.block_kv;
      }
      if (r.e >= 0) {
        const int kt = r.e / p.block_kv;
        atomicOr(&bm[kt >> 5], 1u << (kt & 31));
      }
    }
    atomicMax(&full_lo, fa);
    atomicMin(&full_hi, fb);
  }
  __syncthreads();
  for (int w = threadIdx.x; w < p.wk; w += blockDim.x)
    p.qmap[((size_t)b * p.nq + qt) * p.wk + w] = bm[w];
  if (threadIdx.x == 0) p.qfull[(size_t)b * p.nq + qt] = make_int2(full_lo, full_hi);
}

// One CTA per (KV tile, b): transpose of the query-tile map.
__global__ void kmap_kernel(Params p) {
  pdl_trigger();
  pdl_wait();
  const int kt = blockIdx.x, b = blockIdx.y;
  for (int w = threadIdx.x; w < p.wq; w += blockDim.x) {
    uint32_t word = 0u;
    for (int bit = 0; bit < 32; ++bit) {
      const int qt = w * 32 + bit;
      if (qt >= p.nq) break;
      const uint32_t src = p.qmap[((size_t)b * p.nq + qt) * p.wk + (kt >> 5)];
      word |= ((src >> (kt & 31)) & 1u) << bit;
    }
    p.kmap[((size_t)b * p.nk + kt) * p.wq + w] = word;
  }
}

cudaError_t launch_prepass(const Params& p, bool build_rows, bool build_kmap, cudaStream_t s) {
  if (!build_rows && !build_kmap) return cudaSuccess;
  prof_begin(CAPATTN_KERNEL_PREPASS, s);
  prof_count(CAPATTN_KERNEL_PREPASS, (build_rows ? 1 : 0) + (build_kmap ? 1 : 0));
  cudaError_t e = cudaSuccess;
  if (build_rows) {
    dim3 g1(p.nq, p.B);
    e = launch_pdl(rowmap_kernel, g1, dim3(128), p.wk * sizeof(uint32_t), s, p);
    if (e != cudaSuccess) return e;
  }
  if (build_kmap) {
    dim3 g3(p.nk, p.B);
    e = launch_pdl(kmap_kernel, g3, dim3(32), 0, s, p);
    if (e != cudaSuccess) return e;
  }
  prof_end(CAPATTN_KERNEL_PREPASS, s);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ delta
// fp32 inputs: one warp per (b, i, h) row of D elements, delta[b, h, i] =
// sum_d O * dO.  (The bf16 path computes delta inside the dQ kernel.)
template <int D>
__global__ void delta_kernel(Params p) {
  pdl_trigger();
  pdl_wait();
  constexpr int VEC = D / 32;
  const long long row = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  const long long nrows = (long long)p.B * p.L * p.Hq;
  if (row >= nrows) return;
  const float* o = static_cast<const float*>(p.o) + row * D + lane * VEC;
  const float* g = static_cast<const float*>(p.dO) + row * D + lane * VEC;
  float acc = 0.f;
#pragma unroll
  for (int t = 0; t < VEC; ++t) acc = fmaf(o[t], g[t], acc);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
  if (lane == 0) {
    const int h = (int)(row % p.Hq);
    const long long bi = row / p.Hq;
    const int i = (int)(bi % p.L);
    const int b = (int)(bi / p.L);
    p.delta[((size_t)b * p.Hq + h) * p.L + i] = acc;
  }
}

cudaError_t launch_delta_fp32(const Params& p, cudaStream_t s) {
  const long long nrows = (long long)p.B * p.L * p.Hq;
  const int warps = 8;
  const unsigned grid = (unsigned)((nrows + warps - 1) / warps);
  prof_begin(CAPATTN_KERNEL_DELTA, s);
  prof_count(CAPATTN_KERNEL_DELTA, 1);
  const cudaError_t e = p.D == 64 ? launch_pdl(delta_kernel<64>, dim3(grid), dim3(warps * 32), 0, s, p)
                                  : launch_pdl(delta_kernel<128>, dim3(grid), dim3(warps * 32), 0, s, p);
  if (e != cudaSuccess) return e;
  prof_end(CAPATTN_KERNEL_DELTA, s);
  return cudaGetLastError();
}

// bf16, stored-dX backward: one CTA per (query head, half query tile, b) of 8
// warps, the head fastest: delta[b, h, i] = sum_d O * dO in fp32.  A row's D values are read by
// D / 8 lanes, 16 bytes each, so a warp covers 32 / (D / 8) rows per load and
// the CTA its 64 rows in 64 / (8 * that) rounds; every round's loads are issued
// before any arithmetic (rows past L read row L - 1 and are dropped).
// The first CTA of each query tile of head 0 also ORs the tile's bit into the word of every KV
// tile the tile visits (the key-tile map for the dK/dV kernel, which runs next;
// rowmap_kernel cleared those words), and the first thread zeroes the work
// counter of the dQ GEMM that follows.
template <int D>
__global__ void delta_bf16_kernel(Params p) {
  pdl_trigger();
  pdl_wait();
  constexpr int LPR = D / 8;            // lanes per row
  constexpr int RPW = 32 / LPR;         // rows per warp and round
  constexpr int ROUNDS = 64 / (8 * RPW);
  // the head is the fastest grid index: CTAs that run together read the
  // same rows of every head, one contiguous region of O and dO
  const int h = (int)(blockIdx.x % (unsigned)p.Hq), rest = (int)(blockIdx.x / (unsigned)p.Hq);
  const int qt = rest >> 1, half = rest & 1, b = blockIdx.y;
  const int row0 = qt * 128 + 64 * half;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((blockIdx.x | b | threadIdx.x) == 0) *p.dq_work = 0u;  // the dQ GEMM's work counter
  const uint4* o = static_cast<const uint4*>(p.o);
  const uint4* g = static_cast<const uint4*>(p.dO);
  const int sub = lane / LPR, part = lane % LPR;
  uint4 a[ROUNDS], c[ROUNDS];
#pragma unroll
  for (int k = 0; k < ROUNDS; ++k) {
    const int i = imin32(row0 + (k * 8 + warp) * RPW + sub, p.L - 1);
    const size_t off = (((size_t)b * p.L + i) * p.Hq + h) * LPR + part;
    a[k] = o[off];
    c[k] = g[off];
  }
#pragma unroll
  for (int k = 0; k < ROUNDS; ++k) {
    const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a[k]);
    const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&c[k]);
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 u = __bfloat1622float2(x[e]), v = __bfloat1622float2(y[e]);
      acc = fmaf(u.x, v.x, fmaf(u.y, v.y, acc));
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    const int i = row0 + (k * 8 + warp) * RPW + sub;
    if (part == 0 && i < p.L) p.delta[((size_t)b * p.Hq + h) * p.L + i] = acc;
  }
  if (h == 0 && warp == 0 && half == 0) {
    const uint32_t* map = p.qmap + ((size_t)b * p.nq + qt) * p.wk;
    for (int w = lane; w < p.wk; w += 32) {
      uint32_t bits = map[w];
      while (bits) {
        const int kt = 32 * w + __ffs(bits) - 1;
        bits &= bits - 1u;
        atomicOr(&p.kmap[((size_t)b * p.nk + kt) * p.wq + (qt >> 5)], 1u << (qt & 31));
      }
    }
  }
}

cudaError_t launch_delta_bf16(const Params& p, cudaStream_t s) {
  prof_begin(CAPATTN_KERNEL_DELTA, s);
  prof_count(CAPATTN_KERNEL_DELTA, 1);
  const dim3 grid((unsigned)(p.Hq * 2 * p.nq), p.B);
  const cudaError_t e = p.D == 64 ? launch_pdl(delta_bf16_kernel<64>, grid, dim3(256), 0, s, p)
                                  : launch_pdl(delta_bf16_kernel<128>, grid, dim3(256), 0, s, p);
  if (e != cudaSuccess) return e;
  prof_end(CAPATTN_KERNEL_DELTA, s);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ dtemp
// dtemp[b, i] = sum over query heads h of the two partial sums the dQ kernels
// left for (b, h, i), always added in the order h = 0, 1, ... (deterministic).
__global__ void dtemp_reduce_kernel(Params p) {
  pdl_trigger();
  pdl_wait();
  const long long bi = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (bi >= (long long)p.B * p.L) return;
  const int b = (int)(bi / p.L), i = (int)(bi % p.L);
  const float2* part = reinterpret_cast<const float2*>(p.dtemp_part);
  float acc = 0.f;
  for (int h = 0; h < p.Hq; ++h) {
    const float2 v = part[((size_t)b * p.Hq + h) * p.L + i];
    acc += v.x + v.y;
  }
  p.dtemp[bi] = acc;
}

cudaError_t launch_dtemp_reduce(const Params& p, cudaStream_t s) {
  const long long n = (long long)p.B * p.L;
  const unsigned grid = (unsigned)((n + 255) / 256);
  const cudaError_t e = launch_pdl(dtemp_reduce_kernel, dim3(grid), dim3(256), 0, s, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// One CTA per batch row: the hull [first, last + 1) of the positions carrying
// each of the two ids (empty (0, 0) when absent), and whether each run fills its
// hull (count == length).
__global__ void ranker_bounds_kernel(const int32_t* seg, int L, int32_t hid, int32_t cid,
                                     int32_t* bounds, uint32_t* status) {
  pdl_trigger();
  pdl_wait();
  __shared__ int lo[2], hi[2], cnt[2];
  const int b = blockIdx.x;
  if (threadIdx.x < 2) {
    lo[threadIdx.x] = L;
    hi[threadIdx.x] = -1;
    cnt[threadIdx.x] = 0;
  }
  __syncthreads();
  int l_lo[2] = {L, L}, l_hi[2] = {-1, -1}, l_cnt[2] = {0, 0};
  const int32_t* row = seg + (size_t)b * L;
  for (int i = threadIdx.x; i < L; i += blockDim.x) {
    const int32_t x = row[i];
    if (x == hid) {
      l_lo[0] = min(l_lo[0], i);
      l_hi[0] = max(l_hi[0], i);
      ++l_cnt[0];
    }
    if (x == cid) {
      l_lo[1] = min(l_lo[1], i);
      l_hi[1] = max(l_hi[1], i);
      ++l_cnt[1];
    }
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    if (l_cnt[k] > 0) {
      atomicMin(&lo[k], l_lo[k]);
      atomicMax(&hi[k], l_hi[k]);
      atomicAdd(&cnt[k], l_cnt[k]);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    bool contiguous = true;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const bool any = cnt[k] > 0;
      bounds[(size_t)b * 4 + 2 * k] = any ? lo[k] : 0;
      bounds[(size_t)b * 4 + 2 * k + 1] = any ? hi[k] + 1 : 0;
      if (any && hi[k] + 1 - lo[k] != cnt[k]) contiguous = false;
    }
    if (!contiguous && status) atomicOr(status, kStatusRankerIdsBit);
  }
}

cudaError_t launch_ranker_bounds(const int32_t* seg, int B, int L, int32_t history_id,
                                 int32_t candidate_id, int32_t* bounds, uint32_t* status,
                                 cudaStream_t s) {
  return launch_pdl(ranker_bounds_kernel, dim3(B), dim3(256), 0, s, seg, L, history_id, candidate_id,
                    bounds, status);
}

}  // namespace capattn

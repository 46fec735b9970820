// fp32 path: CUDA-core (FFMA) forward, dQ and dK/dV kernels on 64 x 64 tiles.
//
// fp32 inputs come with a 1e-4 max-abs tolerance, which tf32 tensor-core
// products (about 5e-4 relative error each) cannot meet, so this dtype runs on
// the FMA pipes.  Structure follows the pages' kernels (triton_kernels.py
// forward / dQ / dK-dV kernels): one CTA per query tile (forward, dQ) or per KV
// tile (dK/dV, summing over the query heads of its group), looping over the
// visited tiles of the block visit map.
#include <math.h>

#include "cap_math.cuh"
#include "capattn_internal.h"

namespace capattn {

namespace {

constexpr int BT = 64;        // tile rows (query and key)
constexpr int NT = 256;       // threads per CTA
constexpr int SP = BT + 1;    // padded stride of the 64 x 64 score tile

// Thread t owns tile row t / 4 and columns (t % 4) + 4 * c, c = 0..15.
struct Lane4 {
  int row, sub;
  __device__ Lane4() : row(threadIdx.x >> 2), sub(threadIdx.x & 3) {}
};

template <int D>
__device__ __forceinline__ void load_tile(float* dst, int ld, const float* src, int row0, int L,
                                          size_t row_stride) {
  // dst[r * ld + d] = src[(row0 + r) * row_stride + d], zero past L.
  for (int idx = threadIdx.x; idx < BT * D; idx += NT) {
    const int r = idx / D, d = idx % D;
    const int gr = row0 + r;
    dst[r * ld + d] = gr < L ? src[(size_t)gr * row_stride + d] : 0.f;
  }
}

__device__ __forceinline__ float quad_max(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, 1));
  return fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, 2));
}
__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xFFFFFFFFu, x, 1);
  return x + __shfl_xor_sync(0xFFFFFFFFu, x, 2);
}

__device__ __forceinline__ bool live(const int4& r, int j) {
  return (j >= r.x && j < r.y) || j == r.z;
}

// ------------------------------------------------------------------ forward
template <int D, int METHOD>
__global__ void __launch_bounds__(NT) fwd_fp32_kernel(Params p) {
  extern __shared__ float sm[];
  float* Qs = sm;                    // [BT][D]
  float* Ks = Qs + BT * D;           // [BT][D + 1]
  float* Vs = Ks + BT * (D + 1);     // [BT][D]
  float* Ps = Vs + BT * D;           // [BT][SP]
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / p.G;
  const Lane4 ln;
  const int q0 = qt * BT;
  const int i = q0 + ln.row;
  const size_t qstride = (size_t)p.Hq * D, kstride = (size_t)p.Hkv * D;
  const float* qg = static_cast<const float*>(p.q) + ((size_t)b * p.L * p.Hq + h) * D;
  const float* kg = static_cast<const float*>(p.k) + ((size_t)b * p.Lk * p.Hkv + g) * D;
  const float* vg = static_cast<const float*>(p.v) + ((size_t)b * p.Lk * p.Hkv + g) * D;
  load_tile<D>(Qs, D, qg, q0, p.L, qstride);
  const int4 ri = i < p.L ? p.rowinfo[(size_t)b * p.L + i] : make_int4(0, 0, -1, 0);
  const float tl = (p.temp && i < p.L ? p.temp[(size_t)b * p.L + i] : 1.f) * kLog2e;
  float m = -INFINITY, lsum = 0.f;
  float acc[D / 4];
#pragma unroll
  for (int d = 0; d < D / 4; ++d) acc[d] = 0.f;
  const uint32_t* map = p.qmap + ((size_t)b * p.nq + qt) * p.wk;
  for (int w = 0; w < p.wk; ++w) {
    uint32_t bits = map[w];
    while (bits) {
      const int kt = w * 32 + __ffs(bits) - 1;
      bits &= bits - 1;
      const int k0 = kt * BT;
      __syncthreads();
      load_tile<D>(Ks, D + 1, kg, k0, p.Lk, kstride);
      load_tile<D>(Vs, D, vg, k0, p.Lk, kstride);
      __syncthreads();
      float x[16];
      float tmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int col = ln.sub + 4 * c;
        float s = 0.f;
#pragma unroll 8
        for (int d = 0; d < D; ++d) s = fmaf(Qs[ln.row * D + d], Ks[col * (D + 1) + d], s);
        const float t = cap_value<METHOD>(s * p.sm_scale, p.cap) * tl;
        x[c] = live(ri, k0 + col) ? t : -INFINITY;
        tmax = fmaxf(tmax, x[c]);
      }
      tmax = quad_max(tmax);
      const float mnew = fmaxf(m, tmax);
      const float alpha = (mnew == -INFINITY) ? 1.f : ex2_approx(m - mnew);
      float psum = 0.f;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float pv = (x[c] == -INFINITY) ? 0.f : ex2_approx(x[c] - mnew);
        psum += pv;
        Ps[ln.row * SP + ln.sub + 4 * c] = pv;
      }
      psum = quad_sum(psum);
      lsum = lsum * alpha + psum;
      m = mnew;
      __syncwarp();
#pragma unroll
      for (int dd = 0; dd < D / 4; ++dd) {
        const int d = ln.sub + 4 * dd;
        float a = acc[dd] * alpha;
#pragma unroll 8
        for (int c = 0; c < BT; ++c) a = fmaf(Ps[ln.row * SP + c], Vs[c * D + d], a);
        acc[dd] = a;
      }
    }
  }
  if (i < p.L) {
    float* og = static_cast<float*>(p.o) + ((size_t)(b * p.L + i) * p.Hq + h) * D;
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
    for (int dd = 0; dd < D / 4; ++dd) og[ln.sub + 4 * dd] = acc[dd] * inv;
    if (ln.sub == 0) {
      const size_t r = ((size_t)b * p.Hq + h) * p.L + i;
      const bool any = lsum > 0.f;
      p.lse[r] = any ? (m + log2f(lsum)) * kLn2 : -INFINITY;
      if (p.m) p.m[r] = any ? m * kLn2 : -INFINITY;
      if (p.l) p.l[r] = lsum;
    }
  }
}

// ------------------------------------------------------------------ dQ
template <int D, int METHOD>
__global__ void __launch_bounds__(NT) dq_fp32_kernel(Params p) {
  extern __shared__ float sm[];
  float* Qs = sm;                    // [BT][D]
  float* Gs = Qs + BT * D;           // dO [BT][D]
  float* Ks = Gs + BT * D;           // [BT][D + 1]
  float* Vs = Ks + BT * (D + 1);     // [BT][D + 1]
  float* Ss = Vs + BT * (D + 1);     // dX [BT][SP]
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / p.G;
  const Lane4 ln;
  const int q0 = qt * BT;
  const int i = q0 + ln.row;
  const size_t qstride = (size_t)p.Hq * D, kstride = (size_t)p.Hkv * D;
  const size_t qoff = ((size_t)b * p.L * p.Hq + h) * D;
  const float* kg = static_cast<const float*>(p.k) + ((size_t)b * p.Lk * p.Hkv + g) * D;
  const float* vg = static_cast<const float*>(p.v) + ((size_t)b * p.Lk * p.Hkv + g) * D;
  load_tile<D>(Qs, D, static_cast<const float*>(p.q) + qoff, q0, p.L, qstride);
  load_tile<D>(Gs, D, static_cast<const float*>(p.dO) + qoff, q0, p.L, qstride);
  const bool valid = i < p.L;
  const int4 ri = valid ? p.rowinfo[(size_t)b * p.L + i] : make_int4(0, 0, -1, 0);
  const float temp = (p.temp && valid) ? p.temp[(size_t)b * p.L + i] : 1.f;
  const size_t r = ((size_t)b * p.Hq + h) * p.L + i;
  const float lse = valid ? p.lse[r] : -INFINITY;
  const float dl = valid ? p.delta[r] : 0.f;
  const float gl = (p.dlse && valid) ? p.dlse[r] : 0.f;
  const bool fin = isfinite(lse);
  const float lse2 = fin ? lse * kLog2e : 0.f;
  const float rowadd = -dl + (fin ? p.z_loss_weight * lse + gl : 0.f);
  const float c1 = p.sm_scale * temp;
  const float tl = temp * kLog2e;
  float acc[D / 4];
#pragma unroll
  for (int d = 0; d < D / 4; ++d) acc[d] = 0.f;
  float dta = 0.f;   // this thread's part of sum_j dT c (temperature gradient)
  const uint32_t* map = p.qmap + ((size_t)b * p.nq + qt) * p.wk;
  for (int w = 0; w < p.wk; ++w) {
    uint32_t bits = map[w];
    while (bits) {
      const int kt = w * 32 + __ffs(bits) - 1;
      bits &= bits - 1;
      const int k0 = kt * BT;
      __syncthreads();
      load_tile<D>(Ks, D + 1, kg, k0, p.Lk, kstride);
      load_tile<D>(Vs, D + 1, vg, k0, p.Lk, kstride);
      __syncthreads();
#pragma unroll 4
      for (int c = 0; c < 16; ++c) {
        const int col = ln.sub + 4 * c;
        float s = 0.f, dp = 0.f;
#pragma unroll 8
        for (int d = 0; d < D; ++d) {
          s = fmaf(Qs[ln.row * D + d], Ks[col * (D + 1) + d], s);
          dp = fmaf(Gs[ln.row * D + d], Vs[col * (D + 1) + d], dp);
        }
        float dc;
        const float cv = cap_value_grad<METHOD>(s * p.sm_scale, p.cap, &dc);
        const float pv = live(ri, k0 + col) ? ex2_approx(cv * tl - lse2) : 0.f;
        const float dT = pv * (dp + rowadd);   // gradient of the tempered logit
        Ss[ln.row * SP + col] = c1 * dc * dT;
        if (p.dtemp) dta = fmaf(dT, cv, dta);
      }
      __syncwarp();
#pragma unroll
      for (int dd = 0; dd < D / 4; ++dd) {
        const int d = ln.sub + 4 * dd;
        float a = acc[dd];
#pragma unroll 8
        for (int c = 0; c < BT; ++c) a = fmaf(Ss[ln.row * SP + c], Ks[c * (D + 1) + d], a);
        acc[dd] = a;
      }
    }
  }
  if (p.dtemp) {
    // the four threads of a row add their columns; one slot pair per (head,
    // row), added over the heads in a fixed order afterwards
    dta += __shfl_xor_sync(0xFFFFFFFFu, dta, 1);
    dta += __shfl_xor_sync(0xFFFFFFFFu, dta, 2);
    if (valid && ln.sub == 0) {
      p.dtemp_part[2 * r] = dta;
      p.dtemp_part[2 * r + 1] = 0.f;
    }
  }
  if (valid) {
    float* dq = static_cast<float*>(p.dq) + ((size_t)(b * p.L + i) * p.Hq + h) * D;
#pragma unroll
    for (int dd = 0; dd < D / 4; ++dd) dq[ln.sub + 4 * dd] = acc[dd];
  }
}

// ------------------------------------------------------------------ dK / dV
template <int D, int METHOD>
__global__ void __launch_bounds__(NT) dkv_fp32_kernel(Params p) {
  extern __shared__ float sm[];
  float* Ks = sm;                    // [BT][D + 1]
  float* Vs = Ks + BT * (D + 1);     // [BT][D + 1]
  float* Qs = Vs + BT * (D + 1);     // [BT][D + 1]
  float* Gs = Qs + BT * (D + 1);     // dO [BT][D + 1]
  float* Ps = Gs + BT * (D + 1);     // P^T  [BT kv][SP]
  float* Xs = Ps + BT * SP;          // dX^T [BT kv][SP]
  int4* Ri = reinterpret_cast<int4*>(Xs + BT * SP);   // [BT]
  float* Cq = reinterpret_cast<float*>(Ri + BT);      // per query row: lse2, rowadd, c1, tl
  const int kt = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const Lane4 ln;
  const int k0 = kt * BT;
  const int j = k0 + ln.row;
  const size_t qstride = (size_t)p.Hq * D, kstride = (size_t)p.Hkv * D;
  const size_t koff = ((size_t)b * p.Lk * p.Hkv + g) * D;
  load_tile<D>(Ks, D + 1, static_cast<const float*>(p.k) + koff, k0, p.Lk, kstride);
  load_tile<D>(Vs, D + 1, static_cast<const float*>(p.v) + koff, k0, p.Lk, kstride);
  float dk[D / 4], dv[D / 4];
#pragma unroll
  for (int d = 0; d < D / 4; ++d) dk[d] = dv[d] = 0.f;
  const uint32_t* map = p.kmap + ((size_t)b * p.nk + kt) * p.wq;
  for (int hh = 0; hh < p.G; ++hh) {
    const int h = g * p.G + hh;
    const size_t qoff = ((size_t)b * p.L * p.Hq + h) * D;
    for (int w = 0; w < p.wq; ++w) {
      uint32_t bits = map[w];
      while (bits) {
        const int qt = w * 32 + __ffs(bits) - 1;
        bits &= bits - 1;
        const int q0 = qt * BT;
        __syncthreads();
        load_tile<D>(Qs, D + 1, static_cast<const float*>(p.q) + qoff, q0, p.L, qstride);
        load_tile<D>(Gs, D + 1, static_cast<const float*>(p.dO) + qoff, q0, p.L, qstride);
        if (threadIdx.x < BT) {
          const int i = q0 + threadIdx.x;
          const bool valid = i < p.L;
          Ri[threadIdx.x] = valid ? p.rowinfo[(size_t)b * p.L + i] : make_int4(0, 0, -1, 0);
          const size_t r = ((size_t)b * p.Hq + h) * p.L + i;
          const float lse = valid ? p.lse[r] : -INFINITY;
          const float dl = valid ? p.delta[r] : 0.f;
          const float gl = (p.dlse && valid) ? p.dlse[r] : 0.f;
          const float temp = (p.temp && valid) ? p.temp[(size_t)b * p.L + i] : 1.f;
          const bool fin = isfinite(lse);
          Cq[4 * threadIdx.x + 0] = fin ? lse * kLog2e : 0.f;
          Cq[4 * threadIdx.x + 1] = -dl + (fin ? p.z_loss_weight * lse + gl : 0.f);
          Cq[4 * threadIdx.x + 2] = p.sm_scale * temp;
          Cq[4 * threadIdx.x + 3] = temp * kLog2e;
        }
        __syncthreads();
        // element (kv row ln.row, query column ln.sub + 4c)
#pragma unroll 4
        for (int c = 0; c < 16; ++c) {
          const int col = ln.sub + 4 * c;
          float s = 0.f, dp = 0.f;
#pragma unroll 8
          for (int d = 0; d < D; ++d) {
            s = fmaf(Qs[col * (D + 1) + d], Ks[ln.row * (D + 1) + d], s);
            dp = fmaf(Gs[col * (D + 1) + d], Vs[ln.row * (D + 1) + d], dp);
          }
          float dc;
          const float cv = cap_value_grad<METHOD>(s * p.sm_scale, p.cap, &dc);
          const float pv = live(Ri[col], j) ? ex2_approx(cv * Cq[4 * col + 3] - Cq[4 * col]) : 0.f;
          Ps[ln.row * SP + col] = pv;
          Xs[ln.row * SP + col] = Cq[4 * col + 2] * dc * pv * (dp + Cq[4 * col + 1]);
        }
        __syncwarp();
#pragma unroll
        for (int dd = 0; dd < D / 4; ++dd) {
          const int d = ln.sub + 4 * dd;
          float a = dk[dd], v = dv[dd];
#pragma unroll 8
          for (int c = 0; c < BT; ++c) {
            a = fmaf(Xs[ln.row * SP + c], Qs[c * (D + 1) + d], a);
            v = fmaf(Ps[ln.row * SP + c], Gs[c * (D + 1) + d], v);
          }
          dk[dd] = a;
          dv[dd] = v;
        }
      }
    }
  }
  if (j < p.Lk) {
    float* dkg = static_cast<float*>(p.dk) + ((size_t)(b * p.Lk + j) * p.Hkv + g) * D;
    float* dvg = static_cast<float*>(p.dv) + ((size_t)(b * p.Lk + j) * p.Hkv + g) * D;
#pragma unroll
    for (int dd = 0; dd < D / 4; ++dd) {
      dkg[ln.sub + 4 * dd] = dk[dd];
      dvg[ln.sub + 4 * dd] = dv[dd];
    }
  }
}

template <int D>
constexpr size_t fwd_smem() { return sizeof(float) * (BT * D + BT * (D + 1) + BT * D + BT * SP); }
template <int D>
constexpr size_t dq_smem() { return sizeof(float) * (2 * BT * D + 2 * BT * (D + 1) + BT * SP); }
template <int D>
constexpr size_t dkv_smem() {
  return sizeof(float) * (4 * BT * (D + 1) + 2 * BT * SP) + sizeof(int4) * BT + sizeof(float) * 4 * BT;
}

template <int METHOD>
struct FwdLaunch {
  template <int D>
  static cudaError_t go(const Params& p, cudaStream_t s) {
    auto kern = fwd_fp32_kernel<D, METHOD>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fwd_smem<D>());
    if (e != cudaSuccess) return e;
    prof_begin(CAPATTN_KERNEL_FWD, s);
    prof_count(CAPATTN_KERNEL_FWD, 1);
    kern<<<dim3(p.nq, p.Hq, p.B), NT, fwd_smem<D>(), s>>>(p);
    prof_end(CAPATTN_KERNEL_FWD, s);
    return cudaGetLastError();
  }
  static cudaError_t run(const Params& p, cudaStream_t s) { return p.D == 64 ? go<64>(p, s) : go<128>(p, s); }
};

template <int METHOD>
struct BwdLaunch {
  template <int D>
  static cudaError_t go(const Params& p, cudaStream_t s) {
    auto kdkv = dkv_fp32_kernel<D, METHOD>;
    cudaError_t e = cudaFuncSetAttribute(kdkv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dkv_smem<D>());
    if (e != cudaSuccess) return e;
    prof_begin(CAPATTN_KERNEL_DKV, s);
    prof_count(CAPATTN_KERNEL_DKV, 1);
    kdkv<<<dim3(p.nk, p.Hkv, p.B), NT, dkv_smem<D>(), s>>>(p);
    prof_end(CAPATTN_KERNEL_DKV, s);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto kdq = dq_fp32_kernel<D, METHOD>;
    e = cudaFuncSetAttribute(kdq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dq_smem<D>());
    if (e != cudaSuccess) return e;
    prof_begin(CAPATTN_KERNEL_DQ, s);
    prof_count(CAPATTN_KERNEL_DQ, 1);
    kdq<<<dim3(p.nq, p.Hq, p.B), NT, dq_smem<D>(), s>>>(p);
    prof_end(CAPATTN_KERNEL_DQ, s);
    return cudaGetLastError();
  }
  static cudaError_t run(const Params& p, cudaStream_t s) { return p.D == 64 ? go<64>(p, s) : go<128>(p, s); }
};

}  // namespace

cudaError_t launch_fwd_fp32(const Params& p, cudaStream_t s) {
  return dispatch_cap<FwdLaunch>(p.cap.method, p, s);
}

cudaError_t launch_bwd_fp32(const Params& p, cudaStream_t s) {
  return dispatch_cap<BwdLaunch>(p.cap.method, p, s);
}

}  // namespace capattn

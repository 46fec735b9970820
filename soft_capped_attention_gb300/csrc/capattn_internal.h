// Internal interfaces between the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/capattn.h"
#include "status_bits.h"

namespace capattn {

// Cap constants, precomputed on the host in double precision
// (mosaic_backward.py _apply_cap_mosaic; derivative of each branch).
struct CapConsts {
  int32_t method;     // CAPATTN_CAP_*, NONE when cap <= 0
  float cap;          // tanh: output scale
  float inv_cap;      // tanh: 1/cap (argument scale); soft_sign: 1/cap
  float alsc_a;       // ALSC: z = alsc_a * s + alsc_b, alsc_a = alpha / cap
  float alsc_b;       //       alsc_b = alpha * beta
  float alsc_out;     // ALSC: cap / denom
  float alsc_sb;      // ALSC: sigma(alpha * beta)
  float alsc_dout;    // ALSC: derivative scale alpha / denom
  // ALSC on the FMA pipe: sigma(alsc_a * sm_scale * X + alsc_b) - alsc_sb
  // = X * sum_k alsc_gu[k] X^k for a raw score X with |X| <= alsc_xmax
  // (an interpolating polynomial; alsc_xmax 0: none)
  float alsc_gu[7];
  float alsc_xmax;
};

struct Params {
  // tensors
  const void* q;
  const void* k;
  const void* v;
  const float* temp;      // [B, L] or null
  const int32_t* seg;     // [B, L] or null
  const int32_t* bounds;  // [B, 4] or null
  void* o;
  float* lse;
  float* m;               // nullable
  float* l;               // nullable
  const void* dO;
  void* dq;
  void* dk;
  void* dv;
  float* delta;
  float* dtemp;           // [B, L] gradient of the temperature, or null
  float* dtemp_part;      // [B, Hq, L, 2] per-head partial sums of dtemp (backward workspace)
  const float* dlse;      // [B, Hq, L] upstream gradient of the LSE, or null
  // workspace pieces
  uint32_t* status;
  int4* rowinfo;          // [B, L] (lo, hi, e, 0)
  uint32_t* qmap;         // [B, nq, wk]
  uint32_t* kmap;         // [B, nk, wq]
  int2* qfull;            // [B, nq]: KV tiles [x, y) in which every pair is live
  // Stored-dX backward (bf16; null otherwise): the dK/dV kernel writes each
  // step's dX^T tile (128 keys x 128 queries, bf16, key rows of 256 bytes) to
  // slot ((b Hq + h) nq + qt) dx_wmax + (kt - kt_lo(qt)) of the pool, and the
  // dQ GEMM kernel reads the tiles back.  kt_lo(qt) = max(0, qt - dx_c) with a
  // sliding window (dx_c >= 0), else 0; dx_wmax = the widest band of key tiles
  // a query tile can visit under the configuration's causal / window masks.
  void* dx_pool;
  int32_t dx_wmax, dx_c;
  uint32_t* dq_work;      // work counter of the persistent dQ GEMM (zeroed by the delta kernel)
  uint32_t* fwd_work;     // work counter of the persistent forward (zeroed by rowmap_kernel)
  // shapes (L query rows, Lk keys)
  int32_t B, L, Lk, Hq, Hkv, D, G;
  int32_t block_q, block_kv, nq, nk, wq, wk;
  // method
  float sm_scale;
  int32_t causal, window_len;
  float z_loss_weight;
  CapConsts cap;
};

// `total` is what the forward needs; the backward also holds the per-head
// partial sums of the temperature gradient after it (`total_bwd`), and the
// stored-dX backward its dX pool after that (`total_dx`; equal to total_bwd
// when that backward does not apply: fp32, or a pool above kDxPoolMaxBytes).
// Slot and 32-byte-unit indices of the pool fit 32 bits up to 128 GiB.
struct WorkspaceLayout {
  size_t status_off, rowinfo_off, qmap_off, kmap_off, qfull_off, total, dtemp_part_off, total_bwd;
  size_t dx_off, total_dx;
  int32_t dx_wmax, dx_c;
};
constexpr size_t kDxTileBytes = 128 * 128 * 2;
constexpr size_t kDxPoolMaxBytes = size_t(16) << 30;

WorkspaceLayout workspace_layout(const capattn_config& c, int block_q, int block_kv);

// Optional per-kernel event timing around launches (no-ops unless enabled);
// prof_count adds the number of kernels a launcher issued.
void prof_begin(int kind, cudaStream_t stream);
void prof_end(int kind, cudaStream_t stream);
void prof_count(int kind, int n);

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel of the stream finishes; every kernel launched this
// way waits for its predecessor (griddepcontrol.wait) before it touches global
// memory, and lets its own dependents be scheduled from its start.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

#ifdef __CUDACC__
// Device side of the above: let the next kernel of the stream be scheduled now /
// wait until the previous kernel has completed and its writes are visible.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
#endif

// Launchers.  Each returns cudaGetLastError() after the launch.
// build_rows: rowmap_kernel (spans, query-tile maps, fully covered ranges;
// clears the key-tile map); build_kmap: kmap_kernel (key-tile map from the
// query-tile map, whole words).
cudaError_t launch_prepass(const Params& p, bool build_rows, bool build_kmap, cudaStream_t s);
cudaError_t launch_delta_fp32(const Params& p, cudaStream_t s);
// bf16 delta for the stored-dX backward; also ORs each query tile's bits into
// the key-tile map (rowmap_kernel cleared it).
cudaError_t launch_delta_bf16(const Params& p, cudaStream_t s);
// dQ from the stored dX tiles (bf16, HD = p.D).
cudaError_t launch_dq_gemm(const Params& p, cudaStream_t s);
cudaError_t launch_fwd_fp32(const Params& p, cudaStream_t s);
cudaError_t launch_bwd_fp32(const Params& p, cudaStream_t s);
cudaError_t launch_fwd_bf16(const Params& p, cudaStream_t s);
cudaError_t launch_fwd1_bf16(const Params& p, cudaStream_t s);  // one query tile per CTA
cudaError_t launch_fwd2_bf16(const Params& p, cudaStream_t s);  // one tile, two score buffers
cudaError_t launch_fwd3_bf16(const Params& p, cudaStream_t s);  // persistent, fixed reference
cudaError_t launch_bwd_bf16(const Params& p, cudaStream_t s);
cudaError_t launch_dtemp_reduce(const Params& p, cudaStream_t s);
cudaError_t launch_wait_check(uint32_t* status, uint64_t limit_ns, int ctas, cudaStream_t s);
cudaError_t launch_ranker_bounds(const int32_t* seg, int B, int L, int32_t history_id,
                                 int32_t candidate_id, int32_t* bounds, uint32_t* status,
                                 cudaStream_t s);

}  // namespace capattn

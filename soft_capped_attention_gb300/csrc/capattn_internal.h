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
// partial sums of the temperature gradient after it (`total_bwd`).
struct WorkspaceLayout {
  size_t status_off, rowinfo_off, qmap_off, kmap_off, qfull_off, total, dtemp_part_off, total_bwd;
};

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
cudaError_t launch_fwd_fp32(const Params& p, cudaStream_t s);
cudaError_t launch_bwd_fp32(const Params& p, cudaStream_t s);
cudaError_t launch_fwd_bf16(const Params& p, cudaStream_t s);
cudaError_t launch_bwd_bf16(const Params& p, cudaStream_t s);
cudaError_t launch_dtemp_reduce(const Params& p, cudaStream_t s);
cudaError_t launch_wait_check(uint32_t* status, uint64_t limit_ns, int ctas, cudaStream_t s);
cudaError_t launch_ranker_bounds(const int32_t* seg, int B, int L, int32_t history_id,
                                 int32_t candidate_id, int32_t* bounds, uint32_t* status,
                                 cudaStream_t s);

}  // namespace capattn

// Forward entry point that allocates nothing: capattn_fwd_noalloc.
//
// Some callers cannot hand the library a workspace.  A plugin running inside a
// host framework that owns all device memory (and offers its plugins no
// scratch), or a service held to a fixed memory budget that forbids any
// allocation once it is serving, has no way to call cudaMalloc or to ask for a
// buffer between requests.  For them the forward keeps its scratch (the device
// status word, the per-row live spans and the block visit maps) in a
// file-scope device array of fixed size instead of a caller-provided
// workspace.  Every GPU that loads the library holds that array until the
// process exits.
#include <mutex>

#include "capattn_internal.h"

namespace {

// Fixed scratch: 8 MiB per device.  The forward needs 256 bytes plus 16 bytes
// per (batch row, position) plus the visit maps, so this covers B * L up to
// about 500,000 rows.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array, looked up once per device (the host-side name
// g_noalloc_scratch is only a stand-in and must never be passed to a kernel).
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// The current device's address of the array (set-up on the first call per
// device, with that device current).
capattn_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CAPATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CAPATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> guard(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || !addr)
      return CAPATTN_ERR_CUDA;
    g_scratch_addr[dev] = addr;
  }
  *out = g_scratch_addr[dev];
  return CAPATTN_OK;
}

}  // namespace

extern "C" capattn_status capattn_fwd_noalloc(const capattn_config* cfg, const void* q,
                                              const void* k, const void* v, const float* temp,
                                              const int32_t* seg, const int32_t* bounds, void* o,
                                              float* lse, float* m, float* l,
                                              cudaStream_t stream) {
  capattn_status st = capattn_validate_config(cfg);
  if (st != CAPATTN_OK) return st;
  if (capattn_workspace_bytes(cfg, CAPATTN_PASS_FWD) > kNoAllocScratchBytes)
    return CAPATTN_ERR_TOO_LARGE;
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != CAPATTN_OK) return st;
  // The array keeps the previous call's contents.  Only the status word has to
  // start at zero; the pre-pass rewrites the spans and visit maps on every call.
  if (cudaMemsetAsync(scratch, 0, 256, stream) != cudaSuccess) return CAPATTN_ERR_CUDA;
  return capattn_fwd(cfg, q, k, v, temp, seg, bounds, o, lse, m, l, scratch, kNoAllocScratchBytes,
                     stream);
}

// The status word that the last capattn_fwd_noalloc call on this device left in
// the fixed array: copied into a host word (no device memory is allocated),
// then cleared.  Synchronises `stream`.
extern "C" capattn_status capattn_noalloc_status(cudaStream_t stream, uint32_t* raw_bits) {
  void* scratch = nullptr;
  capattn_status st = scratch_address(&scratch);
  if (st != CAPATTN_OK) return st;
  uint32_t bits = 0;
  if (cudaMemcpyFromSymbolAsync(&bits, g_noalloc_scratch, sizeof(bits), 0, cudaMemcpyDeviceToHost,
                                stream) != cudaSuccess)
    return CAPATTN_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return CAPATTN_ERR_CUDA;
  if (bits) {
    if (cudaMemsetAsync(scratch, 0, sizeof(bits), stream) != cudaSuccess) return CAPATTN_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return CAPATTN_ERR_CUDA;
  }
  if (raw_bits) *raw_bits = bits;
  if (bits & capattn::kStatusTimeoutBit) return CAPATTN_ERR_DEVICE_TIMEOUT;
  if (bits) return CAPATTN_ERR_DEVICE_DATA;
  return CAPATTN_OK;
}

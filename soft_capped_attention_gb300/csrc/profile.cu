// Optional per-kernel timing with CUDA events (capattn_profile_enable/read).
#include <mutex>
#include <vector>

#include "capattn_internal.h"

namespace capattn {

namespace {

struct Pending {
  int kind;
  cudaEvent_t start, stop;
};

struct ProfState {
  std::mutex mu;
  bool on = false;
  unsigned mask = (1u << CAPATTN_KERNEL_KINDS) - 1u;
  std::vector<cudaEvent_t> pool;
  std::vector<Pending> pending;
  Pending open[CAPATTN_KERNEL_KINDS];
  bool is_open[CAPATTN_KERNEL_KINDS] = {};
  double ms[CAPATTN_KERNEL_KINDS] = {};
  int64_t launches[CAPATTN_KERNEL_KINDS] = {};
};

ProfState& state() {
  static ProfState s;
  return s;
}

cudaEvent_t take_event(ProfState& s) {
  if (!s.pool.empty()) {
    cudaEvent_t e = s.pool.back();
    s.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

void prof_begin(int kind, cudaStream_t stream) {
  ProfState& s = state();
  std::lock_guard<std::mutex> g(s.mu);
  if (!s.on || kind < 0 || kind >= CAPATTN_KERNEL_KINDS || !((s.mask >> kind) & 1u)) return;
  Pending p;
  p.kind = kind;
  p.start = take_event(s);
  p.stop = take_event(s);
  if (!p.start || !p.stop) return;
  cudaEventRecord(p.start, stream);
  s.open[kind] = p;
  s.is_open[kind] = true;
}

void prof_end(int kind, cudaStream_t stream) {
  ProfState& s = state();
  std::lock_guard<std::mutex> g(s.mu);
  if (!s.on || kind < 0 || kind >= CAPATTN_KERNEL_KINDS || !s.is_open[kind]) return;
  Pending p = s.open[kind];
  s.is_open[kind] = false;
  cudaEventRecord(p.stop, stream);
  s.pending.push_back(p);
}

void prof_count(int kind, int n) {
  ProfState& s = state();
  std::lock_guard<std::mutex> g(s.mu);
  if (s.on && kind >= 0 && kind < CAPATTN_KERNEL_KINDS) s.launches[kind] += n;
}

}  // namespace capattn

using namespace capattn;

extern "C" {

capattn_status capattn_profile_enable(int on) {
  ProfState& s = state();
  std::lock_guard<std::mutex> g(s.mu);
  s.on = on != 0;
  return CAPATTN_OK;
}

capattn_status capattn_profile_select(unsigned int kind_mask) {
  if (kind_mask >> CAPATTN_KERNEL_KINDS) return CAPATTN_ERR_INVALID_ARG;
  ProfState& s = state();
  std::lock_guard<std::mutex> g(s.mu);
  s.mask = kind_mask;
  return CAPATTN_OK;
}

capattn_status capattn_profile_read(double* ms, int64_t* launches, int n_kinds, int reset) {
  ProfState& s = state();
  std::lock_guard<std::mutex> g(s.mu);
  for (const Pending& p : s.pending) {
    if (cudaEventSynchronize(p.stop) != cudaSuccess) return CAPATTN_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, p.start, p.stop) != cudaSuccess) return CAPATTN_ERR_CUDA;
    s.ms[p.kind] += t;
    s.pool.push_back(p.start);
    s.pool.push_back(p.stop);
  }
  s.pending.clear();
  for (int k = 0; k < n_kinds && k < CAPATTN_KERNEL_KINDS; ++k) {
    if (ms) ms[k] = s.ms[k];
    if (launches) launches[k] = s.launches[k];
  }
  if (reset) {
    for (int k = 0; k < CAPATTN_KERNEL_KINDS; ++k) {
      s.ms[k] = 0.0;
      s.launches[k] = 0;
    }
  }
  return CAPATTN_OK;
}

const char* capattn_kernel_name(int kind) {
  switch (kind) {
    case CAPATTN_KERNEL_PREPASS: return "prepass";
    case CAPATTN_KERNEL_FWD: return "fwd";
    case CAPATTN_KERNEL_DELTA: return "delta";
    case CAPATTN_KERNEL_DKV: return "dkv";
    case CAPATTN_KERNEL_DQ: return "dq";
  }
  return "unknown";
}

}  // extern "C"

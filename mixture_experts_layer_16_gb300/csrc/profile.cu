// profile.cu -- optional per-kernel timing: while enabled, every kernel a forward or
// backward call enqueues is bracketed by two CUDA events on the caller's stream;
// mm_moe_profile_stop synchronises them and reports the summed time per kernel.
#include <cuda_runtime.h>

#include <vector>

#include "internal.h"

namespace mmmoe {

static const char* const kKernelNames[K_COUNT] = {
    "route_count", "route_scan", "route_place", "permute_x", "gemm_gateup_swiglu",
    "gemm_down_weighted", "combine", "permute_dy", "gemm_dgrad_down_dswiglu",
    "gemm_dgrad_gateup", "unpermute_reduce", "gemm_wgrad_down", "gemm_wgrad_gateup", "gemm_wgrad",
    "mx_qdq_rows", "mx_qdq_cols", "fp8block_rows", "fp8block_cols", "fp8block_tiles", "fbq_rows",
    "fbq_cols", "fbq_tiles", "mxq_rows", "mxq_cols",
    "gemm_dense_nt", "gemm_dense_nn", "gemm_dense_tn", "router_topk", "router_dlogits"};

namespace {
struct Rec {
  int id;
  cudaEvent_t a, b;
};
struct Prof {
  bool on = false;
  std::vector<cudaEvent_t> pool;
  size_t used = 0;
  cudaEvent_t pending = nullptr;
  std::vector<Rec> recs;
  double total_ms[K_COUNT] = {};
  int count[K_COUNT] = {};
  cudaEvent_t take() {
    if (used == pool.size()) {
      cudaEvent_t e = nullptr;
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
      pool.push_back(e);
    }
    return pool[used++];
  }
};
thread_local Prof g_prof;
}  // namespace

void prof_begin(const Ctx& c, int id) {
  (void)id;
  Prof& p = g_prof;
  if (!p.on) return;
  p.pending = p.take();
  if (p.pending) cudaEventRecord(p.pending, c.stream);
}

void prof_end(const Ctx& c, int id) {
  ++*c.launches;
  Prof& p = g_prof;
  if (!p.on || p.pending == nullptr) return;
  cudaEvent_t b = p.take();
  if (b == nullptr) return;
  cudaEventRecord(b, c.stream);
  p.recs.push_back(Rec{id, p.pending, b});
  p.pending = nullptr;
}

}  // namespace mmmoe

using namespace mmmoe;

extern "C" MM_MOE_API mm_moe_status mm_moe_profile_start(void) {
  Prof& p = g_prof;
  p.recs.clear();
  p.used = 0;
  p.pending = nullptr;
  for (int i = 0; i < K_COUNT; ++i) {
    p.total_ms[i] = 0.0;
    p.count[i] = 0;
  }
  p.on = true;
  return MM_MOE_OK;
}

extern "C" MM_MOE_API mm_moe_status mm_moe_profile_stop(float* total_ms, int* launches, int n) {
  Prof& p = g_prof;
  p.on = false;
  mm_moe_status st = MM_MOE_OK;
  for (const Rec& r : p.recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
      st = MM_MOE_ECUDA;
      continue;
    }
    p.total_ms[r.id] += ms;
    p.count[r.id] += 1;
  }
  p.recs.clear();
  p.used = 0;
  for (int i = 0; i < n && i < K_COUNT; ++i) {
    if (total_ms) total_ms[i] = static_cast<float>(p.total_ms[i]);
    if (launches) launches[i] = p.count[i];
  }
  return st;
}

extern "C" MM_MOE_API const char* mm_moe_kernel_name(int id) {
  return (id >= 0 && id < K_COUNT) ? kKernelNames[id] : nullptr;
}

extern "C" MM_MOE_API int mm_moe_kernel_count(void) { return K_COUNT; }

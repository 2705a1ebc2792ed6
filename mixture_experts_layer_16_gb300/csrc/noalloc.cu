// noalloc.cu -- mm_moe_route_noalloc: the token routing without any caller-provided
// scratch.  Its working memory is a fixed array in this library's device image, so
// a caller that cannot allocate device memory at call time (an allocator-less
// runtime, a process whose memory pool is owned by another component, code that
// must not fail on an out-of-memory path) can still compute the expert-grouped
// order of its tokens.  The caller passes only inputs and outputs.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace mmmoe {

// Limits of the no-allocation routing (the array below is sized for them).
constexpr int64_t NOALLOC_MAX_ROWS = 262144;  // T * k
constexpr int64_t NOALLOC_MAX_E = 256;
constexpr int64_t NOALLOC_MAX_BLK = (NOALLOC_MAX_ROWS + ROUTE_CHUNK - 1) / ROUTE_CHUNK;
constexpr int64_t NOALLOC_MAX_NT = NOALLOC_MAX_ROWS / BM + NOALLOC_MAX_E;
constexpr int64_t NOALLOC_MAX_RP = NOALLOC_MAX_NT * BM;

constexpr size_t al256(size_t v) { return (v + 255) / 256 * 256; }
constexpr size_t OFF_STATUS = 0;
constexpr size_t OFF_BLK = al256(OFF_STATUS + sizeof(DevStatus));
constexpr size_t OFF_COUNTS = al256(OFF_BLK + 4 * NOALLOC_MAX_BLK * NOALLOC_MAX_E);
constexpr size_t OFF_PADOFF = al256(OFF_COUNTS + 4 * NOALLOC_MAX_E);
constexpr size_t OFF_ORDER = al256(OFF_PADOFF + 4 * (NOALLOC_MAX_E + 1));
constexpr size_t OFF_META = al256(OFF_ORDER + 4 * NOALLOC_MAX_E);
constexpr size_t OFF_TEXP = al256(OFF_META + 4 * 16);
constexpr size_t OFF_TROWS = al256(OFF_TEXP + 4 * NOALLOC_MAX_NT);
constexpr size_t OFF_PROW = al256(OFF_TROWS + 4 * NOALLOC_MAX_NT);
constexpr size_t OFF_ROWFLAT = al256(OFF_PROW + 4 * NOALLOC_MAX_ROWS);
constexpr size_t OFF_WROW = al256(OFF_ROWFLAT + 4 * NOALLOC_MAX_RP);
constexpr size_t NOALLOC_BYTES = al256(OFF_WROW + 4 * NOALLOC_MAX_RP);
constexpr size_t NOALLOC_ARRAY_BYTES = 4u << 20;  // 4 MiB
static_assert(NOALLOC_BYTES <= NOALLOC_ARRAY_BYTES, "routing scratch does not fit");

// The working memory.  Every device that loads the library holds these 4 MiB until
// the process exits; all calls share them.
static __device__ __align__(256) unsigned char g_route_scratch[NOALLOC_ARRAY_BYTES];

// Device address of g_route_scratch on each device.  In host code the array's name
// is only a host-side stand-in, so the address is looked up once per device (with
// that device current) and then passed to the kernels.
static unsigned char* scratch_address(int dev, cudaError_t* err) {
  static std::mutex mu;
  static unsigned char* addr[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) {
      *err = e;
      return nullptr;
    }
    addr[dev] = static_cast<unsigned char*>(p);
  }
  *err = cudaSuccess;
  return addr[dev];
}

}  // namespace mmmoe

using namespace mmmoe;

extern "C" MM_MOE_API mm_moe_status mm_moe_route_noalloc(const mm_moe_shape* shape,
                                                         const int32_t* topk_idx,
                                                         const float* topk_w, int32_t* offsets,
                                                         int32_t* perm, int32_t* inv,
                                                         void* stream) {
  if (shape == nullptr || shape->T < 1 || shape->k < 1 || shape->E < 1 || shape->k > shape->E)
    return MM_MOE_EINVAL;
  if (shape->E > NOALLOC_MAX_E || shape->T > NOALLOC_MAX_ROWS / shape->k) return MM_MOE_EINVAL;
  auto ok4 = [](const void* p) {
    return p != nullptr && (reinterpret_cast<uintptr_t>(p) % 4) == 0;
  };
  if (!ok4(topk_idx) || !ok4(topk_w) || !ok4(offsets) || !ok4(perm) || !ok4(inv))
    return MM_MOE_EINVAL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MM_MOE_ECUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MM_MOE_ECUDA;
  if (major != 10 || minor != 3) return MM_MOE_ENOTSUP;
  cudaError_t err = cudaSuccess;
  unsigned char* base = scratch_address(dev, &err);
  if (base == nullptr) return MM_MOE_ECUDA;

  const int R = static_cast<int>(shape->T * shape->k), E = static_cast<int>(shape->E);
  RouteBufs b;
  b.status = reinterpret_cast<DevStatus*>(base + OFF_STATUS);
  b.blk_counts = reinterpret_cast<int*>(base + OFF_BLK);
  b.counts = reinterpret_cast<int*>(base + OFF_COUNTS);
  b.offsets = offsets;
  b.pad_off = reinterpret_cast<int*>(base + OFF_PADOFF);
  b.expert_order = reinterpret_cast<int*>(base + OFF_ORDER);
  b.tile_expert = reinterpret_cast<int*>(base + OFF_TEXP);
  b.tile_rows = reinterpret_cast<int*>(base + OFF_TROWS);
  b.meta = reinterpret_cast<int*>(base + OFF_META);
  b.perm = perm;
  b.inv = inv;
  b.prow = reinterpret_cast<int*>(base + OFF_PROW);
  b.rowflat = reinterpret_cast<int*>(base + OFF_ROWFLAT);
  b.w_row = reinterpret_cast<float*>(base + OFF_WROW);
  int launches = 0;
  Ctx c{static_cast<cudaStream_t>(stream), 0, &launches};
  // the status word keeps the previous call's value: start from zero
  if (cudaMemsetAsync(b.status, 0, sizeof(DevStatus), c.stream) != cudaSuccess)
    return MM_MOE_ECUDA;
  if (launch_route_to(c, R, E, BM, topk_idx, topk_w, b) != cudaSuccess) return MM_MOE_ECUDA;
  return MM_MOE_OK;
}

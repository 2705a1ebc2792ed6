// router.cu -- the top-k router in front of the layer: logits, top-k selection with
// a softmax over the chosen experts, and the backward through the routing weights.
//
// The Prime Mega MoE pages say that each token goes to a small subset of the experts
// ("Why is MoE training communication-bound?") and that the tested models pick 8 of
// 128 ("TL;DR"); the router is not described.  Readings: logits = x W_router^T with
// no bias; the k largest logits of a token in descending order, equal logits to the
// lower expert index; weights = softmax over the chosen logits (the full softmax
// renormalised over them); the gradient flows through the weights only.
//
// The three matrix products (x W_router^T; dlogits^T x; dlogits W_router) are dense
// GEMMs on the library's own tcgen05 kernel (bf16 operands, fp32 accumulation; the
// dense kinds of gemm.cuh; dlogits^T x, with few output tiles and K = T, splits its K
// over a cluster and sums the partial tiles through distributed shared memory).  The selection, the softmax and the logit gradient are this
// file's kernels: one warp per token.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"

namespace mmmoe {

constexpr int ROUTER_MAX_K = 32;

// (v, i) ranks before (w, j): larger logit first, equal logits by lower index
__device__ __forceinline__ bool before(float v, int i, float w, int j) {
  return v > w || (v == w && i < j);
}

// One warp per token: lane l holds logits l, l + 32, ...; k rounds of a warp argmax.
template <int PL>
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ logits,
                                                          int64_t T, int E, int k,
                                                          int32_t* __restrict__ topk_idx,
                                                          float* __restrict__ topk_w) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;  // whole warps leave together
  const float* row = logits + t * E;
  float v[PL];
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? __ldg(row + e) : -INFINITY;
  }
  uint32_t taken = 0;
  int my_idx = 0;
  float my_val = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;  // with the sentinel index every finite or -inf logit beats it
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !(taken >> i & 1u) && before(v[i], e, bv, bi)) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (before(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    // (a token whose logits are all NaN finds no candidate: bi stays the sentinel)
    if (bi != 0x7fffffff && (bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) {
      my_idx = bi;
      my_val = bv;
    }
  }
  // softmax over the k chosen logits (lane 0 holds the largest)
  const float m = __shfl_sync(0xffffffffu, my_val, 0);
  const float ex = lane < k ? expf(my_val - m) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane < k) {
    topk_idx[t * k + lane] = my_idx;
    topk_w[t * k + lane] = ex / sum;
  }
}

// One warp per token: dlogits[t, e_j] = w_j (g_j - sum_i w_i g_i), zero elsewhere,
// written as a dense bf16 row for the two backward GEMMs.
template <int PL>
__global__ void __launch_bounds__(256) router_dlogits_kernel(const int32_t* __restrict__ topk_idx,
                                                             const float* __restrict__ topk_w,
                                                             const float* __restrict__ dtopk_w,
                                                             int64_t T, int E, int k,
                                                             __nv_bfloat16* __restrict__ dlogits) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const float w = lane < k ? __ldg(topk_w + t * k + lane) : 0.f;
  const float g = lane < k ? __ldg(dtopk_w + t * k + lane) : 0.f;
  const int e_mine = lane < k ? __ldg(topk_idx + t * k + lane) : -1;
  float s = w * g;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  const float d_mine = w * (g - s);
  float out[PL];
#pragma unroll
  for (int i = 0; i < PL; ++i) out[i] = 0.f;
  for (int j = 0; j < k; ++j) {
    const int e = __shfl_sync(0xffffffffu, e_mine, j);
    const float d = __shfl_sync(0xffffffffu, d_mine, j);
#pragma unroll
    for (int i = 0; i < PL; ++i)
      if (e == lane + 32 * i) out[i] = d;
  }
  __nv_bfloat16* row = dlogits + t * E;
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) row[e] = __float2bfloat16_rn(out[i]);
  }
}

static bool router_shape_ok(const mm_moe_shape* s) {
  return s != nullptr && s->T >= 1 && s->H >= 1 && s->E >= 1 && s->k >= 1 && s->k <= s->E &&
         s->k <= ROUTER_MAX_K && s->E <= 1024 && s->H % 8 == 0 && s->E % 8 == 0 &&
         s->T <= (int64_t{1} << 31) / s->E;
}

static bool device_ok(int* sms) {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return false;
  return major == 10 && minor == 3;
}

template <int PL>
static void launch_topk(const Ctx& c, const float* logits, int64_t T, int E, int k,
                        int32_t* idx, float* w) {
  const int64_t blocks = (T * 32 + 255) / 256;
  prof_begin(c, K_ROUTER_TOPK);
  launch_k(c.stream, router_topk_kernel<PL>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
           logits, T, E, k, idx, w);
  prof_end(c, K_ROUTER_TOPK);
}

template <int PL>
static void launch_dlogits(const Ctx& c, const int32_t* idx, const float* w, const float* g,
                           int64_t T, int E, int k, __nv_bfloat16* dl) {
  const int64_t blocks = (T * 32 + 255) / 256;
  prof_begin(c, K_ROUTER_DLOGITS);
  launch_k(c.stream, router_dlogits_kernel<PL>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
           idx, w, g, T, E, k, dl);
  prof_end(c, K_ROUTER_DLOGITS);
}

}  // namespace mmmoe

using namespace mmmoe;

static bool al(const void* p, uintptr_t a) {
  return p != nullptr && reinterpret_cast<uintptr_t>(p) % a == 0;
}

extern "C" MM_MOE_API mm_moe_status mm_moe_router_forward(const mm_moe_shape* shape,
                                                          const uint16_t* x,
                                                          const uint16_t* W_router, float* logits,
                                                          int32_t* topk_idx, float* topk_w,
                                                          void* stream) {
  if (!router_shape_ok(shape)) return MM_MOE_EINVAL;
  if (!al(x, 16) || !al(W_router, 16) || !al(logits, 16) || !al(topk_idx, 4) || !al(topk_w, 4))
    return MM_MOE_EINVAL;
  int sms = 0;
  if (!device_ok(&sms)) return MM_MOE_ENOTSUP;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int T = static_cast<int>(shape->T), H = static_cast<int>(shape->H),
            E = static_cast<int>(shape->E), k = static_cast<int>(shape->k);
  int launches = 0;
  const Ctx c{st, sms, &launches};
  // logits [T, E] = x [T, H] . W_router [E, H]^T
  if (launch_dense(c, GEMM_DENSE_NT, x, W_router, logits, T, E, H) != cudaSuccess)
    return MM_MOE_ECUDA;
  if (E <= 128)
    launch_topk<4>(c, logits, T, E, k, topk_idx, topk_w);
  else if (E <= 256)
    launch_topk<8>(c, logits, T, E, k, topk_idx, topk_w);
  else
    launch_topk<32>(c, logits, T, E, k, topk_idx, topk_w);
  return cudaGetLastError() == cudaSuccess ? MM_MOE_OK : MM_MOE_ECUDA;
}

extern "C" MM_MOE_API mm_moe_status mm_moe_router_backward(
    const mm_moe_shape* shape, const uint16_t* x, const uint16_t* W_router,
    const int32_t* topk_idx, const float* topk_w, const float* dtopk_w, uint16_t* dlogits,
    uint16_t* dx, uint16_t* dW_router, void* stream) {
  if (!router_shape_ok(shape)) return MM_MOE_EINVAL;
  if (!al(x, 16) || !al(W_router, 16) || !al(topk_idx, 4) || !al(topk_w, 4) ||
      !al(dtopk_w, 4) || !al(dlogits, 16) || !al(dx, 16) || !al(dW_router, 16))
    return MM_MOE_EINVAL;
  int sms = 0;
  if (!device_ok(&sms)) return MM_MOE_ENOTSUP;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int T = static_cast<int>(shape->T), H = static_cast<int>(shape->H),
            E = static_cast<int>(shape->E), k = static_cast<int>(shape->k);
  int launches = 0;
  const Ctx c{st, sms, &launches};
  __nv_bfloat16* dl = reinterpret_cast<__nv_bfloat16*>(dlogits);
  if (E <= 128)
    launch_dlogits<4>(c, topk_idx, topk_w, dtopk_w, T, E, k, dl);
  else if (E <= 256)
    launch_dlogits<8>(c, topk_idx, topk_w, dtopk_w, T, E, k, dl);
  else
    launch_dlogits<32>(c, topk_idx, topk_w, dtopk_w, T, E, k, dl);
  if (cudaGetLastError() != cudaSuccess) return MM_MOE_ECUDA;
  // dW_router [E, H] = dlogits [T, E]^T . x [T, H]
  if (launch_dense(c, GEMM_DENSE_TN, dlogits, x, dW_router, E, H, T) != cudaSuccess)
    return MM_MOE_ECUDA;
  // dx [T, H] += dlogits [T, E] . W_router [E, H]
  if (launch_dense(c, GEMM_DENSE_NN, dlogits, W_router, dx, T, H, E) != cudaSuccess)
    return MM_MOE_ECUDA;
  return MM_MOE_OK;
}

// mx.cu -- MXFP8 quantise-dequantise of GEMM operands.
//
// Prime Mega MoE pages, "How does the fused kernel work?": MXFP8 is the layer's
// Blackwell low-precision type, and the training extension's fp8_bwd mode runs the
// forward in BF16 and the backward in FP8.  Each GEMM operand is quantised in
// blocks of 32 elements along that GEMM's contraction axis (OCP Microscaling v1.0):
// the block's shared scale is the power of two 2^(floor(log2 amax) - 8) (8 = the
// largest E4M3 exponent; 2^-127 for an all-zero block), each element is rounded to
// E4M3 (nearest even, saturating at +-448) after dividing by the scale.  The kernels
// here write the dequantised values e4m3 * scale as bf16, which holds them exactly,
// so a bf16 tensor-core GEMM with fp32 accumulation computes the MXFP8 product.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace mmmoe {

// Shared-scale exponent of a block with absolute maximum amax (>= 0).
__device__ __forceinline__ int mx_scale_exp(float amax) {
  if (!(amax > 0.f)) return -127;
  const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 127 - 8;
  return max(-127, min(127, e));  // a subnormal amax gives a very negative e: clamp
}

__device__ __forceinline__ float mx_qdq(float v, int e) {
  const float q = ldexpf(v, -e);
  const __nv_fp8_storage_t s = __nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3);
  const __half_raw hr = __nv_cvt_fp8_to_halfraw(s, __NV_E4M3);
  return ldexpf(__half2float(__half(hr)), e);
}

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ uint16_t to_bf(float f) {
  const __nv_bfloat16 h = __float2bfloat16_rn(f);  // exact for e4m3 * 2^e values
  return *reinterpret_cast<const uint16_t*>(&h);
}

__device__ __forceinline__ int64_t used_rows(int64_t rows, const int* meta) {
  const int64_t used = static_cast<int64_t>(__ldg(meta + META_NUM_TILES)) * BM;
  return used < rows ? used : rows;
}

// Blocks of 32 consecutive elements of each row ([rows, C], C % 32 == 0): a thread
// takes 8 elements, four neighbouring threads one block.  `meta` (device, may be
// null) caps the rows processed at meta[META_NUM_TILES] * BM, the end of the padded
// routed rows; the same holds for the column kernel below.
__global__ void __launch_bounds__(256) mx_qdq_rows_kernel(const uint4* __restrict__ in,
                                                          uint4* __restrict__ out, int64_t rows,
                                                          int C8, const int* __restrict__ meta) {
  if (meta != nullptr) rows = used_rows(rows, meta);
  const int64_t n = rows * C8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  // every thread of a warp runs the same number of iterations (shuffles below)
  for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x; i0 < n; i0 += stride) {
    const int64_t i = i0 + threadIdx.x;
    uint4 w = make_uint4(0, 0, 0, 0);
    if (i < n) w = __ldg(in + i);
    uint16_t h[8];
    *reinterpret_cast<uint4*>(h) = w;
    float v[8], amax = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] = bf(h[j]);
      amax = fmaxf(amax, fabsf(v[j]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int e = mx_scale_exp(amax);
#pragma unroll
    for (int j = 0; j < 8; ++j) h[j] = to_bf(mx_qdq(v[j], e));
    if (i < n) out[i] = *reinterpret_cast<uint4*>(h);
  }
}

// Blocks of 32 consecutive rows of each column ([rows, C], rows % 32 == 0, C even): a
// thread takes two neighbouring columns of one 32-row block, so a warp reads 128
// contiguous bytes of each row.
__global__ void __launch_bounds__(256) mx_qdq_cols_kernel(const uint32_t* __restrict__ in,
                                                          uint32_t* __restrict__ out, int64_t rows,
                                                          int C2, const int* __restrict__ meta) {
  if (meta != nullptr) rows = used_rows(rows, meta);
  const int64_t n = (rows / 32) * C2;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t blk = i / C2, c = i - blk * C2;
    const uint32_t* src = in + blk * 32 * C2 + c;
    uint32_t w[32];
    float amax0 = 0.f, amax1 = 0.f;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      w[r] = __ldg(src + static_cast<int64_t>(r) * C2);
      amax0 = fmaxf(amax0, fabsf(bf(static_cast<uint16_t>(w[r] & 0xFFFFu))));
      amax1 = fmaxf(amax1, fabsf(bf(static_cast<uint16_t>(w[r] >> 16))));
    }
    const int e0 = mx_scale_exp(amax0), e1 = mx_scale_exp(amax1);
    uint32_t* dst = out + blk * 32 * C2 + c;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      const uint32_t lo = to_bf(mx_qdq(bf(static_cast<uint16_t>(w[r] & 0xFFFFu)), e0));
      const uint32_t hi = to_bf(mx_qdq(bf(static_cast<uint16_t>(w[r] >> 16)), e1));
      dst[static_cast<int64_t>(r) * C2] = lo | (hi << 16);
    }
  }
}

cudaError_t launch_mx_qdq(const Ctx& c, const uint16_t* in, uint16_t* out, int64_t rows,
                          int64_t cols, bool along_rows, const int* meta) {
  const int grid = c.num_sms * 8;
  const int id = along_rows ? K_MX_QDQ_ROWS : K_MX_QDQ_COLS;
  prof_begin(c, id);
  if (along_rows)
    mx_qdq_rows_kernel<<<grid, 256, 0, c.stream>>>(reinterpret_cast<const uint4*>(in),
                                                   reinterpret_cast<uint4*>(out), rows,
                                                   static_cast<int>(cols / 8), meta);
  else
    mx_qdq_cols_kernel<<<grid, 256, 0, c.stream>>>(reinterpret_cast<const uint32_t*>(in),
                                                   reinterpret_cast<uint32_t*>(out), rows,
                                                   static_cast<int>(cols / 2), meta);
  prof_end(c, id);
  return cudaGetLastError();
}

}  // namespace mmmoe

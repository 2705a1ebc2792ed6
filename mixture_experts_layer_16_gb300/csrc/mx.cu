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
#include <cuda_runtime.h>

#include "internal.h"
#include "mx.cuh"

namespace mmmoe {

using mx::bf;
using mx::qdq2;
using mx::scale_exp;
using mx::to_bf;

__device__ __forceinline__ int64_t used_rows(int64_t rows, const int* meta) {
  const int64_t used = static_cast<int64_t>(__ldg(meta + META_NUM_TILES)) * BM;
  return used < rows ? used : rows;
}

// Blocks of 32 consecutive elements of each row ([rows, C], C % 32 == 0): a thread
// takes 8 elements (16 bytes), four neighbouring threads one block; each thread has
// ROW_UNROLL such pieces in flight.  `meta` (device, may be null) caps the rows
// processed at meta[META_NUM_TILES] * BM, the end of the padded routed rows; the
// same holds for the column kernel below.
constexpr int ROW_UNROLL = 4;

__global__ void __launch_bounds__(256) mx_qdq_rows_kernel(const uint4* in, uint4* out, int64_t rows,
                                                          int C8, const int* __restrict__ meta) {
  pdl_wait();
  pdl_trigger();
  if (meta != nullptr) rows = used_rows(rows, meta);
  const int64_t n = rows * C8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  // every thread of a warp runs the same number of iterations (shuffles below)
  for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x; i0 < n;
       i0 += stride * ROW_UNROLL) {
    uint4 w[ROW_UNROLL];
#pragma unroll
    for (int u = 0; u < ROW_UNROLL; ++u) {
      const int64_t i = i0 + u * stride + threadIdx.x;
      w[u] = i < n ? in[i] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < ROW_UNROLL; ++u) {
      uint16_t h[8];
      *reinterpret_cast<uint4*>(h) = w[u];
      float v[8], amax = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[j] = bf(h[j]);
        amax = fmaxf(amax, fabsf(v[j]));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const int e = scale_exp(amax);
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        qdq2(v[j], v[j + 1], e, e);
        h[j] = to_bf(v[j]);
        h[j + 1] = to_bf(v[j + 1]);
      }
      const int64_t i = i0 + u * stride + threadIdx.x;
      if (i < n) out[i] = *reinterpret_cast<uint4*>(h);
    }
  }
}

// Blocks of 32 consecutive rows of each column ([rows, C], rows % 32 == 0, C % 32 == 0).
// A CTA takes a tile of 32 rows x COL_TILE columns: thread t holds 8 columns
// (16 bytes) of rows t/64, t/64 + 4, ..., so a warp reads 512 contiguous bytes of a
// row; the four partial column maxima meet in shared memory.  With out_rows non-null
// the same read also yields the blocks along rows (four neighbouring lanes hold one
// 32-column block of a row), written to out_rows.  With a gather the rows come from a
// token-major `in` (padding rows read as zeros).
constexpr int COL_TILE = 512;

__global__ void __launch_bounds__(256) mx_qdq_cols_kernel(const uint4* in, uint4* out,
                                                          uint4* out_rows,
                                                          int64_t rows, int C8,
                                                          const int* __restrict__ meta,
                                                          const RowGather gather) {
  pdl_wait();
  pdl_trigger();
  __shared__ float part[4][COL_TILE];
  __shared__ int src_row[32];  // the row block's source rows (-1: zero)
  if (meta != nullptr) rows = used_rows(rows, meta);
  const int col_tiles = (C8 * 8 + COL_TILE - 1) / COL_TILE;
  const int64_t row_blocks = rows / 32;
  const int cg = threadIdx.x % 64, rs = threadIdx.x / 64;
  // a CTA takes whole 32-row blocks, their column tiles in turn: the block's source
  // rows are resolved once
  for (int64_t rb = blockIdx.x; rb < row_blocks; rb += gridDim.x) {
    if (threadIdx.x < 32) src_row[threadIdx.x] = gather_src(rb * 32 + threadIdx.x, gather);
    __syncthreads();
    for (int ct = 0; ct < col_tiles; ++ct) {
      const int c8 = ct * (COL_TILE / 8) + cg;
      const bool active = c8 < C8;
      uint4 w[8];
      float amax[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) amax[j] = 0.f;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int sr = src_row[rs + 4 * r];
        w[r] = active && sr >= 0 ? in[static_cast<int64_t>(sr) * C8 + c8] : make_uint4(0, 0, 0, 0);
        const uint16_t* h = reinterpret_cast<const uint16_t*>(&w[r]);
#pragma unroll
        for (int j = 0; j < 8; ++j) amax[j] = fmaxf(amax[j], fabsf(bf(h[j])));
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) part[rs][cg * 8 + j] = amax[j];
      if (out_rows != nullptr) {  // uniform: every lane takes part in the shuffles
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          uint4 o = w[r];
          uint16_t* h = reinterpret_cast<uint16_t*>(&o);
          float ra = 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) ra = fmaxf(ra, fabsf(bf(h[j])));
          ra = fmaxf(ra, __shfl_xor_sync(0xffffffffu, ra, 1));
          ra = fmaxf(ra, __shfl_xor_sync(0xffffffffu, ra, 2));
          const int re = scale_exp(ra);
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            float x0 = bf(h[j]), x1 = bf(h[j + 1]);
            qdq2(x0, x1, re, re);
            h[j] = to_bf(x0);
            h[j + 1] = to_bf(x1);
          }
          if (active) out_rows[rb * 32 * C8 + c8 + static_cast<int64_t>(rs + 4 * r) * C8] = o;
        }
      }
      __syncthreads();
      int e[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = cg * 8 + j;
        e[j] = scale_exp(fmaxf(fmaxf(part[0][c], part[1][c]), fmaxf(part[2][c], part[3][c])));
      }
      __syncthreads();  // part[] (and, at the next row block, src_row[]) is rewritten
      if (active) {
        uint4* dst = out + rb * 32 * C8 + c8;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          uint16_t* h = reinterpret_cast<uint16_t*>(&w[r]);
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            float x0 = bf(h[j]), x1 = bf(h[j + 1]);
            qdq2(x0, x1, e[j], e[j + 1]);
            h[j] = to_bf(x0);
            h[j + 1] = to_bf(x1);
          }
          dst[static_cast<int64_t>(rs + 4 * r) * C8] = w[r];
        }
      }
    }
  }
}

cudaError_t launch_mx_qdq(const Ctx& c, const uint16_t* in, uint16_t* out, int64_t rows,
                          int64_t cols, bool along_rows, const int* meta, uint16_t* out_rows,
                          RowGather gather) {
  const int id = along_rows ? K_MX_QDQ_ROWS : K_MX_QDQ_COLS;
  prof_begin(c, id);
  if (along_rows) {
    launch_k(c.stream, mx_qdq_rows_kernel, dim3(c.num_sms * 8), dim3(256), 0,
        reinterpret_cast<const uint4*>(in), reinterpret_cast<uint4*>(out), rows,
        static_cast<int>(cols / 8), meta);
  } else {
    // with `meta` the row count is known only on the device: size the grid for the
    // capacity and let surplus CTAs exit
    const int64_t blocks = rows / 32;  // 32-row blocks (a CTA takes whole ones)
    const int64_t grid = blocks < c.num_sms * 6 ? blocks : c.num_sms * 6;
    launch_k(c.stream, mx_qdq_cols_kernel, dim3(static_cast<int>(grid > 0 ? grid : 1)), dim3(256), 0,
        reinterpret_cast<const uint4*>(in), reinterpret_cast<uint4*>(out),
        reinterpret_cast<uint4*>(out_rows), rows, static_cast<int>(cols / 8), meta, gather);
  }
  prof_end(c, id);
  return cudaGetLastError();
}

}  // namespace mmmoe

using namespace mmmoe;

extern "C" MM_MOE_API mm_moe_status mm_moe_mx_qdq(const uint16_t* in, uint16_t* out, int64_t rows,
                                                  int64_t cols, int axis, void* stream) {
  if (in == nullptr || out == nullptr || rows < 1 || cols < 1) return MM_MOE_EINVAL;
  if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) % 16 != 0)
    return MM_MOE_EINVAL;
  if (axis == 1 ? cols % 32 != 0 : (axis != 0 || rows % 32 != 0 || cols % 8 != 0))
    return MM_MOE_EINVAL;
  if (rows > (int64_t{1} << 40) / cols) return MM_MOE_EINVAL;
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MM_MOE_ECUDA;
  if (major != 10 || minor != 3) return MM_MOE_ENOTSUP;
  int launches = 0;
  const Ctx c{static_cast<cudaStream_t>(stream), sms, &launches};
  if (launch_mx_qdq(c, in, out, rows, cols, axis == 1, nullptr) != cudaSuccess)
    return MM_MOE_ECUDA;
  return MM_MOE_OK;
}

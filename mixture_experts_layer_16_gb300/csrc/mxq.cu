// mxq.cu -- MXFP8 quantisation of GEMM operands into what the block-scaled tensor
// cores read: e4m3 codes (one byte per element, the operand's row-major layout) and
// E8M0 block scales in the atom arrangement of mx::sf_offset.
//
// Prime Mega MoE pages, "How does the fused kernel work?": MXFP8 is the layer's
// Blackwell low-precision type (fp8_bwd: BF16 forward, FP8 backward).  OCP
// Microscaling v1.0: a block of 32 elements along the GEMM's contraction axis shares
// the scale 2^(floor(log2 amax) - 8) (8 = the largest E4M3 exponent; 2^-127 for an
// all-zero block) and each element is rounded to E4M3 (nearest even, saturating at
// +-448) after dividing by it.  The input is always the bf16 value the layer stores.
#include <cuda_runtime.h>

#include "internal.h"
#include "mx.cuh"

namespace mmmoe {

using mx::bf;
using mx::codes8;
using mx::e8m0;
using mx::scale_exp;
using mx::sf_offset;

__device__ __forceinline__ int64_t rows_in_use(int64_t rows, const int* meta) {
  if (meta == nullptr) return rows;
  const int64_t used = static_cast<int64_t>(__ldg(meta + META_NUM_TILES)) * BM;
  return used < rows ? used : rows;
}

// ---------------------------------------------------------------- blocks along rows
// [rows, K] bf16, K % 128 == 0.  A thread takes 8 elements (16 bytes in, 8 bytes of
// codes out); four neighbouring lanes form a block, sixteen a group of four blocks
// whose four scale codes make one 32-bit word of the scale layout (written by the
// group's first lane).
constexpr int QROW_UNROLL = 4;

__global__ void __launch_bounds__(256) mxq_rows_kernel(const uint4* __restrict__ in,
                                                       uint2* __restrict__ codes,
                                                       uint8_t* __restrict__ sf, int64_t rows,
                                                       int K8, int64_t mn_blocks,
                                                       const int* __restrict__ meta) {
  rows = rows_in_use(rows, meta);
  const int64_t n = rows * K8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int lane = threadIdx.x & 31;
  // every lane of a warp runs the same iterations (shuffles below); piece i sits in
  // lane i % 32, so a block's four pieces and a group's sixteen are lane-aligned
  for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x; i0 < n;
       i0 += stride * QROW_UNROLL) {
    uint4 w[QROW_UNROLL];
#pragma unroll
    for (int u = 0; u < QROW_UNROLL; ++u) {
      const int64_t i = i0 + u * stride + threadIdx.x;
      w[u] = i < n ? __ldg(in + i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < QROW_UNROLL; ++u) {
      const int64_t i = i0 + u * stride + threadIdx.x;
      const uint16_t* h = reinterpret_cast<const uint16_t*>(&w[u]);
      float v[8], amax = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[j] = bf(h[j]);
        amax = fmaxf(amax, fabsf(v[j]));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const int e = scale_exp(amax);
      const uint2 c = codes8(v, e);
      // the group's word: the exponents of its lanes 0, 4, 8, 12
      const int g0 = lane & ~15;
      uint32_t word = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b)
        word |= e8m0(__shfl_sync(0xffffffffu, e, g0 + 4 * b)) << (8 * b);
      if (i < n) {
        codes[i] = c;
        if ((lane & 15) == 0) {
          const int64_t row = i / K8;
          const int64_t kb = (i - row * K8) / 4;
          *reinterpret_cast<uint32_t*>(sf + sf_offset(row, kb, mn_blocks)) = word;
        }
      }
    }
  }
}

// ---------------------------------------------------------------- blocks down columns
// [rows, C] bf16 (rows % 32 == 0, C % 128 == 0): blocks of 32 rows of each column,
// the operand layout of a GEMM whose K runs along the rows (its MMA rows are the
// columns).  A CTA takes whole 32-row blocks (their source rows resolved once) and
// their column tiles in turn: thread t holds 8 columns (16 bytes) of rows t/64,
// t/64 + 4, ..., the four partial column maxima meet in shared memory.  The scale of
// column c in row block rb is byte sf_offset(c, rb, C / 128).  With codes_rows
// non-null the same read also gives the blocks along the rows (four neighbouring
// lanes hold one 32-column block of a row; scales at sf_offset(row, col / 32,
// rows / 128) of sf_rows).  With a gather the rows come from a token-major source
// (padding rows read as zeros).
constexpr int QCOL_TILE = 512;

__global__ void __launch_bounds__(256) mxq_cols_kernel(const uint4* __restrict__ in,
                                                       uint2* __restrict__ codes,
                                                       uint8_t* __restrict__ sf,
                                                       uint2* __restrict__ codes_rows,
                                                       uint8_t* __restrict__ sf_rows,
                                                       int64_t rows, int64_t rows_total,
                                                       int C8, const int* __restrict__ meta,
                                                       const RowGather gather) {
  __shared__ float part[4][QCOL_TILE];
  __shared__ int src_row[32];  // the row block's source rows (-1: zero)
  rows = rows_in_use(rows, meta);
  const int col_tiles = (C8 * 8 + QCOL_TILE - 1) / QCOL_TILE;
  const int64_t row_blocks = rows / 32;
  const int64_t mnb = C8 / 16;                 // 128-column blocks
  const int64_t mnb_rows = rows_total / 128;   // 128-row blocks (row scales)
  const int cg = threadIdx.x % 64, rs = threadIdx.x / 64, lane = threadIdx.x & 31;
  for (int64_t rb = blockIdx.x; rb < row_blocks; rb += gridDim.x) {
    if (threadIdx.x < 32) src_row[threadIdx.x] = gather_src(rb * 32 + threadIdx.x, gather);
    __syncthreads();
    for (int ct = 0; ct < col_tiles; ++ct) {
      const int c8 = ct * (QCOL_TILE / 8) + cg;
      const bool active = c8 < C8;
      uint4 w[8];
      float amax[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) amax[j] = 0.f;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int sr = src_row[rs + 4 * r];
        w[r] = active && sr >= 0 ? __ldg(in + static_cast<int64_t>(sr) * C8 + c8)
                                 : make_uint4(0, 0, 0, 0);
        const uint16_t* h = reinterpret_cast<const uint16_t*>(&w[r]);
#pragma unroll
        for (int j = 0; j < 8; ++j) amax[j] = fmaxf(amax[j], fabsf(bf(h[j])));
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) part[rs][cg * 8 + j] = amax[j];
      if (codes_rows != nullptr) {  // uniform: every lane takes part in the shuffles
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const uint16_t* h = reinterpret_cast<const uint16_t*>(&w[r]);
          float v[8], ra = 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            v[j] = bf(h[j]);
            ra = fmaxf(ra, fabsf(v[j]));
          }
          ra = fmaxf(ra, __shfl_xor_sync(0xffffffffu, ra, 1));
          ra = fmaxf(ra, __shfl_xor_sync(0xffffffffu, ra, 2));
          const int re = scale_exp(ra);
          const int g0 = lane & ~15;
          uint32_t word = 0;
#pragma unroll
          for (int b = 0; b < 4; ++b)
            word |= e8m0(__shfl_sync(0xffffffffu, re, g0 + 4 * b)) << (8 * b);
          const int64_t row = rb * 32 + rs + 4 * r;
          if (active) {
            codes_rows[row * C8 + c8] = codes8(v, re);
            if ((lane & 15) == 0)
              *reinterpret_cast<uint32_t*>(sf_rows + sf_offset(row, c8 / 4, mnb_rows)) = word;
          }
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
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const uint16_t* h = reinterpret_cast<const uint16_t*>(&w[r]);
          uint32_t p[4];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            p[j] = mx::codes2e(bf(h[2 * j]), e[2 * j], bf(h[2 * j + 1]), e[2 * j + 1]);
          codes[(rb * 32 + rs + 4 * r) * C8 + c8] =
              make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
        }
        if (rs == 0) {
#pragma unroll
          for (int j = 0; j < 8; ++j) sf[sf_offset(static_cast<int64_t>(c8) * 8 + j, rb, mnb)] = e8m0(e[j]);
        }
      }
    }
  }
}

cudaError_t launch_mxq(const Ctx& c, const MxqArgs& a) {
  if (a.along_rows) {
    prof_begin(c, K_MXQ_ROWS);
    mxq_rows_kernel<<<c.num_sms * 8, 256, 0, c.stream>>>(
        reinterpret_cast<const uint4*>(a.in), reinterpret_cast<uint2*>(a.codes), a.sf, a.rows,
        static_cast<int>(a.cols / 8), a.rows / 128, a.meta);
    prof_end(c, K_MXQ_ROWS);
  } else {
    // with `meta` the row count is known only on the device: size the grid for the
    // capacity and let surplus CTAs exit
    const int64_t blocks = a.rows / 32;
    const int64_t grid = blocks < c.num_sms * 6 ? blocks : c.num_sms * 6;
    prof_begin(c, K_MXQ_COLS);
    mxq_cols_kernel<<<static_cast<int>(grid > 0 ? grid : 1), 256, 0, c.stream>>>(
        reinterpret_cast<const uint4*>(a.in), reinterpret_cast<uint2*>(a.codes), a.sf,
        reinterpret_cast<uint2*>(a.codes_rows), a.sf_rows, a.rows, a.rows,
        static_cast<int>(a.cols / 8), a.meta, a.gather);
    prof_end(c, K_MXQ_COLS);
  }
  return cudaGetLastError();
}

}  // namespace mmmoe

using namespace mmmoe;

extern "C" MM_MOE_API mm_moe_status mm_moe_mx_quantize(const uint16_t* in, uint8_t* codes,
                                                       uint8_t* scales, int64_t rows,
                                                       int64_t cols, int axis, void* stream) {
  if (in == nullptr || codes == nullptr || scales == nullptr || rows < 1 || cols < 1)
    return MM_MOE_EINVAL;
  if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(codes) |
       reinterpret_cast<uintptr_t>(scales)) % 16 != 0)
    return MM_MOE_EINVAL;
  if (rows % 128 != 0 || cols % 128 != 0 || (axis != 0 && axis != 1)) return MM_MOE_EINVAL;
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
  MxqArgs a{};
  a.in = in;
  a.codes = codes;
  a.sf = scales;
  a.rows = rows;
  a.cols = cols;
  a.along_rows = axis == 1;
  if (launch_mxq(c, a) != cudaSuccess) return MM_MOE_ECUDA;
  return MM_MOE_OK;
}

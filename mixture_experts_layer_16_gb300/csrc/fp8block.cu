// fp8block.cu -- blockwise FP8 quantisation of GEMM operands.
//
// Prime Mega MoE pages, "How does the fused kernel work?": blockwise FP8 is the Hopper
// low-precision type of the fused kernel.  Here it takes the form Blackwell tensor
// cores take: activations in blocks of 128 elements along each GEMM's contraction
// axis (128 rows along the token axis for the weight gradients), weights in 128 x 128
// blocks, one power-of-two scale per block, 2^ceil(log2(amax / 448)) -- the smallest
// that keeps every element within E4M3's +-448 -- and elements rounded to E4M3 (nearest
// even).  The layer's GEMMs read e4m3 codes and E8M0 scale codes (the fbq_* kernels) on
// the block-scaled tensor cores; the fb_* kernels write the dequantised values
// e4m3 * scale as bf16, which holds them exactly (mm_moe_fp8_block_qdq).
#include <cuda_runtime.h>

#include "fp8block.cuh"
#include "internal.h"
#include "mx.cuh"

namespace mmmoe {

using mx::bf;
using mx::codes4;
using mx::qdq2;
using mx::to_bf;
using fb::ceil_exp;
using fb::FB;

__device__ __forceinline__ uint4 qdq8(uint4 w, const int (&e)[8]) {
  uint16_t* h = reinterpret_cast<uint16_t*>(&w);
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    float x0 = bf(h[j]), x1 = bf(h[j + 1]);
    qdq2(x0, x1, e[j], e[j + 1]);
    h[j] = to_bf(x0);
    h[j + 1] = to_bf(x1);
  }
  return w;
}

__device__ __forceinline__ float amax8(const uint4 w) {
  const uint16_t* h = reinterpret_cast<const uint16_t*>(&w);
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(bf(h[j])));
  return m;
}

__device__ __forceinline__ int64_t used(int64_t rows, const int* meta) {
  if (meta == nullptr) return rows;
  const int64_t u = static_cast<int64_t>(__ldg(meta + META_NUM_TILES)) * BM;
  return u < rows ? u : rows;
}

// Blocks of 128 consecutive elements of each row ([rows, C], C % 128 == 0): a thread
// takes 8 elements, 16 neighbouring lanes one block.
__global__ void __launch_bounds__(256) fb_rows_kernel(const uint4* in, uint4* out, int64_t rows,
                                                      int C8, const int* __restrict__ meta) {
  pdl_wait();
  pdl_trigger();
  const int64_t n = used(rows, meta) * C8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  // every lane of a warp runs the same iterations (shuffles)
  for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x; i0 < n; i0 += stride) {
    const int64_t i = i0 + threadIdx.x;
    const uint4 w = i < n ? in[i] : make_uint4(0, 0, 0, 0);
    float m = amax8(w);
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    int e[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) e[j] = ceil_exp(m);
    if (i < n) out[i] = qdq8(w, e);
  }
}

// Blocks of 128 consecutive rows of each column ([rows, C], rows % 128 == 0, C % 8 ==
// 0), tiles of 128 rows x 512 columns: thread t holds 8 columns of rows t/64, t/64 + 4,
// ...; a first pass finds the column maxima (met in shared memory), a second reads
// the tile again (from L2) and writes it quantised.  With out_rows non-null the
// second pass also writes the blocks along rows (16 lanes hold one 128-column block of
// a row; C % 128 == 0).  out and out_rows may equal in: every element is read and
// written by one thread, in that order.  With a gather the rows come from a
// token-major `in` (padding rows read as zeros).
constexpr int FB_TILE = 512;

__global__ void __launch_bounds__(256) fb_cols_kernel(const uint4* in, uint4* out,
                                                      uint4* out_rows, int64_t rows, int C8,
                                                      const int* __restrict__ meta,
                                                      const RowGather gather) {
  pdl_wait();
  pdl_trigger();
  __shared__ float part[4][FB_TILE];
  __shared__ int src_row[FB];  // the tile's source rows (-1: zero), resolved once
  const int64_t R = used(rows, meta);
  const int col_tiles = (C8 * 8 + FB_TILE - 1) / FB_TILE;
  const int64_t tiles = (R / FB) * col_tiles;
  const int cg = threadIdx.x % 64, rs = threadIdx.x / 64;
  for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int64_t rb = tile / col_tiles;
    const int c8 = static_cast<int>(tile - rb * col_tiles) * (FB_TILE / 8) + cg;
    const bool active = c8 < C8;
    const int64_t base = rb * FB * C8 + c8;
    __syncthreads();  // the previous tile's second pass has read src_row[]
    if (threadIdx.x < FB) src_row[threadIdx.x] = gather_src(rb * FB + threadIdx.x, gather);
    __syncthreads();
    float m[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) m[j] = 0.f;
    if (active) {
#pragma unroll 8
      for (int r = 0; r < FB / 4; ++r) {
        const int sr = src_row[rs + 4 * r];
        const uint4 w = sr >= 0 ? in[static_cast<int64_t>(sr) * C8 + c8] : make_uint4(0, 0, 0, 0);
        const uint16_t* h = reinterpret_cast<const uint16_t*>(&w);
#pragma unroll
        for (int j = 0; j < 8; ++j) m[j] = fmaxf(m[j], fabsf(bf(h[j])));
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) part[rs][cg * 8 + j] = m[j];
    __syncthreads();
    int e[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = cg * 8 + j;
      e[j] = ceil_exp(fmaxf(fmaxf(part[0][c], part[1][c]), fmaxf(part[2][c], part[3][c])));
    }
    __syncthreads();  // part[] is rewritten by the next tile
#pragma unroll 4
    for (int r = 0; r < FB / 4; ++r) {
      const int64_t at = base + static_cast<int64_t>(rs + 4 * r) * C8;
      const int sr = src_row[rs + 4 * r];
      const uint4 w = active && sr >= 0 ? in[static_cast<int64_t>(sr) * C8 + c8]
                                        : make_uint4(0, 0, 0, 0);
      if (out_rows != nullptr) {  // uniform: every lane takes part in the shuffles
        float rm = amax8(w);
#pragma unroll
        for (int off = 1; off < 16; off <<= 1)
          rm = fmaxf(rm, __shfl_xor_sync(0xffffffffu, rm, off));
        int re[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) re[j] = ceil_exp(rm);
        if (active) out_rows[at] = qdq8(w, re);
      }
      if (active) out[at] = qdq8(w, e);
    }
  }
}

// 128 x 128 tiles of a [rows, C] matrix (rows % 128 == 0, C % 128 == 0): one CTA per
// tile (grid-stride), 16 lanes per tile row, 16 rows per pass, 8 passes.
__global__ void __launch_bounds__(256) fb_tiles_kernel(const uint4* in, uint4* out, int64_t rows,
                                                       int C8) {
  pdl_wait();
  pdl_trigger();
  __shared__ float wmax[8];
  const int col_tiles = C8 / (FB / 8);
  const int64_t tiles = (rows / FB) * col_tiles;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cq = threadIdx.x % 16, rq = threadIdx.x / 16;
  for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int64_t rb = tile / col_tiles;
    const int cb = static_cast<int>(tile - rb * col_tiles);
    const int64_t base = rb * FB * C8 + cb * (FB / 8) + cq;
    uint4 w[8];
    float m = 0.f;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      w[p] = in[base + static_cast<int64_t>(rq + 16 * p) * C8];
      m = fmaxf(m, amax8(w[p]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) wmax[warp] = m;
    __syncthreads();
    float t = wmax[0];
#pragma unroll
    for (int q = 1; q < 8; ++q) t = fmaxf(t, wmax[q]);
    __syncthreads();  // wmax[] is rewritten by the next tile
    int e[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) e[j] = ceil_exp(t);
#pragma unroll
    for (int p = 0; p < 8; ++p) out[base + static_cast<int64_t>(rq + 16 * p) * C8] = qdq8(w[p], e);
  }
}

// ---------------------------------------------------------------- codes and scales
// The same blocks in the form the block-scaled tensor cores read (the GEMMs' MXFP8
// instantiations): e4m3 codes, one byte per element in the operand's own [rows, C]
// layout, and E8M0 scale codes in the atom arrangement of mx::sf_offset.  A 128-element
// block is four 32-element scale blocks with the same scale, i.e. one 32-bit word of
// four equal codes (along the rows: the word of the row and 128-column block; down the
// columns: the word of the column and 128-row block).
__device__ __forceinline__ uint2 codes8(const uint4 w, float m) {
  return make_uint2(mx::codes4(w.x, w.y, m, m, m, m), mx::codes4(w.z, w.w, m, m, m, m));
}
__device__ __forceinline__ uint2 codes8c(const uint4 w, const float (&m)[8]) {
  return make_uint2(mx::codes4(w.x, w.y, m[0], m[1], m[2], m[3]),
                    mx::codes4(w.z, w.w, m[4], m[5], m[6], m[7]));
}
__device__ __forceinline__ uint32_t sf_word(int e) { return mx::e8m0(e) * 0x01010101u; }

// Blocks of 128 consecutive elements of each row ([rows, C], C % 128 == 0): a thread
// takes 8 elements, 16 neighbouring lanes one block; the block's first lane writes its
// scale word (row, 128-column block) over mnb = rows / 128 row blocks.
__global__ void __launch_bounds__(256) fbq_rows_kernel(const uint4* in, uint2* codes, uint8_t* sf,
                                                       int64_t rows, int C8, int64_t mnb,
                                                       const int* __restrict__ meta) {
  pdl_wait();
  pdl_trigger();
  const int64_t n = used(rows, meta) * C8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  // every lane of a warp runs the same iterations (shuffles)
  for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x; i0 < n; i0 += stride) {
    const int64_t i = i0 + threadIdx.x;
    const uint4 w = i < n ? in[i] : make_uint4(0, 0, 0, 0);
    float m = amax8(w);
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const int e = ceil_exp(m);
    if (i < n) {
      codes[i] = codes8(w, mx::pow2f(-e));
      if ((i & 15) == 0) {
        const int64_t row = i / C8;
        const int col = static_cast<int>(i - row * C8) * 8;
        *reinterpret_cast<uint32_t*>(sf + mx::sf_offset(row, col / 32, mnb)) = sf_word(e);
      }
    }
  }
}

// Blocks of 128 consecutive rows of each column ([rows, C], rows % 128 == 0, C % 8 == 0),
// as fb_cols_kernel (two passes over 128 x 512 tiles, the second from L2): codes to
// `codes` and the scale words (column, 128-row block) over C / 128 column blocks to
// `sf`; with codes_rows non-null also the blocks along the rows (C % 128 == 0), scale
// words over rows_total / 128 row blocks to sf_rows.  With a gather the rows come from
// a token-major `in` (padding rows read as zeros).
__global__ void __launch_bounds__(256) fbq_cols_kernel(const uint4* in, uint2* codes, uint8_t* sf,
                                                       uint2* codes_rows, uint8_t* sf_rows,
                                                       int64_t rows, int C8,
                                                       const int* __restrict__ meta,
                                                       const RowGather gather) {
  pdl_wait();
  pdl_trigger();
  __shared__ float part[4][FB_TILE];
  __shared__ int src_row[FB];
  const int64_t R = used(rows, meta);
  const int col_tiles = (C8 * 8 + FB_TILE - 1) / FB_TILE;
  const int64_t tiles = (R / FB) * col_tiles;
  const int64_t mnb_cols = C8 / 16, mnb_rows = rows / FB;
  const int cg = threadIdx.x % 64, rs = threadIdx.x / 64;
  for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int64_t rb = tile / col_tiles;
    const int c8 = static_cast<int>(tile - rb * col_tiles) * (FB_TILE / 8) + cg;
    const bool active = c8 < C8;
    const int64_t base = rb * FB * C8 + c8;
    __syncthreads();  // the previous tile's second pass has read src_row[]
    if (threadIdx.x < FB) src_row[threadIdx.x] = gather_src(rb * FB + threadIdx.x, gather);
    __syncthreads();
    float m[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) m[j] = 0.f;
    if (active) {
#pragma unroll 8
      for (int r = 0; r < FB / 4; ++r) {
        const int sr = src_row[rs + 4 * r];
        const uint4 w = sr >= 0 ? in[static_cast<int64_t>(sr) * C8 + c8] : make_uint4(0, 0, 0, 0);
        const uint16_t* h = reinterpret_cast<const uint16_t*>(&w);
#pragma unroll
        for (int j = 0; j < 8; ++j) m[j] = fmaxf(m[j], fabsf(bf(h[j])));
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) part[rs][cg * 8 + j] = m[j];
    __syncthreads();
    int e[8];
    float mul[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = cg * 8 + j;
      e[j] = ceil_exp(fmaxf(fmaxf(part[0][c], part[1][c]), fmaxf(part[2][c], part[3][c])));
      mul[j] = mx::pow2f(-e[j]);
    }
    __syncthreads();  // part[] is rewritten by the next tile
    if (active && rs == 0) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint32_t*>(sf + mx::sf_offset(c8 * 8 + j, 4 * rb, mnb_cols)) =
            sf_word(e[j]);
    }
#pragma unroll 4
    for (int r = 0; r < FB / 4; ++r) {
      const int64_t at = base + static_cast<int64_t>(rs + 4 * r) * C8;
      const int sr = src_row[rs + 4 * r];
      const uint4 w = active && sr >= 0 ? in[static_cast<int64_t>(sr) * C8 + c8]
                                        : make_uint4(0, 0, 0, 0);
      if (codes_rows != nullptr) {  // uniform: every lane takes part in the shuffles
        float rm = amax8(w);
#pragma unroll
        for (int off = 1; off < 16; off <<= 1)
          rm = fmaxf(rm, __shfl_xor_sync(0xffffffffu, rm, off));
        const int re = ceil_exp(rm);
        if (active) {
          codes_rows[at] = codes8(w, mx::pow2f(-re));
          if ((cg & 15) == 0)
            *reinterpret_cast<uint32_t*>(
                sf_rows + mx::sf_offset(rb * FB + rs + 4 * r, c8 / 4, mnb_rows)) = sf_word(re);
        }
      }
      if (active) codes[at] = codes8c(w, mul);
    }
  }
}

// 128 x 128 tiles of a weight matrix [rows, C] (rows % 128 == 0, C % 128 == 0), one CTA
// per tile: the codes (one copy, whichever axis a GEMM contracts) and the tile's scale in
// both arrangements, each one whole 512-byte atom of equal codes: sf_k for the GEMMs
// that contract the columns (MMA rows = the matrix rows, rows / 128 row blocks), sf_mn
// for those that contract the rows (MMA rows = the columns, C / 128 column blocks).
__global__ void __launch_bounds__(256) fbq_tiles_kernel(const uint4* in, uint2* codes,
                                                        uint8_t* sf_k, uint8_t* sf_mn,
                                                        int64_t rows, int C8) {
  pdl_wait();
  pdl_trigger();
  __shared__ float wmax[8];
  const int col_tiles = C8 / (FB / 8);
  const int64_t tiles = (rows / FB) * col_tiles;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cq = threadIdx.x % 16, rq = threadIdx.x / 16;
  for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int64_t rb = tile / col_tiles;
    const int cb = static_cast<int>(tile - rb * col_tiles);
    const int64_t base = rb * FB * C8 + cb * (FB / 8) + cq;
    uint4 w[8];
    float m = 0.f;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      w[p] = in[base + static_cast<int64_t>(rq + 16 * p) * C8];
      m = fmaxf(m, amax8(w[p]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) wmax[warp] = m;
    __syncthreads();
    float t = wmax[0];
#pragma unroll
    for (int q = 1; q < 8; ++q) t = fmaxf(t, wmax[q]);
    __syncthreads();  // wmax[] is rewritten by the next tile
    const int e = ceil_exp(t);
    const float mul = mx::pow2f(-e);
#pragma unroll
    for (int p = 0; p < 8; ++p) codes[base + static_cast<int64_t>(rq + 16 * p) * C8] = codes8(w[p], mul);
    const uint32_t word = sf_word(e);
    if (threadIdx.x < 64) {  // 32 x 16 bytes per atom
      uint8_t* atom = threadIdx.x < 32 ? sf_k + (static_cast<int64_t>(cb) * (rows / FB) + rb) * 512
                                       : sf_mn + (rb * (C8 / 16) + cb) * 512;
      reinterpret_cast<uint4*>(atom)[threadIdx.x & 31] = make_uint4(word, word, word, word);
    }
  }
}

cudaError_t launch_fbq(const Ctx& c, const FbqArgs& a) {
  const int C8 = static_cast<int>(a.cols / 8);
  const uint4* i4 = reinterpret_cast<const uint4*>(a.in);
  uint2* c2 = reinterpret_cast<uint2*>(a.codes);
  if (a.layout == FB_ROWS) {
    prof_begin(c, K_FBQ_ROWS);
    launch_k(c.stream, fbq_rows_kernel, dim3(c.num_sms * 8), dim3(256), 0, i4, c2, a.sf, a.rows,
             C8, a.rows / FB, a.meta);
    prof_end(c, K_FBQ_ROWS);
  } else if (a.layout == FB_COLS) {
    const int64_t tiles = (a.rows / FB) * ((a.cols + FB_TILE - 1) / FB_TILE);
    const int64_t cap = static_cast<int64_t>(c.num_sms) * 4;
    const int grid = static_cast<int>(tiles < cap ? (tiles > 0 ? tiles : 1) : cap);
    prof_begin(c, K_FBQ_COLS);
    launch_k(c.stream, fbq_cols_kernel, dim3(grid), dim3(256), 0, i4, c2, a.sf,
             reinterpret_cast<uint2*>(a.codes_rows), a.sf_rows, a.rows, C8, a.meta, a.gather);
    prof_end(c, K_FBQ_COLS);
  } else {
    const int64_t tiles = (a.rows / FB) * (a.cols / FB);
    const int64_t cap = static_cast<int64_t>(c.num_sms) * 8;
    const int grid = static_cast<int>(tiles < cap ? (tiles > 0 ? tiles : 1) : cap);
    prof_begin(c, K_FBQ_TILES);
    launch_k(c.stream, fbq_tiles_kernel, dim3(grid), dim3(256), 0, i4, c2, a.sf, a.sf_mn, a.rows,
             C8);
    prof_end(c, K_FBQ_TILES);
  }
  return cudaGetLastError();
}

cudaError_t launch_fb_qdq(const Ctx& c, const uint16_t* in, uint16_t* out, int64_t rows,
                          int64_t cols, int layout, const int* meta, uint16_t* out_rows,
                          RowGather gather) {
  const int C8 = static_cast<int>(cols / 8);
  const uint4* i4 = reinterpret_cast<const uint4*>(in);
  uint4* o4 = reinterpret_cast<uint4*>(out);
  if (layout == FB_ROWS) {
    prof_begin(c, K_FB_ROWS);
    launch_k(c.stream, fb_rows_kernel, dim3(c.num_sms * 8), dim3(256), 0, i4, o4, rows, C8, meta);
    prof_end(c, K_FB_ROWS);
  } else if (layout == FB_COLS) {
    const int64_t tiles = (rows / FB) * ((cols + FB_TILE - 1) / FB_TILE);
    const int64_t cap = static_cast<int64_t>(c.num_sms) * 4;
    const int grid = static_cast<int>(tiles < cap ? (tiles > 0 ? tiles : 1) : cap);
    prof_begin(c, K_FB_COLS);
    launch_k(c.stream, fb_cols_kernel, dim3(grid), dim3(256), 0, i4, o4, reinterpret_cast<uint4*>(out_rows), rows,
                                               C8, meta, gather);
    prof_end(c, K_FB_COLS);
  } else {
    const int64_t tiles = (rows / FB) * (cols / FB);
    const int64_t cap = static_cast<int64_t>(c.num_sms) * 8;
    const int grid = static_cast<int>(tiles < cap ? (tiles > 0 ? tiles : 1) : cap);
    prof_begin(c, K_FB_TILES);
    launch_k(c.stream, fb_tiles_kernel, dim3(grid), dim3(256), 0, i4, o4, rows, C8);
    prof_end(c, K_FB_TILES);
  }
  return cudaGetLastError();
}

}  // namespace mmmoe

using namespace mmmoe;

extern "C" MM_MOE_API mm_moe_status mm_moe_fp8_block_qdq(const uint16_t* in, uint16_t* out,
                                                         int64_t rows, int64_t cols, int layout,
                                                         void* stream) {
  if (in == nullptr || out == nullptr || rows < 1 || cols < 1) return MM_MOE_EINVAL;
  if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) % 16 != 0)
    return MM_MOE_EINVAL;
  const bool ok = layout == FB_ROWS   ? cols % FB == 0
                  : layout == FB_COLS ? (rows % FB == 0 && cols % 8 == 0)
                  : layout == FB_TILES ? (rows % FB == 0 && cols % FB == 0)
                                        : false;
  if (!ok || rows > (int64_t{1} << 40) / cols) return MM_MOE_EINVAL;
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MM_MOE_ECUDA;
  if (major != 10 || minor != 3) return MM_MOE_ENOTSUP;
  int launches = 0;
  const Ctx c{static_cast<cudaStream_t>(stream), sms, &launches};
  if (launch_fb_qdq(c, in, out, rows, cols, layout, nullptr, nullptr) != cudaSuccess)
    return MM_MOE_ECUDA;
  return MM_MOE_OK;
}

extern "C" MM_MOE_API mm_moe_status mm_moe_fp8_block_quantize(const uint16_t* in, uint8_t* codes,
                                                              uint8_t* scales, int64_t rows,
                                                              int64_t cols, int layout,
                                                              void* stream) {
  if (in == nullptr || codes == nullptr || scales == nullptr || rows < 1 || cols < 1)
    return MM_MOE_EINVAL;
  if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(codes) |
       reinterpret_cast<uintptr_t>(scales)) % 16 != 0)
    return MM_MOE_EINVAL;
  if (rows % FB != 0 || cols % FB != 0 || layout < FB_ROWS || layout > FB_TILES)
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
  FbqArgs a{};
  a.in = in;
  a.codes = codes;
  a.sf = scales;
  a.sf_mn = scales + rows * cols / 32;
  a.rows = rows;
  a.cols = cols;
  a.layout = layout;
  if (launch_fbq(c, a) != cudaSuccess) return MM_MOE_ECUDA;
  return MM_MOE_OK;
}

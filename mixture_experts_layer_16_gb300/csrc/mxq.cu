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
#include "ptx.cuh"

namespace mmmoe {

using mx::bf;
using mx::codes8;
using mx::e8m0;
using mx::scale_exp;
using mx::bf16_scale_exp;
using mx::codes4;
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
  pdl_wait();
  pdl_trigger();
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
// columns); the scale of column c in row block rb is byte sf_offset(c, rb, C / 128).
// With codes_rows non-null the same read also gives the blocks along the rows (scales
// at sf_offset(row, col / 32, rows_total / 128) of sf_rows).  With a gather the rows come from a
// token-major source (padding rows read as zeros).
//
// Each warp is its own pipeline over tiles of 32 rows x 128 columns (8 KB of bf16):
// lane r brings row r of a tile into shared memory by one bulk asynchronous copy,
// QC_STAGES tiles ahead, rows QC_ROW bytes apart (a 16-byte skew per row, so that
// both a row read across the lanes and one row per lane hit distinct banks); the lane
// of a zero row (gather padding) writes its zeros there itself.  For the blocks down
// the columns lane l holds columns 4l .. 4l+3 of all 32 rows in registers; for the
// blocks along the rows (two-way) lane l takes row l.  Block maxima are absolute
// maxima of bf16 pairs (one instruction per pair; finite values), and a block's scale
// exponent comes straight from the exponent field of its maximum.
// W warps per CTA, one CTA per SM: twelve for reads from HBM; thirteen (which the
// rings just fit in shared memory) where the rows are gathered through L2, whose
// latency more warps hide better (the gathered passes 83 -> 76 us each on the
// 16k-token workload; the weights' two-way passes ran slower with thirteen).
constexpr int QC_WARPS = 12;
constexpr int QC_WARPS_GATHER = 13;
constexpr int QC_STAGES = 2;
constexpr int QC_TC = 128;                     // columns per tile
constexpr int QC_ROW = QC_TC * 2 + 16;         // bytes between rows in shared memory
constexpr int QC_TILE_BYTES = 32 * QC_ROW;
constexpr int qc_smem(int warps) { return warps * QC_STAGES * QC_TILE_BYTES; }
constexpr uint64_t QC_WAIT_NS = 2000000000ull;

// Absolute maxima of two bf16 pairs, pair by pair (the result's sign bits are not
// meaningful: clear them before use).
__device__ __forceinline__ uint32_t amax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

template <int W>
__global__ void __launch_bounds__(32 * W, 1) mxq_cols_kernel(
    const uint16_t* __restrict__ in, uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
    uint8_t* __restrict__ codes_rows, uint8_t* __restrict__ sf_rows, int64_t rows,
    int64_t rows_total, int C, const int* __restrict__ meta, const RowGather gather,
    DevStatus* status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t qbuf[];
  __shared__ __align__(8) uint64_t bar[W][QC_STAGES];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  rows = rows_in_use(rows, meta);
  const int col_tiles = C / QC_TC;
  const int64_t n_tiles = (rows / 32) * col_tiles;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * W + warp;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * W;
  const int64_t my_n = gw < n_tiles ? (n_tiles - 1 - gw) / nw + 1 : 0;
  const int64_t mnb = C / 128, mnb_rows = rows_total / 128;
  uint8_t* ring = qbuf + warp * (QC_STAGES * QC_TILE_BYTES);
  uint64_t* wbar = bar[warp];
  if (lane == 0) {
    for (int s = 0; s < QC_STAGES; ++s) ptx::mbar_init(&wbar[s], 1);
    ptx::fence_barrier_init();
  }
  __syncwarp();

  // bring tile i of this warp into its stage: lane r copies row r, or writes a zero
  // row (read by the other lanes after the warp synchronisations between this issue
  // and the tile's turn)
  auto issue = [&](int64_t i) {
    const int64_t t = gw + i * nw;
    const int64_t rb = t / col_tiles;
    const int c0 = static_cast<int>(t - rb * col_tiles) * QC_TC;
    const int src = gather_src(rb * 32 + lane, gather);
    const uint32_t valid = __ballot_sync(0xffffffffu, src >= 0);
    const int s = static_cast<int>(i % QC_STAGES);
    uint8_t* dst = ring + s * QC_TILE_BYTES + lane * QC_ROW;
    if (lane == 0)
      ptx::mbar_arrive_expect_tx(&wbar[s], static_cast<uint32_t>(__popc(valid)) * QC_TC * 2);
    if (src >= 0) {
      ptx::bulk_load(dst, in + static_cast<int64_t>(src) * C + c0, QC_TC * 2, &wbar[s]);
    } else {
#pragma unroll
      for (int j = 0; j < QC_TC * 2 / 16; ++j)
        reinterpret_cast<uint4*>(dst)[j] = make_uint4(0, 0, 0, 0);
    }
  };
  for (int64_t i = 0; i < QC_STAGES && i < my_n; ++i) issue(i);
  __syncwarp();  // (later issues are followed by the loop's own synchronisations)

  int no_abort = 0;
  for (int64_t i = 0; i < my_n; ++i) {
    const int s = static_cast<int>(i % QC_STAGES);
    const uint32_t parity = static_cast<uint32_t>((i / QC_STAGES) & 1);
    int ok = 1;
    if (lane == 0) ok = ptx::mbar_wait(&wbar[s], parity, &no_abort, QC_WAIT_NS) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {  // a copy never landed: report, let the other issued copies land, stop
      if (lane == 0) {
        if (status != nullptr && atomicCAS(&status->code, 0, MM_MOE_ETIMEOUT) == 0)
          status->detail = -2;
        for (int64_t j = i + 1; j < i + QC_STAGES && j < my_n; ++j)
          ptx::mbar_wait(&wbar[j % QC_STAGES], static_cast<uint32_t>((j / QC_STAGES) & 1),
                         &no_abort, QC_WAIT_NS);
      }
      __syncwarp();
      return;
    }
    // every lane observes the completed phase (returns at once): the bytes are visible
    if (lane != 0) ptx::mbar_wait(&wbar[s], parity, &no_abort, QC_WAIT_NS);
    const int64_t t = gw + i * nw;
    const int64_t rb = t / col_tiles;
    const int c0 = static_cast<int>(t - rb * col_tiles) * QC_TC;
    const int col = c0 + 4 * lane;
    const uint8_t* tile = ring + s * QC_TILE_BYTES;
    uint2 w[32];  // this lane's four columns of the tile's rows
    uint32_t m01 = 0, m23 = 0;  // column absolute maxima as bf16 pairs
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      w[r] = *reinterpret_cast<const uint2*>(tile + r * QC_ROW + 8 * lane);
      m01 = amax2(m01, w[r].x);
      m23 = amax2(m23, w[r].y);
    }
    m01 &= 0x7FFF7FFFu;
    m23 &= 0x7FFF7FFFu;
    if (codes_rows != nullptr) {
      // blocks along the rows: lane l quantises row l's four 32-column blocks
      const int64_t row = rb * 32 + lane;
      const uint4* rp = reinterpret_cast<const uint4*>(tile + lane * QC_ROW);
      uint32_t word = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        uint4 q[4];
        uint32_t m = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          q[j] = rp[4 * b + j];
          m = amax2(m, amax2(amax2(q[j].x, q[j].y), amax2(q[j].z, q[j].w)));
        }
        m &= 0x7FFF7FFFu;
        const int re = bf16_scale_exp(max(m & 0xFFFFu, m >> 16));
        const float sr = mx::pow2f(-re);
        uint32_t cw[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          cw[2 * j] = codes4(q[j].x, q[j].y, sr, sr, sr, sr);
          cw[2 * j + 1] = codes4(q[j].z, q[j].w, sr, sr, sr, sr);
        }
        uint4* dst = reinterpret_cast<uint4*>(codes_rows + row * C + c0 + 32 * b);
        dst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
        dst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
        word |= e8m0(re) << (8 * b);
      }
      *reinterpret_cast<uint32_t*>(sf_rows + sf_offset(row, c0 / 32, mnb_rows)) = word;
    }
    const int e0 = bf16_scale_exp(m01 & 0xFFFFu), e1 = bf16_scale_exp(m01 >> 16);
    const int e2 = bf16_scale_exp(m23 & 0xFFFFu), e3 = bf16_scale_exp(m23 >> 16);
    const float s0 = mx::pow2f(-e0), s1 = mx::pow2f(-e1), s2 = mx::pow2f(-e2),
                s3 = mx::pow2f(-e3);
    // the stage is refilled by the asynchronous proxy after these generic reads
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (i + QC_STAGES < my_n) issue(i + QC_STAGES);
#pragma unroll
    for (int r = 0; r < 32; ++r)
      *reinterpret_cast<uint32_t*>(codes + (rb * 32 + r) * C + col) =
          codes4(w[r].x, w[r].y, s0, s1, s2, s3);
    sf[sf_offset(col, rb, mnb)] = static_cast<uint8_t>(e8m0(e0));
    sf[sf_offset(col + 1, rb, mnb)] = static_cast<uint8_t>(e8m0(e1));
    sf[sf_offset(col + 2, rb, mnb)] = static_cast<uint8_t>(e8m0(e2));
    sf[sf_offset(col + 3, rb, mnb)] = static_cast<uint8_t>(e8m0(e3));
  }
}

cudaError_t launch_mxq(const Ctx& c, const MxqArgs& a) {
  if (a.along_rows) {
    prof_begin(c, K_MXQ_ROWS);
    launch_k(c.stream, mxq_rows_kernel, dim3(c.num_sms * 8), dim3(256), 0,
        reinterpret_cast<const uint4*>(a.in), reinterpret_cast<uint2*>(a.codes), a.sf, a.rows,
        static_cast<int>(a.cols / 8), a.rows / 128, a.meta);
    prof_end(c, K_MXQ_ROWS);
  } else {
    // one CTA (W warp pipelines) per SM; with `meta` the row count is known only on
    // the device, so the grid is sized for the capacity and surplus warps exit
    auto go = [&](auto kern, int w) {
      const int smem = qc_smem(w);
      cudaError_t e =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      const int64_t tiles = (a.rows / 32) * (a.cols / QC_TC);
      const int64_t want = (tiles + w - 1) / w;
      const int64_t grid = want < c.num_sms ? want : c.num_sms;
      prof_begin(c, K_MXQ_COLS);
      launch_k(c.stream, kern, dim3(static_cast<int>(grid > 0 ? grid : 1)), dim3(32 * w), smem,
               a.in, a.codes, a.sf, a.codes_rows, a.sf_rows, a.rows, a.rows,
               static_cast<int>(a.cols), a.meta, a.gather, a.status);
      prof_end(c, K_MXQ_COLS);
      return cudaSuccess;
    };
    cudaError_t e = a.gather.rowflat != nullptr
                        ? go(mxq_cols_kernel<QC_WARPS_GATHER>, QC_WARPS_GATHER)
                        : go(mxq_cols_kernel<QC_WARPS>, QC_WARPS);
    if (e != cudaSuccess) return e;
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

// route.cu -- token routing (expert histogram, prefix scan, stable placement), the
// row permutation into the expert-grouped layout, and the fixed-order gathers and
// sums back to token order (forward combine, backward un-permute).
//
// Prime Mega MoE pages, "Why is MoE training communication-bound?": before the
// expert math the GPU sorts tokens by destination expert; results come back per
// token afterwards.  On one GPU "sending" becomes a permutation of rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "fp8block.cuh"
#include "internal.h"
#include "mx.cuh"
#include "ptx.cuh"

namespace mmmoe {

__device__ __forceinline__ void set_status(DevStatus* st, int code, int detail) {
  if (atomicCAS(&st->code, 0, code) == 0) st->detail = detail;
}

// ---------------------------------------------------------------- 1. histogram
// One block per ROUTE_CHUNK flat indices: per-block expert counts.
__global__ void __launch_bounds__(ROUTE_THREADS) route_count_kernel(
    const int32_t* __restrict__ topk_idx, int R, int E, int* __restrict__ blk_counts,
    DevStatus* status) {
  pdl_wait();
  pdl_trigger();
  __shared__ int hist[MAX_E];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int base = blockIdx.x * ROUTE_CHUNK;
  for (int i0 = 0; i0 < ROUTE_CHUNK; i0 += blockDim.x) {
    const int f = base + i0 + threadIdx.x;
    int e = -1;
    if (f < R) {
      e = __ldg(topk_idx + f);
      if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
        set_status(status, MM_MOE_EBADIDX, f);
        e = -1;  // the pair is dropped
      }
    }
    // warp-aggregated: one shared-memory add per distinct expert in the warp
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[e], __popc(peers));
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    blk_counts[static_cast<int64_t>(blockIdx.x) * E + e] = hist[e];
}

// ---------------------------------------------------------------- 2. scan (one block)
// counts, offsets (exclusive scan), padded offsets, per-block exclusive prefixes
// (in place in blk_counts), the M-tile list and the experts ordered by row count.
__global__ void __launch_bounds__(1024) route_scan_kernel(
    int* __restrict__ blk_counts, int nblk, int E, int pad, int* __restrict__ counts,
    int* __restrict__ offsets, int* __restrict__ pad_off, int* __restrict__ expert_order,
    int* __restrict__ tile_expert, int* __restrict__ tile_rows, int* __restrict__ meta) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_cnt[MAX_E];
  __shared__ int s_a[MAX_E];
  __shared__ int s_b[MAX_E];
  const int e = threadIdx.x;
  int cnt = 0;
  if (e < E) {
    // SCAN_BATCH independent loads in flight, then their running sums
    constexpr int SCAN_BATCH = 16;
    int b = 0;
    for (; b + SCAN_BATCH <= nblk; b += SCAN_BATCH) {
      int c[SCAN_BATCH];
#pragma unroll
      for (int j = 0; j < SCAN_BATCH; ++j) c[j] = blk_counts[static_cast<int64_t>(b + j) * E + e];
#pragma unroll
      for (int j = 0; j < SCAN_BATCH; ++j) {
        blk_counts[static_cast<int64_t>(b + j) * E + e] = cnt;
        cnt += c[j];
      }
    }
    for (; b < nblk; ++b) {
      const int64_t i = static_cast<int64_t>(b) * E + e;
      const int c = blk_counts[i];
      blk_counts[i] = cnt;
      cnt += c;
    }
  }
  const int padded = (cnt + pad - 1) / pad * pad;
  if (e < MAX_E) {
    s_cnt[e] = (e < E) ? cnt : 0;
    s_a[e] = (e < E) ? cnt : 0;
    s_b[e] = (e < E) ? padded : 0;
  }
  __syncthreads();
  // inclusive Hillis-Steele scans over the experts
  for (int d = 1; d < MAX_E; d <<= 1) {
    int va = 0, vb = 0;
    if (e < MAX_E && e >= d) {
      va = s_a[e - d];
      vb = s_b[e - d];
    }
    __syncthreads();
    if (e < MAX_E && e >= d) {
      s_a[e] += va;
      s_b[e] += vb;
    }
    __syncthreads();
  }
  if (e < E) {
    const int off = s_a[e] - cnt;
    const int poff = s_b[e] - padded;
    counts[e] = cnt;
    offsets[e] = off;
    pad_off[e] = poff;
    const int nt = padded / BM;
    for (int i = 0; i < nt; ++i) {
      tile_expert[poff / BM + i] = e;
      tile_rows[poff / BM + i] = max(0, min(BM, cnt - i * BM));  // 0: all padding
    }
    // rank by descending row count, ties by expert index
    int rank = 0;
    for (int o = 0; o < E; ++o) {
      const int c = s_cnt[o];
      rank += (c > cnt) || (c == cnt && o < e);
    }
    expert_order[rank] = e;
  }
  if (e == E - 1) {
    offsets[E] = s_a[e];
    pad_off[E] = s_b[e];
    meta[META_NUM_TILES] = s_b[e] / BM;
  }
}

// ---------------------------------------------------------------- 3. stable placement
// Each warp walks its 256 consecutive flat indices in order, 32 at a time; the
// rank of an index among the earlier ones of the same expert is the warp's running
// count plus the number of lower lanes with the same expert (__match_any_sync).
// Block-level prefixes over warps and the scan's per-block prefixes complete the
// stable position.  No atomics decide a position.
__global__ void __launch_bounds__(ROUTE_THREADS) route_place_kernel(
    const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w, int R, int E,
    const int* __restrict__ blk_prefix, const int* __restrict__ offsets,
    const int* __restrict__ pad_off, int* __restrict__ perm, int* __restrict__ inv,
    int* __restrict__ prow, int* __restrict__ rowflat, float* __restrict__ w_row) {
  pdl_wait();
  pdl_trigger();
  constexpr int WARPS = ROUTE_THREADS / 32;
  constexpr int PER_WARP = ROUTE_CHUNK / WARPS;  // 256
  constexpr int ROUNDS = PER_WARP / 32;          // 8
  __shared__ int wrun[WARPS][MAX_E];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < WARPS * MAX_E; i += blockDim.x) (&wrun[0][0])[i] = 0;
  __syncthreads();
  const int base = blockIdx.x * ROUTE_CHUNK + warp * PER_WARP;
  int my_e[ROUNDS], my_rank[ROUNDS];
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    const int f = base + r * 32 + lane;
    int e = -1;
    if (f < R) {
      e = __ldg(topk_idx + f);
      if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) e = -1;  // dropped
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    int rank = 0;
    if (e >= 0) rank = wrun[warp][e] + __popc(peers & lt);
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) wrun[warp][e] += __popc(peers);
    __syncwarp();
    my_e[r] = e;
    my_rank[r] = rank;
  }
  __syncthreads();
  // exclusive prefix over warps, per expert (in place)
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < WARPS; ++w) {
      const int c = wrun[w][e];
      wrun[w][e] = run;
      run += c;
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    const int e = my_e[r];
    const int f = base + r * 32 + lane;
    if (e < 0) {
      if (f < R) {  // a dropped pair: the reductions skip it
        inv[f] = -1;
        prow[f] = -1;
      }
      continue;
    }
    const int local = blk_prefix[static_cast<int64_t>(blockIdx.x) * E + e] + wrun[warp][e] + my_rank[r];
    const int row = offsets[e] + local;
    const int prw = pad_off[e] + local;
    perm[row] = f;
    inv[f] = row;
    prow[f] = prw;
    rowflat[prw] = f;
    w_row[prw] = __ldg(topk_w + f);
  }
}

cudaError_t launch_route(const Ctx& c, const Layout& L, const int32_t* topk_idx,
                         const float* topk_w, char* saved, char* scratch) {
  const int R = static_cast<int>(L.R), E = static_cast<int>(L.E);
  const int nblk = static_cast<int>(L.nblk);
  DevStatus* st = reinterpret_cast<DevStatus*>(scratch + L.status);
  int* blk = reinterpret_cast<int*>(scratch + L.blk_counts);
  prof_begin(c, K_ROUTE_COUNT);
  launch_k(c.stream, route_count_kernel, dim3(nblk), dim3(ROUTE_THREADS), 0, topk_idx, R, E, blk, st);
  prof_end(c, K_ROUTE_COUNT);
  prof_begin(c, K_ROUTE_SCAN);
  launch_k(c.stream, route_scan_kernel, dim3(1), dim3(1024), 0,
      blk, nblk, E, static_cast<int>(L.pad), reinterpret_cast<int*>(saved + L.counts),
      reinterpret_cast<int*>(saved + L.offsets), reinterpret_cast<int*>(saved + L.pad_off),
      reinterpret_cast<int*>(saved + L.expert_order), reinterpret_cast<int*>(saved + L.tile_expert),
      reinterpret_cast<int*>(saved + L.tile_rows), reinterpret_cast<int*>(saved + L.meta));
  prof_end(c, K_ROUTE_SCAN);
  prof_begin(c, K_ROUTE_PLACE);
  launch_k(c.stream, route_place_kernel, dim3(nblk), dim3(ROUTE_THREADS), 0,
      topk_idx, topk_w, R, E, blk, reinterpret_cast<const int*>(saved + L.offsets),
      reinterpret_cast<const int*>(saved + L.pad_off), reinterpret_cast<int*>(saved + L.perm),
      reinterpret_cast<int*>(saved + L.inv), reinterpret_cast<int*>(saved + L.prow),
      reinterpret_cast<int*>(saved + L.rowflat), reinterpret_cast<float*>(saved + L.w_row));
  prof_end(c, K_ROUTE_PLACE);
  return cudaGetLastError();
}

// The same three routing kernels with every buffer given explicitly.
cudaError_t launch_route_to(const Ctx& c, int R, int E, int pad, const int32_t* topk_idx,
                            const float* topk_w, const RouteBufs& b) {
  const int nblk = (R + ROUTE_CHUNK - 1) / ROUTE_CHUNK;
  prof_begin(c, K_ROUTE_COUNT);
  launch_k(c.stream, route_count_kernel, dim3(nblk), dim3(ROUTE_THREADS), 0, topk_idx, R, E, b.blk_counts,
                                                           b.status);
  prof_end(c, K_ROUTE_COUNT);
  prof_begin(c, K_ROUTE_SCAN);
  launch_k(c.stream, route_scan_kernel, dim3(1), dim3(1024), 0, b.blk_counts, nblk, E, pad, b.counts, b.offsets,
                                              b.pad_off, b.expert_order, b.tile_expert,
                                              b.tile_rows, b.meta);
  prof_end(c, K_ROUTE_SCAN);
  prof_begin(c, K_ROUTE_PLACE);
  launch_k(c.stream, route_place_kernel, dim3(nblk), dim3(ROUTE_THREADS), 0,
      topk_idx, topk_w, R, E, b.blk_counts, b.offsets, b.pad_off, b.perm, b.inv, b.prow,
      b.rowflat, b.w_row);
  prof_end(c, K_ROUTE_PLACE);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- 4. permute
// dst[prow[t*k + j]] = src[t] for every routed pair, and zero padding rows.  Tokens
// are walked in order so that each source row is read from HBM once and stored to
// its k destinations.  Whole rows move by TMA bulk copies: lane 0 of each CTA drives
// a ring of PERM_SLOTS row buffers, loading PERM_AHEAD tokens ahead of the one it
// stores.  Padding rows are then stored from a zero row; in the forward their
// routing weight is zeroed too (valid rows got theirs from the placement kernel).
// QM = QS_MX / QS_BLOCK: the warp turns each row into its MXFP8 / blockwise FP8 form
// in shared memory between its load and its stores (e4m3 codes, H bytes, stored to the
// k destination rows of a [Rp, H] byte tensor; the H / 32 scale codes -- for blockwise
// FP8 each 128-element block's scale four times -- written as words of the scale
// arrangement mx::sf_offset over the padded rows).  A zero row quantises to zero codes
// and zero scale codes.
constexpr int PERM_SLOTS = 8;
constexpr int PERM_AHEAD = 6;
constexpr uint64_t PERM_WAIT_NS = 2000000000ull;

// Blockwise FP8 form of one bf16 row of n elements in shared memory (all 32 lanes):
// the n e4m3 codes over the start of the same buffer, each 128-element block's scale
// as a word of four equal E8M0 codes to `scales` (n / 128 words).  Two neighbouring
// lanes take one block per round (64 elements each, the maximum met by a shuffle) and
// hold their halves in registers, so that no lane writes codes before every lane has
// read its half.
__device__ __forceinline__ void quantise_row_fb(uint8_t* row, uint8_t* scales, int n, int lane) {
  const int nh = n / 64;  // half blocks (even: n % 128 == 0)
  for (int h0 = 0; h0 < nh; h0 += 32) {
    const int hb = h0 + lane;  // (lane ^ 1 takes the other half of the same block)
    const bool act = hb < nh;
    uint4 w[8];
    float m = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      w[q] = act ? reinterpret_cast<const uint4*>(row + hb * 128)[q] : make_uint4(0, 0, 0, 0);
      const uint16_t* h = reinterpret_cast<const uint16_t*>(&w[q]);
#pragma unroll
      for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(mx::bf(h[j])));
    }
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    __syncwarp();
    if (act) {
      const int e = fb::ceil_exp(m);
      const float mul = mx::pow2f(-e);
      uint4* d4 = reinterpret_cast<uint4*>(row + hb * 64);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        d4[q] = make_uint4(mx::codes4(w[2 * q].x, w[2 * q].y, mul, mul, mul, mul),
                           mx::codes4(w[2 * q].z, w[2 * q].w, mul, mul, mul, mul),
                           mx::codes4(w[2 * q + 1].x, w[2 * q + 1].y, mul, mul, mul, mul),
                           mx::codes4(w[2 * q + 1].z, w[2 * q + 1].w, mul, mul, mul, mul));
      if ((hb & 1) == 0) reinterpret_cast<uint32_t*>(scales)[hb / 2] = mx::e8m0(e) * 0x01010101u;
    }
    __syncwarp();
  }
}

// MXFP8 form of one bf16 row of n elements in shared memory (all 32 lanes): the n
// e4m3 codes over the start of the same buffer, the n / 32 scale codes to `scales`.
// A lane takes one 32-element block per round; every lane reads its round's block
// before any lane writes codes (which land on bytes of this round's or earlier
// rounds' blocks only).
__device__ __forceinline__ void quantise_row_mx(uint8_t* row, uint8_t* scales, int n, int lane) {
  const int nb = n / 32;
  for (int b0 = 0; b0 < nb; b0 += 32) {
    const int b = b0 + lane;
    float v[32];
    if (b < nb) {
      const uint4* r4 = reinterpret_cast<const uint4*>(row + b * 64);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 w = r4[q];
        const uint16_t* h = reinterpret_cast<const uint16_t*>(&w);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[8 * q + j] = mx::bf(h[j]);
      }
    }
    __syncwarp();
    if (b < nb) {
      uint2 c[4];
      const int e = mx::quant_row32(v, c);
      uint4* d4 = reinterpret_cast<uint4*>(row + b * 32);
      d4[0] = make_uint4(c[0].x, c[0].y, c[1].x, c[1].y);
      d4[1] = make_uint4(c[2].x, c[2].y, c[3].x, c[3].y);
      scales[b] = static_cast<uint8_t>(mx::e8m0(e));
    }
    __syncwarp();
  }
}

template <int QM>
__global__ void __launch_bounds__(32) permute_rows_kernel(
    const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int row_bytes, int T, int k,
    const int* __restrict__ meta, const int* __restrict__ tile_rows,
    const int* __restrict__ prow, float* __restrict__ w_row, DevStatus* status,
    uint8_t* __restrict__ sf, int64_t sf_mnb) {
  pdl_wait();
  pdl_trigger();
  // PERM_SLOTS rows, a zero row, then (FP8) PERM_SLOTS rows of scale codes
  extern __shared__ __align__(128) uint8_t pbuf[];
  __shared__ __align__(8) uint64_t bar[PERM_SLOTS];
  const int lane = threadIdx.x;
  uint8_t* zero = pbuf + PERM_SLOTS * row_bytes;
  const int n_el = row_bytes / 2;                            // elements of a row
  const int out_bytes = QM != QS_NONE ? n_el : row_bytes;    // bytes stored per row
  uint8_t* sbuf = zero + row_bytes;                          // FP8 scale codes
  const int n_words = n_el / 128;                            // FP8 scale words per row
  for (int i = lane * 16; i < row_bytes; i += 32 * 16)
    *reinterpret_cast<uint4*>(zero + i) = make_uint4(0, 0, 0, 0);
  ptx::fence_proxy_async_smem();  // the zero row is read by bulk stores
  if (lane == 0) {
    for (int s = 0; s < PERM_SLOTS; ++s) ptx::mbar_init(&bar[s], 1);
    ptx::fence_barrier_init();
  }
  __syncwarp();
  if (QM == QS_NONE && lane != 0) return;
  const int first = static_cast<int>(blockIdx.x), step = static_cast<int>(gridDim.x);
  // --- routed rows, token by token
  const int n_my = T > first ? (T - 1 - first) / step + 1 : 0;
  auto issue = [&](int i) {  // load my i-th token's row into slot i % PERM_SLOTS
    const int s = i % PERM_SLOTS;
    const int64_t t = first + static_cast<int64_t>(i) * step;
    ptx::mbar_arrive_expect_tx(&bar[s], static_cast<uint32_t>(row_bytes));
    ptx::bulk_load(pbuf + s * row_bytes, src + t * row_bytes, row_bytes, &bar[s]);
  };
  if (lane == 0)
    for (int i = 0; i < PERM_AHEAD && i < n_my; ++i) issue(i);
  int dummy = 0;
  for (int i = 0; i < n_my; ++i) {
    if (lane == 0 && i + PERM_AHEAD < n_my) {
      // the slot of token i + PERM_AHEAD last held token i + PERM_AHEAD - PERM_SLOTS,
      // whose stores (one group, PERM_SLOTS - PERM_AHEAD groups ago) must have read it
      ptx::bulk_wait_read<PERM_SLOTS - PERM_AHEAD - 1>();
      issue(i + PERM_AHEAD);
    }
    const int s = i % PERM_SLOTS;
    const uint32_t parity = static_cast<uint32_t>((i / PERM_SLOTS) & 1);
    int ok = 1;
    if (lane == 0) ok = ptx::mbar_wait(&bar[s], parity, &dummy, PERM_WAIT_NS) ? 1 : 0;
    if constexpr (QM != QS_NONE) ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) {
        if (atomicCAS(&status->code, 0, MM_MOE_ETIMEOUT) == 0) status->detail = -1;
        // the loads already issued land before the CTA exits (bounded as well)
        for (int j = i + 1; j < i + PERM_AHEAD + 1 && j < n_my; ++j)
          ptx::mbar_wait(&bar[j % PERM_SLOTS], static_cast<uint32_t>((j / PERM_SLOTS) & 1),
                         &dummy, PERM_WAIT_NS);
        ptx::bulk_wait_all();
      }
      return;
    }
    if constexpr (QM != QS_NONE) {
      // the other lanes observe the completed phase too (it returns at once), which
      // makes the row's bytes visible to them
      if (lane != 0) ptx::mbar_wait(&bar[s], parity, &dummy, PERM_WAIT_NS);
      if constexpr (QM == QS_MX)
        quantise_row_mx(pbuf + s * row_bytes, sbuf + s * (n_el / 32), n_el, lane);
      else
        quantise_row_fb(pbuf + s * row_bytes, sbuf + s * (n_el / 32), n_el, lane);
      ptx::fence_proxy_async_smem();  // the stores below read the quantised row
      __syncwarp();
    }
    const int64_t f0 = (first + static_cast<int64_t>(i) * step) * k;
    if (lane == 0) {
      for (int j = 0; j < k; ++j) {
        const int pr = __ldg(prow + f0 + j);
        if (pr >= 0)
          ptx::bulk_store(dst + static_cast<int64_t>(pr) * out_bytes, pbuf + s * row_bytes,
                          out_bytes);
      }
      ptx::bulk_commit();
    }
    if constexpr (QM != QS_NONE) {  // the row's scale words, to each of its k rows
      const uint32_t* words = reinterpret_cast<const uint32_t*>(sbuf + s * (n_el / 32));
      for (int j = 0; j < k; ++j) {
        const int pr = __ldg(prow + f0 + j);
        if (pr < 0) continue;
        for (int g = lane; g < n_words; g += 32)
          *reinterpret_cast<uint32_t*>(sf + mx::sf_offset(pr, 4 * g, sf_mnb)) = words[g];
      }
      __syncwarp();  // the slot's scale codes are rewritten PERM_SLOTS tokens later
    }
  }
  if (QM == QS_NONE && lane != 0) return;
  // --- padding rows of the M tiles (FP8: zero scale words too, by every lane)
  const int n_tiles = __ldg(meta + META_NUM_TILES);
  for (int mb = first; mb < n_tiles; mb += step) {
    for (int r = max(0, __ldg(tile_rows + mb)); r < BM; ++r) {
      const int64_t pr = static_cast<int64_t>(mb) * BM + r;
      if (lane == 0) {
        ptx::bulk_store(dst + pr * out_bytes, zero, out_bytes);
        if (w_row != nullptr) w_row[pr] = 0.f;
      }
      if constexpr (QM != QS_NONE)
        for (int g = lane; g < n_words; g += 32)
          *reinterpret_cast<uint32_t*>(sf + mx::sf_offset(pr, 4 * g, sf_mnb)) = 0u;
    }
  }
  if (lane == 0) {
    ptx::bulk_commit();
    ptx::bulk_wait_all();
  }
}

cudaError_t launch_permute(const Ctx& c, const Layout& L, const uint16_t* src, void* dst,
                           const char* saved, float* w_row_out, int kernel_id, char* scratch,
                           int quant, uint8_t* sf) {
  const int row_bytes = static_cast<int>(L.H * 2);
  const int smem = (PERM_SLOTS + 1) * row_bytes +
                   (quant != QS_NONE ? PERM_SLOTS * static_cast<int>(L.H / 32) : 0);
  auto* kern = quant == QS_MX      ? permute_rows_kernel<QS_MX>
               : quant == QS_BLOCK ? permute_rows_kernel<QS_BLOCK>
                                   : permute_rows_kernel<QS_NONE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int per_sm = std::max(1, std::min(16, (200 * 1024) / (smem + 1024)));
  prof_begin(c, kernel_id);
  launch_k(c.stream, kern, dim3(c.num_sms * per_sm), dim3(32), smem,
      reinterpret_cast<const uint8_t*>(src), reinterpret_cast<uint8_t*>(dst), row_bytes,
      static_cast<int>(L.T), static_cast<int>(L.k), reinterpret_cast<const int*>(saved + L.meta),
      reinterpret_cast<const int*>(saved + L.tile_rows),
      reinterpret_cast<const int*>(saved + L.prow), w_row_out,
      reinterpret_cast<DevStatus*>(scratch + L.status), sf, L.Rp / 128);
  prof_end(c, kernel_id);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- 5. reductions
__device__ __forceinline__ void acc_bf16x8(float (&acc)[8], const uint4 v) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(p[i]);
    acc[2 * i] += f.x;
    acc[2 * i + 1] += f.y;
  }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&acc)[8]) {
  uint4 v;
  __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
  return v;
}

// out[t] = sum_j rows[prow[t*k + j]] in fp32, j ascending (one warp per token): the
// k expert-grouped rows of a token, each H contiguous bf16.  With dtopk_w: also
// dtopk_w[t][j] = sum_n pw[prow[t*k+j]][n], n ascending.  Pairs dropped by the
// routing (prow < 0) contribute nothing.  KU > 0: k <= KU, and each lane issues the
// loads of all k rows of a 16-byte column before it sums them (in the same order).
template <int KU>
__global__ void __launch_bounds__(256) slot_reduce_kernel(
    const uint4* __restrict__ rows, uint4* __restrict__ out, int T, int k, int H8,
    const int* __restrict__ prow, const float* __restrict__ pw, int n_pw,
    float* __restrict__ dtopk_w) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
    const int64_t fb = static_cast<int64_t>(t) * k;
    const int my_row = lane < k ? __ldg(prow + fb + lane) : -1;
    uint4* o = out + static_cast<int64_t>(t) * H8;
    if constexpr (KU > 0) {
      int r[KU];
#pragma unroll
      for (int j = 0; j < KU; ++j) r[j] = __shfl_sync(0xffffffffu, my_row, j);  // -1 past k
      for (int i = lane; i < H8; i += 32) {
        uint4 v[KU];
#pragma unroll
        for (int j = 0; j < KU; ++j)
          if (r[j] >= 0) v[j] = __ldg(rows + static_cast<int64_t>(r[j]) * H8 + i);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < KU; ++j)
          if (r[j] >= 0) acc_bf16x8(acc, v[j]);
        o[i] = pack_bf16x8(acc);
      }
    } else {
      for (int i0 = 0; i0 < H8; i0 += 32) {
        const int i = i0 + lane;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < k; ++j) {
          const int r = k <= 32 ? __shfl_sync(0xffffffffu, my_row, j) : __ldg(prow + fb + j);
          if (r >= 0 && i < H8) acc_bf16x8(acc, __ldg(rows + static_cast<int64_t>(r) * H8 + i));
        }
        if (i < H8) o[i] = pack_bf16x8(acc);
      }
    }
    if (dtopk_w != nullptr) {
      for (int j = lane; j < k; j += 32) {
        const int r = __ldg(prow + fb + j);
        float acc = 0.f;
        if (r >= 0) {
          const float* p = pw + static_cast<int64_t>(r) * n_pw;
          for (int n = 0; n < n_pw; ++n) acc += p[n];
        }
        dtopk_w[fb + j] = acc;
      }
    }
  }
}

// k <= 8 (every workload here) takes the unrolled form
static void launch_slot_reduce(const Ctx& c, const uint4* rows, uint4* out, int T, int k, int H8,
                               const int* prow, const float* pw, int n_pw, float* dtopk_w) {
  if (k <= 8)
    launch_k(c.stream, slot_reduce_kernel<8>, dim3(c.num_sms * 8), dim3(256), 0, rows, out, T, k,
             H8, prow, pw, n_pw, dtopk_w);
  else
    launch_k(c.stream, slot_reduce_kernel<0>, dim3(c.num_sms * 8), dim3(256), 0, rows, out, T, k,
             H8, prow, pw, n_pw, dtopk_w);
}

cudaError_t launch_combine(const Ctx& c, const Layout& L, const uint16_t* slots,
                           const char* saved, uint16_t* out) {
  prof_begin(c, K_COMBINE);
  launch_slot_reduce(c, reinterpret_cast<const uint4*>(slots), reinterpret_cast<uint4*>(out),
                     static_cast<int>(L.T), static_cast<int>(L.k), static_cast<int>(L.H / 8),
                     reinterpret_cast<const int*>(saved + L.prow), nullptr, 0, nullptr);
  prof_end(c, K_COMBINE);
  return cudaGetLastError();
}

cudaError_t launch_unpermute(const Ctx& c, const Layout& L, const uint16_t* slots,
                             const char* saved, const float* pw, uint16_t* dx, float* dtopk_w) {
  prof_begin(c, K_UNPERMUTE);
  launch_slot_reduce(c, reinterpret_cast<const uint4*>(slots), reinterpret_cast<uint4*>(dx),
                     static_cast<int>(L.T), static_cast<int>(L.k), static_cast<int>(L.H / 8),
                     reinterpret_cast<const int*>(saved + L.prow), pw,
                     static_cast<int>(L.n_pw), dtopk_w);
  prof_end(c, K_UNPERMUTE);
  return cudaGetLastError();
}

}  // namespace mmmoe

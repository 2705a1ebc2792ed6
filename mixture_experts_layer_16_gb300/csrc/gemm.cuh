// gemm.cuh -- the expert GEMMs of the layer as one persistent, warp-specialised
// tcgen05 kernel template for sm_103a (TMA -> 128B-swizzled shared memory ring ->
// tcgen05.mma with fp32 accumulators in TMEM -> epilogue warps), instantiated for
// bf16 operands (kind::f16) in gemm.cu and for MXFP8 operands
// (kind::mxf8f6f4.block_scale) in gemm_fp8.cu.
//
// Prime Mega MoE pages, "How does the fused kernel work?": the two expert linear
// layers with SwiGLU between them and the combine in the forward, and the
// matching backward.  Seven kinds share the main loop:
//   GATEUP       [g|u] = x_perm . [W_gate;W_up]^T  per expert M block, SwiGLU epilogue
//   DOWN         o = a . W_down^T                   epilogue w*o (expert-grouped rows)
//   DGRAD_DOWN   g' = dy_perm . W_down               dSwiGLU epilogue (dh, w*a, <a,g'>)
//   DGRAD_GATEUP dx = dh . [W_gate;W_up]             epilogue dx (expert-grouped rows)
//   WGRAD_DOWN   dW_down[e] = dy_perm^T . (w*a)      K = the expert's rows
//   WGRAD_GATEUP [dW_gate;dW_up][e] = dh^T . x_perm   K = the expert's rows
//   WGRAD_BOTH   the two weight gradients in one launch: each expert's WGRAD_DOWN
//                tiles, then its WGRAD_GATEUP tiles, experts by descending row count
//                (one list evens out the clusters' loads: the per-kind lists leave
//                a tail of 9-17 % on skewed routing, the joint one about 3 %)
//
// CTAS = 2 runs each tile on an SM pair: the two CTAs of a 2-CTA cluster each stage
// 128 rows of A and half of the N columns of B, and one tcgen05.mma.cta_group::2 of
// M = 256 reads both halves.  CTAS = 1 runs 128-row tiles on single SMs (shapes the
// pair tiles do not divide, and the weight-gradient GEMMs of small experts).
//
// FP8 = true: the operands are MXFP8 -- e4m3 codes (1 byte per element, so a stage of
// 128-byte rows carries K = 128) and E8M0 scales per 32 elements along K in the atom
// arrangement of mx::sf_offset.  Each stage also brings one 512-byte scale atom per
// 128 MMA rows of A (this CTA's) and of B (all BN of the tile, in each CTA); the MMA
// thread copies them to TMEM (tcgen05.cp) and issues four kind::mxf8f6f4.block_scale
// MMAs of K = 32, k-block j reading byte j of each scale word.  TMEM then holds the
// scales beside the accumulators: BN = 256 tiles keep one accumulator (256 columns +
// scales fill the 512), narrower tiles two.  The gate/up epilogue of an FP8 forward
// also writes a in MXFP8 (codes and scales along I) for the down projection.
//
// MC (bf16 grouped GEMMs under MM_MOE_MULTICAST): clusters of two SM pairs share each
// M tile's A rows by TMA multicast (see the kernel).  Dense A^T.B may split its K over
// a cluster of CTAs whose partial tiles are summed through distributed shared memory.
//
// Roles (256 threads per CTA; 384 with the split epilogue's eight warps): warp 0 lane 0
// = TMA producer, warp 1 lane 0 of the pair's first CTA = MMA issuer, warp 2 = TMEM
// allocator, warps 4.. = epilogue (warp 4+q reads TMEM lanes 32q..32q+31, i.e. the
// CTA's tile rows 32q..32q+31).
// The epilogue moves data through per-warp 32 x 32 blocks in shared memory: outputs
// leave by TMA stores and the dSwiGLU inputs arrive by TMA loads.  Every wait is
// bounded: on expiry the kernel records MM_MOE_ETIMEOUT in the status word and every
// role unwinds.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "mx.cuh"
#include "ptx.cuh"

namespace mmmoe {
namespace gemm {

constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s

struct GemmParams {
  CUtensorMap tmA;
  CUtensorMap tmA_half;  // A-multicast launches: A with boxes of BM / 2 rows
  CUtensorMap tmB0;
  CUtensorMap tmB1;
  CUtensorMap tmC0;  // epilogue outputs stored by TMA (32 x 32 boxes, 64-byte swizzle)
  CUtensorMap tmC1;
  CUtensorMap tmD0;  // epilogue inputs loaded by TMA (dSwiGLU: h and a)
  CUtensorMap tmD1;
  CUtensorMap tmA2;  // WGRAD_BOTH: the dW_down part's operands and output
  CUtensorMap tmB2;
  CUtensorMap tmC2;
  // FP8: the scale tensors of A, B0, B1, A2, B2 (byte tensors seen as rows of 128
  // bytes; one box = one 512-byte atom) and their numbers of 128-row MN blocks
  CUtensorMap tmSA, tmSB0, tmSB1, tmSA2, tmSB2;
  int sfa_mnb, sfb_mnb, sfa2_mnb, sfb2_mnb;
  // FP8 gate/up: a in MXFP8 along I for the down projection (codes [Rp, I], scales
  // over q_mnb = Rp / 128 row blocks), or null
  uint8_t* q_codes;
  uint8_t* q_sf;
  int q_mnb;
  int H, I, E;
  int n_tiles;  // N tiles per M block (grouped kinds) or per expert M row (per-expert kinds)
  int m_tiles;  // M tiles (of BM * CTAS rows) per expert (per-expert kinds)
  int n_tiles2;  // WGRAD_BOTH: N and M tiles per expert of the dW_down part (n_tiles
  int m_tiles2;  // and m_tiles are then those of the dW_gate / dW_up part)
  int k_iters;  // K iterations per tile (grouped kinds)
  int n_pw;
  int max_tiles;
  int dm, dn;  // dense products: the output's rows and columns
  // A^T.B (GEMM_DENSE_TN): K split over clusters of ksplit CTAs (1: not split), kper K
  // iterations each; the partial tiles are summed through distributed shared memory
  int ksplit, kper;
  int stall;  // failure-path test: CTA 0 arms its first stage but issues no copy
  const int* meta;
  const int* tile_expert;
  const int* tile_rows;
  const int* pad_off;
  const int* counts;
  const int* expert_order;
  const int* rowflat;
  const float* w_row;
  uint16_t* out0;
  uint16_t* out1;
  float* outf;
  DevStatus* status;
};

template <int KIND, int BN_, int CTAS_, bool FP8_>
struct Cfg {
  static constexpr bool FP8 = FP8_;
  static constexpr int BN = BN_;      // N of one MMA (both CTAs of a pair together)
  static constexpr int CTAS = CTAS_;
  static constexpr bool DENSE = KIND >= GEMM_DENSE_NT;
  static constexpr bool PER_EXPERT = KIND >= GEMM_WGRAD_DOWN && !DENSE;
  static constexpr bool A_MN = PER_EXPERT || KIND == GEMM_DENSE_TN;
  static constexpr bool B_MN = (KIND >= GEMM_DGRAD_DOWN && !DENSE) || KIND == GEMM_DENSE_NN ||
                               KIND == GEMM_DENSE_TN;
  static constexpr int B_ROWS = BN / CTAS;  // B rows (K-major) or columns (M/N-major) per CTA
  // each stage holds 128 bytes of K per operand row: 64 bf16 or 128 e4m3 elements;
  // an M/N-major box spans 128 bytes of M/N (64 bf16 or 128 e4m3 elements)
  static constexpr int KSTEP = FP8 ? 128 : BK;
  static constexpr int MN_BOX = FP8 ? 128 : 64;
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = B_ROWS * 128;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // FP8: the stage's scale atoms (this CTA's 128 rows of A, then all BN rows of B)
  static constexpr int SF_BYTES = FP8 ? 512 * (1 + BN / 128) : 0;
  // accumulators in TMEM: FP8 tiles of BN = 256 leave room for one beside the scales
  static constexpr int NACC = (FP8 && BN == 256) ? 1 : 2;
  // epilogue staging per epilogue warp, in 2 KB blocks (32 rows x 32 bf16): TMA-loaded
  // inputs (dSwiGLU: g, u, a) and a ring of output blocks for TMA stores
  // SPLIT (the FP8 tiles with one accumulator): eight epilogue warps, two per TMEM
  // lane quadrant, each taking half of the tile's columns; they move their columns
  // to registers and hand TMEM back to the MMA issuer before most of their work
  // (EARLY_RELEASE), so the next tile's main loop overlaps the stores
  static constexpr bool SPLIT = NACC == 1;
  static constexpr bool EARLY_RELEASE = SPLIT;
  static constexpr int EPI_WARPS = SPLIT ? 8 : 4;
  static constexpr int THREADS = 128 + 32 * EPI_WARPS;
  static constexpr int EPI_IN = KIND == GEMM_DGRAD_DOWN ? 3 : KIND == GEMM_DENSE_NN ? BN / 32 : 0;
  // (SPLIT: one output block per warp, which leaves room for a sixth pipeline stage,
  // two in the dSwiGLU epilogue, where they fit beside its four stages; a warp's
  // next block waits for the store before last to have read it)
  static constexpr int EPI_OUT = SPLIT ? (KIND == GEMM_DGRAD_DOWN ? 2 : 1) : 4;
  static constexpr int EPI_WARP_BYTES = (EPI_IN + EPI_OUT) * 2048;
  static constexpr int EPI_BYTES = EPI_WARPS * EPI_WARP_BYTES;
  static constexpr int SMEM_CAP = 232448 - 1024;  // opt-in limit minus static shared memory
  static constexpr int STAGES_FIT = (SMEM_CAP - 1024 - EPI_BYTES) / (STAGE_BYTES + SF_BYTES);
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int SMEM_BYTES = STAGES * (STAGE_BYTES + SF_BYTES) + EPI_BYTES + 1024;
  static constexpr uint32_t TMEM_COLS = FP8 ? 512 : 2 * BN;
  // FP8: each pipeline stage has its own 16 TMEM columns for its scales (A's 4, then
  // B's 4 per 128 rows), so the copy of a stage's scales never waits for the MMAs of
  // the previous stage to finish reading theirs
  static constexpr uint32_t SF_COL0 = 256, SF_COLS_PER_STAGE = 16;
  // FP8 dSwiGLU epilogue on SPLIT tiles: TMEM columns past the scale ring where each
  // warp parks three of its four 32-column chunks of g' (96 columns per column half)
  static constexpr uint32_t STASH_COL0 = SF_COL0 + STAGES * SF_COLS_PER_STAGE;
  static constexpr uint32_t IDESC = FP8 ? ptx::idesc_mxf8(BM * CTAS, BN, A_MN, B_MN)
                                        : ptx::idesc_bf16_f32(BM * CTAS, BN, A_MN, B_MN);
  static_assert(BN == 64 || BN == 128 || BN == 256, "BN");
  static_assert(CTAS == 1 || (CTAS == 2 && B_ROWS >= 64), "CTAS");
  static_assert(!(KIND == GEMM_GATEUP && (CTAS == 2 || FP8) && BN != 256), "gate/up tile");
  static_assert(!FP8 || BN >= 128, "FP8 scale atoms cover 128 rows of B");
  static_assert(!DENSE || (CTAS == 1 && !FP8), "dense products: single-SM bf16 tiles");
  static_assert(!(FP8 && B_MN && B_ROWS % 128 != 0), "FP8 M/N-major boxes are 128 wide");
  static_assert(!FP8 || NACC * BN <= static_cast<int>(SF_COL0), "TMEM columns");
  static_assert(!FP8 || SF_COL0 + STAGES * SF_COLS_PER_STAGE <= TMEM_COLS, "TMEM scale ring");
  static_assert(!(SPLIT && KIND == GEMM_DGRAD_DOWN) || STASH_COL0 + 2 * 96 <= TMEM_COLS,
                "TMEM stash");
  static_assert(STAGES >= 2, "stages");
};

struct TileInfo {
  int e, mb, m0, n0, k_iters, k_row0;
  int down;  // per-expert kinds: 1 = a dW_down tile, 0 = a dW_gate / dW_up tile
};

// Per-expert tiles of kind KIND: (dW_down tiles, dW_gate / dW_up tiles) per expert.
template <int KIND>
__device__ __forceinline__ int2 expert_tiles(const GemmParams& p) {
  if constexpr (KIND == GEMM_WGRAD_DOWN) return make_int2(p.m_tiles * p.n_tiles, 0);
  else if constexpr (KIND == GEMM_WGRAD_GATEUP) return make_int2(0, p.m_tiles * p.n_tiles);
  else return make_int2(p.m_tiles2 * p.n_tiles2, p.m_tiles * p.n_tiles);
}

// Decode tile t for this CTA (rank within the pair).  Grouped kinds: t -> (group of
// CTAS 128-row blocks of padded routed rows, N tile), N fastest; the CTA takes block
// CTAS*group + rank.  Per-expert kinds: experts in descending row count, then (M, N)
// tiles of BM*CTAS x BN (an expert's dW_down tiles first); the CTA takes rows
// rank*BM.. of the M tile.
// MC (A multicast, grouped kinds on SM pairs): a cluster of two pairs takes N tiles
// 2j and 2j + 1 of one M tile, pair rank >> 1 the one of its parity, and `rank` is the
// CTA's rank in that four-CTA cluster (the CTA's place in its pair is rank & 1).
// Dense kinds: `ks` is the CTA's place in a split-K cluster (0 when K is not split);
// k_row0 is then the first K element of its share.
template <int KIND, int BN, int CTAS, bool FP8, bool MC = false>
__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, int t, int rank,
                                                int ks = 0) {
  using C = Cfg<KIND, BN, CTAS, FP8>;
  TileInfo ti;
  ti.down = 0;
  if constexpr (C::DENSE) {
    const int mt = t / p.n_tiles;
    ti.e = 0;
    ti.mb = mt;
    ti.m0 = mt * BM;
    ti.n0 = (t - mt * p.n_tiles) * BN;
    if (KIND == GEMM_DENSE_TN && p.ksplit > 1) {
      ti.k_iters = max(0, min(p.kper, p.k_iters - ks * p.kper));
      ti.k_row0 = ks * p.kper * C::KSTEP;
    } else {
      ti.k_iters = p.k_iters;
      ti.k_row0 = 0;
    }
  } else if constexpr (C::PER_EXPERT) {
    const int2 per = expert_tiles<KIND>(p);
    const int per_e = per.x + per.y;
    const int ei = t / per_e;
    int rem = t - ei * per_e;
    ti.down = rem < per.x ? 1 : 0;
    if (!ti.down) rem -= per.x;
    const int ntl = ti.down && KIND == GEMM_WGRAD_BOTH ? p.n_tiles2 : p.n_tiles;
    const int mt = rem / ntl;
    const int nt = rem - mt * ntl;
    ti.e = __ldg(p.expert_order + ei);
    ti.mb = 0;
    ti.m0 = mt * BM * CTAS + rank * BM;
    ti.n0 = nt * BN;
    ti.k_row0 = __ldg(p.pad_off + ti.e);
    // K stops at the last stage (64 rows bf16, 128 rows FP8) holding a routed row (the
    // rows after it, up to the padded end, are zero)
    ti.k_iters = (__ldg(p.counts + ti.e) + C::KSTEP - 1) / C::KSTEP;
  } else if constexpr (MC) {
    const int half = p.n_tiles >> 1;
    const int pmb = t / half;
    const int nt = 2 * (t - pmb * half) + (rank >> 1);
    ti.mb = pmb * CTAS + (rank & 1);
    ti.e = __ldg(p.tile_expert + ti.mb);
    ti.m0 = ti.mb * BM;
    ti.n0 = nt * (KIND == GEMM_GATEUP ? BN / 2 : BN);
    ti.k_iters = p.k_iters;
    ti.k_row0 = 0;
  } else {
    const int pmb = t / p.n_tiles;
    const int nt = t - pmb * p.n_tiles;
    ti.mb = pmb * CTAS + rank;
    ti.e = __ldg(p.tile_expert + ti.mb);
    ti.m0 = ti.mb * BM;
    ti.n0 = nt * (KIND == GEMM_GATEUP ? BN / 2 : BN);
    ti.k_iters = p.k_iters;
    ti.k_row0 = 0;
  }
  return ti;
}

template <int KIND, int BN, int CTAS, bool FP8, bool MC = false>
__device__ __forceinline__ int total_tiles(const GemmParams& p) {
  if constexpr (Cfg<KIND, BN, CTAS, FP8>::DENSE) {
    return p.m_tiles * p.n_tiles;
  } else if constexpr (Cfg<KIND, BN, CTAS, FP8>::PER_EXPERT) {
    const int2 per = expert_tiles<KIND>(p);
    return p.E * (per.x + per.y);
  } else {
    int nt = __ldg(p.meta + META_NUM_TILES);
    nt = min(nt, p.max_tiles);
    return (nt / CTAS) * (MC ? p.n_tiles >> 1 : p.n_tiles);
  }
}

// The abort flags of the other CTAs of a cluster (shared::cluster addresses): none on
// single SMs, the peer's on an SM pair, all three others in a two-pair cluster.
struct Peers {
  uint32_t a[3] = {0u, 0u, 0u};
  int n = 0;
};

// A wait ran out: this CTA's roles give up (*abort), and so do the other CTAs of its
// cluster (their abort flags set through `peers`), so that none waits out its own
// limits for work another will never do.
__device__ __forceinline__ void record_timeout(GemmParams const& p, volatile int* abort,
                                               int detail, const Peers& peers = Peers{}) {
  *abort = 1;
  for (int i = 0; i < peers.n; ++i) ptx::st_cluster_u32(peers.a[i], 1u);
  if (p.status != nullptr && atomicCAS(&p.status->code, 0, MM_MOE_ETIMEOUT) == 0)
    p.status->detail = detail;
}

// ------------------------------------------------------------------ epilogue helpers
// Each epilogue thread owns one accumulator row (TMEM lane); its 32-column chunks
// go through a per-warp 32 x 32 bf16 block in shared memory laid out with the
// 64-byte swizzle (16-byte chunk j of row r at r*64 + ((j ^ ((r >> 1) & 3)) * 16)),
// conflict-free for the row-per-thread accesses and the layout the TMA engine uses.
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint8_t* swz(uint8_t* buf, int r, int j) {
  return buf + r * 64 + ((j ^ ((r >> 1) & 3)) << 4);
}

__device__ __forceinline__ void stage32(uint8_t* buf, int r, const float (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(swz(buf, r, j)) =
        make_uint4(pack2(v[8 * j], v[8 * j + 1]), pack2(v[8 * j + 2], v[8 * j + 3]),
                   pack2(v[8 * j + 4], v[8 * j + 5]), pack2(v[8 * j + 6], v[8 * j + 7]));
}

__device__ __forceinline__ void unstage32(uint8_t* buf, int r, float (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 w = *reinterpret_cast<const uint4*>(swz(buf, r, j));
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[8 * j + 2 * i] = __uint_as_float(ww[i] << 16);
      v[8 * j + 2 * i + 1] = __uint_as_float(ww[i] & 0xFFFF0000u);
    }
  }
}

__device__ __forceinline__ void as_float(const uint32_t (&r)[32], float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ float sigmoidf_(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }

// Per-warp epilogue state.
struct EpiWarp {
  uint8_t* in;        // input blocks (dSwiGLU)
  uint8_t* out;       // output ring
  uint64_t* ld_bar;   // input-load barrier of this warp
  uint32_t ld_phase;
  bool ld_pending;
  int ob;             // next ring slot
  int lane;
};

// Store this warp's 32 x 32 block (row r = lane) at element coordinates (c0, c1) of
// tensor map m through the next slot of a ring of NB blocks.
template <int NB>
__device__ __forceinline__ void store_block(EpiWarp& w, const CUtensorMap* m, int c0, int c1,
                                            const float (&v)[32]) {
  uint8_t* buf = w.out + w.ob * 2048;
  if (w.lane == 0) ptx::bulk_wait_read<NB - 1>();  // the slot's previous store has read it
  __syncwarp();
  stage32(buf, w.lane, v);
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (w.lane == 0) {
    ptx::tma_store_2d(m, buf, c0, c1);
    ptx::bulk_commit();
  }
  w.ob = (w.ob + 1 == NB) ? 0 : w.ob + 1;
}

// The next slot of a warp's ring of NB output blocks, once the store that last used
// it has read it; end_block sends the block to coordinates (c0, c1) of tensor map m.
template <int NB>
__device__ __forceinline__ uint8_t* begin_block(EpiWarp& w) {
  uint8_t* buf = w.out + w.ob * 2048;
  if (w.lane == 0) ptx::bulk_wait_read<NB - 1>();
  __syncwarp();
  return buf;
}
template <int NB>
__device__ __forceinline__ void end_block(EpiWarp& w, const CUtensorMap* m, int c0, int c1,
                                          uint8_t* buf) {
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (w.lane == 0) {
    ptx::tma_store_2d(m, buf, c0, c1);
    ptx::bulk_commit();
  }
  w.ob = (w.ob + 1 == NB) ? 0 : w.ob + 1;
}

// Packed bf16 pairs: 32 values in 16 words.
__device__ __forceinline__ void pack32(const float (&v)[32], uint32_t (&pk)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) pk[i] = pack2(v[2 * i], v[2 * i + 1]);
}
__device__ __forceinline__ void unpack32(const uint32_t (&pk)[16], float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[2 * i] = __uint_as_float(pk[i] << 16);
    v[2 * i + 1] = __uint_as_float(pk[i] & 0xFFFF0000u);
  }
}

// store_block for values already packed to bf16.
template <int NB>
__device__ __forceinline__ void store_block_p(EpiWarp& w, const CUtensorMap* m, int c0, int c1,
                                              const uint32_t (&pk)[16]) {
  uint8_t* buf = w.out + w.ob * 2048;
  if (w.lane == 0) ptx::bulk_wait_read<NB - 1>();
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(swz(buf, w.lane, j)) =
        make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (w.lane == 0) {
    ptx::tma_store_2d(m, buf, c0, c1);
    ptx::bulk_commit();
  }
  w.ob = (w.ob + 1 == NB) ? 0 : w.ob + 1;
}

// dSwiGLU inputs of one 32-column chunk: g, u (from h) and a, rows row0..row0+31.
__device__ __forceinline__ void load_inputs(EpiWarp& w, const GemmParams& p, int row0, int col) {
  if (w.lane == 0) {
    ptx::fence_proxy_async_smem();
    ptx::mbar_arrive_expect_tx(w.ld_bar, 3 * 2048);
    ptx::tma_load_2d(w.in, &p.tmD0, w.ld_bar, col, row0);
    ptx::tma_load_2d(w.in + 2048, &p.tmD0, w.ld_bar, p.I + col, row0);
    ptx::tma_load_2d(w.in + 4096, &p.tmD1, w.ld_bar, col, row0);
  }
  w.ld_pending = true;
}

// C += A.B: the warp's BN / 32 blocks of C (rows row0..row0+31 from column n0) in one
// go, before the tile's accumulator is ready.
template <int BN>
__device__ __forceinline__ void load_c_blocks(EpiWarp& w, const GemmParams& p, int row0, int n0) {
  if (w.lane == 0) {
    ptx::fence_proxy_async_smem();
    ptx::mbar_arrive_expect_tx(w.ld_bar, BN / 32 * 2048);
#pragma unroll
    for (int j = 0; j < BN / 32; ++j)
      ptx::tma_load_2d(w.in + j * 2048, &p.tmD0, w.ld_bar, n0 + 32 * j, row0);
  }
  w.ld_pending = true;
}

__device__ __forceinline__ bool wait_inputs(EpiWarp& w, volatile int* abort) {
  int ok = 1;
  if (w.lane == 0) ok = ptx::mbar_wait(w.ld_bar, w.ld_phase, abort, WAIT_LIMIT_NS) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) {
    w.ld_phase ^= 1u;
    w.ld_pending = false;
  }
  return ok != 0;
}

// Epilogue of one tile for one warp (row = lane of the warp's 32 rows, q = warp).
// `next` is the tile this CTA processes after this one (dSwiGLU prefetch), or null.
template <int KIND, int BN, int CTAS, bool FP8>
__device__ __forceinline__ bool epilogue_tile(const GemmParams& p, const TileInfo& ti,
                                              const TileInfo* next, int q, uint32_t tbase,
                                              EpiWarp& w, volatile int* abort) {
  using C = Cfg<KIND, BN, CTAS, FP8>;
  const int lane = w.lane, row = q * 32 + lane;
  const int row0 = ti.m0 + q * 32;
  if constexpr (KIND == GEMM_GATEUP) {
    constexpr int HALF = BN / 2;
#pragma unroll 1
    for (int c = 0; c < HALF; c += 32) {
      uint32_t rg[32], ru[32];
      ptx::tmem_ld32(tbase + c, rg);
      ptx::tmem_ld32(tbase + HALF + c, ru);
      ptx::tmem_wait_ld(rg);
      ptx::reg_fence(ru);
      float g[32], u[32], a[32];
      as_float(rg, g);
      as_float(ru, u);
#pragma unroll
      for (int i = 0; i < 32; ++i) a[i] = g[i] * sigmoidf_(g[i]) * u[i];
      store_block<C::EPI_OUT>(w, &p.tmC0, ti.n0 + c, row0, g);
      store_block<C::EPI_OUT>(w, &p.tmC0, p.I + ti.n0 + c, row0, u);
      store_block<C::EPI_OUT>(w, &p.tmC1, ti.n0 + c, row0, a);
      if constexpr (FP8) {
        if (p.q_codes != nullptr) {  // the down projection's operand: a in MXFP8 along I
          uint2 cq[4];
          const int e = mx::quant_row32(a, cq);  // from a's stored (bf16) value
          const int64_t r = row0 + lane;
          uint4* dq = reinterpret_cast<uint4*>(p.q_codes + r * p.I + ti.n0 + c);
          dq[0] = make_uint4(cq[0].x, cq[0].y, cq[1].x, cq[1].y);
          dq[1] = make_uint4(cq[2].x, cq[2].y, cq[3].x, cq[3].y);
          p.q_sf[mx::sf_offset(r, (ti.n0 + c) / 32, p.q_mnb)] = static_cast<uint8_t>(mx::e8m0(e));
        }
      }
    }
  } else if constexpr (KIND == GEMM_DOWN || KIND == GEMM_DGRAD_GATEUP) {
    // rows stay in expert-grouped order; padding rows carry weight 0 (DOWN) or zero
    // inputs (DGRAD_GATEUP) and are never read back
    const float wgt = KIND == GEMM_DOWN ? __ldg(p.w_row + ti.m0 + row) : 1.0f;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t r[32];
      ptx::tmem_ld32(tbase + c, r);
      ptx::tmem_wait_ld(r);
      float v[32];
      as_float(r, v);
      if (KIND == GEMM_DOWN) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= wgt;
      }
      store_block<C::EPI_OUT>(w, &p.tmC0, ti.n0 + c, row0, v);
    }
  } else if constexpr (KIND == GEMM_DGRAD_DOWN) {
    const int64_t pr = ti.m0 + row;
    const float wgt = __ldg(p.w_row + pr);
    float dot = 0.f;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      if (!w.ld_pending) load_inputs(w, p, row0, ti.n0 + c);
      if (!wait_inputs(w, abort)) return false;
      float g[32], u[32], av[32];
      unstage32(w.in, lane, g);
      unstage32(w.in + 2048, lane, u);
      unstage32(w.in + 4096, lane, av);
      __syncwarp();
      if (c + 32 < BN) load_inputs(w, p, row0, ti.n0 + c + 32);
      else if (next != nullptr) load_inputs(w, p, next->m0 + q * 32, next->n0);
      uint32_t r[32];
      ptx::tmem_ld32(tbase + c, r);
      ptx::tmem_wait_ld(r);
      float dg[32], du[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float gp = __uint_as_float(r[i]);
        const float s = sigmoidf_(g[i]);
        const float sg = g[i] * s;               // silu(g)
        dot += av[i] * gp;                       // the forward's a (from fp32 g, u)
        const float da = wgt * gp;
        dg[i] = da * u[i] * s * (1.0f + g[i] * (1.0f - s));
        du[i] = da * sg;
        av[i] *= wgt;                            // w * a, the dW_down operand
      }
      store_block<C::EPI_OUT>(w, &p.tmC0, ti.n0 + c, row0, dg);
      store_block<C::EPI_OUT>(w, &p.tmC0, p.I + ti.n0 + c, row0, du);
      store_block<C::EPI_OUT>(w, &p.tmC1, ti.n0 + c, row0, av);
    }
    p.outf[pr * p.n_pw + ti.n0 / BN] = dot;
  } else if constexpr (KIND == GEMM_DENSE_NT) {
    // fp32 rows straight to global memory (rows / columns past the output skipped)
    const int r = ti.m0 + row;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t rr[32];
      ptx::tmem_ld32(tbase + c, rr);
      ptx::tmem_wait_ld(rr);
      const int col = ti.n0 + c;
      if (r < p.dm && col < p.dn) {
        float* dst = p.outf + static_cast<int64_t>(r) * p.dn + col;
        if (col + 32 <= p.dn) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            reinterpret_cast<float4*>(dst)[j] =
                make_float4(__uint_as_float(rr[4 * j]), __uint_as_float(rr[4 * j + 1]),
                            __uint_as_float(rr[4 * j + 2]), __uint_as_float(rr[4 * j + 3]));
        } else {
          for (int j = 0; j < p.dn - col; ++j) dst[j] = __uint_as_float(rr[j]);
        }
      }
    }
  } else if constexpr (KIND == GEMM_DENSE_NN) {
    // C += A.B: the warp's blocks of C came in by TMA ahead of the accumulator (the
    // next tile's are requested once these are read); each takes the sum in fp32 and
    // goes back rounded to bf16 (TMA clips the blocks at the output's edges)
    if (!w.ld_pending) load_c_blocks<BN>(w, p, row0, ti.n0);
    if (!wait_inputs(w, abort)) return false;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      float old[32];
      unstage32(w.in + (c / 32) * 2048, lane, old);
      if (c + 32 == BN) {
        __syncwarp();
        if (next != nullptr) load_c_blocks<BN>(w, p, next->m0 + q * 32, next->n0);
      }
      uint32_t rr[32];
      ptx::tmem_ld32(tbase + c, rr);
      ptx::tmem_wait_ld(rr);
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = old[i] + __uint_as_float(rr[i]);
      store_block<C::EPI_OUT>(w, &p.tmC0, ti.n0 + c, row0, v);
    }
  } else if constexpr (KIND == GEMM_DENSE_TN) {
    static_assert(BN == 64 && C::EPI_OUT * 2048 == 32 * BN * 4, "one fp32 row of 64 a lane");
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t rr[32];
      ptx::tmem_ld32(tbase + c, rr);
      ptx::tmem_wait_ld(rr);
      if (p.ksplit > 1) {
        // split K: this CTA's partial of the warp's 32 rows stays in its output
        // staging, one 256-byte fp32 row a lane, 16-byte piece j of row r at piece
        // j ^ (r & 15) (conflict-free for the row-per-lane writes and reads)
        uint8_t* row = w.out + lane * (BN * 4);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int piece = (c / 4 + j) ^ (lane & 15);
          *reinterpret_cast<uint4*>(row + piece * 16) =
              make_uint4(rr[4 * j], rr[4 * j + 1], rr[4 * j + 2], rr[4 * j + 3]);
        }
      } else {
        float v[32];
        as_float(rr, v);
        store_block<C::EPI_OUT>(w, &p.tmC0, ti.n0 + c, row0, v);
      }
    }
  } else {  // weight gradients: dW_down [E*H, I]; dW_gate / dW_up [E*I, H]
    const CUtensorMap* m;
    int orow;
    if (ti.down) {
      m = KIND == GEMM_WGRAD_BOTH ? &p.tmC2 : &p.tmC0;
      orow = ti.e * p.H + row0;
    } else {
      const bool gate = row0 < p.I;
      m = gate ? &p.tmC0 : &p.tmC1;
      orow = ti.e * p.I + (gate ? row0 : row0 - p.I);
    }
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t r[32];
      ptx::tmem_ld32(tbase + c, r);
      ptx::tmem_wait_ld(r);
      float v[32];
      as_float(r, v);
      store_block<C::EPI_OUT>(w, m, ti.n0 + c, orow, v);
    }
  }
  return true;
}

// MXFP8 codes and scale of one 32-column block of a (the down projection's operand).
__device__ __forceinline__ void store_qa(const GemmParams& p, int64_t r, int col,
                                         const uint32_t (&pa)[16]) {
  float a[32];
  unpack32(pa, a);
  uint2 cq[4];
  const int e = mx::quant_row32(a, cq);
  uint4* dq = reinterpret_cast<uint4*>(p.q_codes + r * p.I + col);
  dq[0] = make_uint4(cq[0].x, cq[0].y, cq[1].x, cq[1].y);
  dq[1] = make_uint4(cq[2].x, cq[2].y, cq[3].x, cq[3].y);
  p.q_sf[mx::sf_offset(r, col / 32, p.q_mnb)] = static_cast<uint8_t>(mx::e8m0(e));
}

// Epilogue of one tile for one warp of a SPLIT tile (BN = 256): quadrant q (rows),
// half hh of the columns.  With EARLY_RELEASE the warp's accumulator columns go to
// registers first and release() hands TMEM back before any store.
template <int KIND, int BN, int CTAS, bool FP8, class Release>
__device__ __forceinline__ bool epilogue_tile_split(const GemmParams& p, const TileInfo& ti,
                                                    const TileInfo* next, int q, int hh,
                                                    uint32_t tbase, EpiWarp& w,
                                                    volatile int* abort, Release release) {
  using C = Cfg<KIND, BN, CTAS, FP8>;
  static_assert(BN == 256, "split tiles are 256 wide");
  const int lane = w.lane, row = q * 32 + lane;
  const int row0 = ti.m0 + q * 32;
  if constexpr (KIND == GEMM_GATEUP) {
    // gate columns hh*64 .. hh*64+63, up columns 128 + the same: all four chunks to
    // registers (fp32), TMEM back, then the SwiGLU (its exponentials would otherwise
    // hold the accumulator while the tensor cores wait)
    uint32_t rg[2][32], ru[2][32];
    ptx::tmem_ld32(tbase + hh * 64, rg[0]);
    ptx::tmem_ld32(tbase + 128 + hh * 64, ru[0]);
    ptx::tmem_ld32(tbase + hh * 64 + 32, rg[1]);
    ptx::tmem_ld32(tbase + 128 + hh * 64 + 32, ru[1]);
    ptx::tmem_wait_ld(rg[0]);
    ptx::reg_fence(ru[0]);
    ptx::reg_fence(rg[1]);
    ptx::reg_fence(ru[1]);
    release();
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int c = ti.n0 + hh * 64 + 32 * j;
      float g[32], u[32], a[32];
      as_float(rg[j], g);
      as_float(ru[j], u);
#pragma unroll
      for (int i = 0; i < 32; ++i) a[i] = g[i] * sigmoidf_(g[i]) * u[i];
      uint32_t pk[16];
      pack32(g, pk);
      store_block_p<C::EPI_OUT>(w, &p.tmC0, c, row0, pk);
      pack32(u, pk);
      store_block_p<C::EPI_OUT>(w, &p.tmC0, p.I + c, row0, pk);
      pack32(a, pk);
      store_block_p<C::EPI_OUT>(w, &p.tmC1, c, row0, pk);
      if (p.q_codes != nullptr) store_qa(p, row0 + lane, c, pk);  // from a's bf16 value
    }
  } else if constexpr (KIND == GEMM_DGRAD_DOWN) {
    // g' stays fp32, as the accumulator holds it.  The warp parks chunks 1-3 of its
    // 128 columns in spare TMEM columns (tcgen05.st), takes chunk 0 to registers and
    // hands the accumulator back to the MMA issuer; the dSwiGLU then works chunk by
    // chunk, each chunk's inputs (g, u, a) arriving by TMA during the previous one.
    const int64_t pr = ti.m0 + row;
    const float wgt = __ldg(p.w_row + pr);
    const uint32_t t0 = tbase + hh * 128;
    const uint32_t stash = tbase + C::STASH_COL0 + hh * 96;  // (one accumulator, at column 0)
    float dot = 0.f;
    auto chunk = [&](int j, const uint32_t (&gp)[32]) -> bool {
      const int c = hh * 128 + 32 * j;
      if (!w.ld_pending) load_inputs(w, p, row0, ti.n0 + c);
      if (!wait_inputs(w, abort)) return false;
      // the inputs to registers (bf16 pairs), then the next chunk's (or the next
      // tile's first) are requested while this one is computed
      uint32_t gw[16], uw[16], aw[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 G = *reinterpret_cast<const uint4*>(swz(w.in, lane, k));
        const uint4 U = *reinterpret_cast<const uint4*>(swz(w.in + 2048, lane, k));
        const uint4 A = *reinterpret_cast<const uint4*>(swz(w.in + 4096, lane, k));
        gw[4 * k] = G.x, gw[4 * k + 1] = G.y, gw[4 * k + 2] = G.z, gw[4 * k + 3] = G.w;
        uw[4 * k] = U.x, uw[4 * k + 1] = U.y, uw[4 * k + 2] = U.z, uw[4 * k + 3] = U.w;
        aw[4 * k] = A.x, aw[4 * k + 1] = A.y, aw[4 * k + 2] = A.z, aw[4 * k + 3] = A.w;
      }
      __syncwarp();
      if (j < 3) load_inputs(w, p, row0, ti.n0 + c + 32);
      else if (next != nullptr) load_inputs(w, p, next->m0 + q * 32, next->n0 + hh * 128);
      auto lo = [](uint32_t v) { return __uint_as_float(v << 16); };
      auto hi = [](uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); };
      // dg, du, w*a: one output block each, 8 columns at a time
      uint8_t* b = begin_block<C::EPI_OUT>(w);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int x = 4 * k + i;
          float v[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float g = h ? hi(gw[x]) : lo(gw[x]), u = h ? hi(uw[x]) : lo(uw[x]);
            const float sg = sigmoidf_(g);
            v[h] = wgt * __uint_as_float(gp[2 * x + h]) * u * sg * (1.0f + g * (1.0f - sg));
          }
          o[i] = pack2(v[0], v[1]);
        }
        *reinterpret_cast<uint4*>(swz(b, lane, k)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
      end_block<C::EPI_OUT>(w, &p.tmC0, ti.n0 + c, row0, b);
      b = begin_block<C::EPI_OUT>(w);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int x = 4 * k + i;
          float v[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float g = h ? hi(gw[x]) : lo(gw[x]);
            v[h] = wgt * __uint_as_float(gp[2 * x + h]) * g * sigmoidf_(g);
          }
          o[i] = pack2(v[0], v[1]);
        }
        *reinterpret_cast<uint4*>(swz(b, lane, k)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
      end_block<C::EPI_OUT>(w, &p.tmC0, p.I + ti.n0 + c, row0, b);
      b = begin_block<C::EPI_OUT>(w);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int x = 4 * k + i;
          const float a0 = lo(aw[x]), a1 = hi(aw[x]);
          dot += a0 * __uint_as_float(gp[2 * x]) + a1 * __uint_as_float(gp[2 * x + 1]);
          o[i] = pack2(a0 * wgt, a1 * wgt);  // w * a, the dW_down operand
        }
        *reinterpret_cast<uint4*>(swz(b, lane, k)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
      end_block<C::EPI_OUT>(w, &p.tmC1, ti.n0 + c, row0, b);
      return true;
    };
    uint32_t r[32];
#pragma unroll 1
    for (int j = 1; j < 4; ++j) {
      ptx::tmem_ld32(t0 + 32 * j, r);
      ptx::tmem_wait_ld(r);
      ptx::tmem_st32(stash + 32 * (j - 1), r);
    }
    ptx::tmem_ld32(t0, r);
    ptx::tmem_wait_ld(r);
    ptx::tmem_wait_st();
    release();
    if (!chunk(0, r)) return false;
#pragma unroll 1
    for (int j = 1; j < 4; ++j) {
      ptx::tmem_ld32(stash + 32 * (j - 1), r);
      ptx::tmem_wait_ld(r);
      if (!chunk(j, r)) return false;
    }
    // two partial sums per row and N tile, one per column half
    p.outf[pr * p.n_pw + (ti.n0 / BN) * 2 + hh] = dot;
  } else {
    const CUtensorMap* m = &p.tmC0;
    int orow = row0;
    float wgt = 1.0f;
    if constexpr (KIND == GEMM_DOWN) {
      wgt = __ldg(p.w_row + ti.m0 + row);
    } else if constexpr (KIND != GEMM_DGRAD_GATEUP) {  // weight gradients
      if (ti.down) {
        m = KIND == GEMM_WGRAD_BOTH ? &p.tmC2 : &p.tmC0;
        orow = ti.e * p.H + row0;
      } else {
        const bool gate = row0 < p.I;
        m = gate ? &p.tmC0 : &p.tmC1;
        orow = ti.e * p.I + (gate ? row0 : row0 - p.I);
      }
    }
    // the warp's 128 accumulator columns to registers, then TMEM goes back at once
    uint32_t r[4][32];
    ptx::tmem_ld32(tbase + hh * 128, r[0]);
    ptx::tmem_ld32(tbase + hh * 128 + 32, r[1]);
    ptx::tmem_ld32(tbase + hh * 128 + 64, r[2]);
    ptx::tmem_ld32(tbase + hh * 128 + 96, r[3]);
    ptx::tmem_wait_ld(r[0]);
    ptx::reg_fence(r[1]);
    ptx::reg_fence(r[2]);
    ptx::reg_fence(r[3]);
    release();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float v[32];
      as_float(r[j], v);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] *= wgt;
      uint32_t pk[16];
      pack32(v, pk);
      store_block_p<C::EPI_OUT>(w, m, ti.n0 + hh * 128 + 32 * j, orow, pk);
    }
  }
  return true;
}

// Zero tile of a per-expert GEMM whose expert has no rows (K = 0).
// (SPLIT: this warp's half hh of the columns)
template <int KIND, int BN, int CTAS, bool FP8>
__device__ __forceinline__ void zero_tile(const GemmParams& p, const TileInfo& ti, int q, int hh,
                                          EpiWarp& w) {
  using C = Cfg<KIND, BN, CTAS, FP8>;
  const int row0 = ti.m0 + q * 32;
  const CUtensorMap* m;
  int orow;
  if (ti.down) {
    m = KIND == GEMM_WGRAD_BOTH ? &p.tmC2 : &p.tmC0;
    orow = ti.e * p.H + row0;
  } else {
    const bool gate = row0 < p.I;
    m = gate ? &p.tmC0 : &p.tmC1;
    orow = ti.e * p.I + (gate ? row0 : row0 - p.I);
  }
  float z[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) z[i] = 0.f;
  const int c0 = C::SPLIT ? hh * (BN / 2) : 0, c1 = C::SPLIT ? c0 + BN / 2 : BN;
#pragma unroll 1
  for (int c = c0; c < c1; c += 32) store_block<C::EPI_OUT>(w, m, ti.n0 + c, orow, z);
}

// ------------------------------------------------------------------ producer loads
template <int CTAS>
__device__ __forceinline__ void tma(void* dst, const CUtensorMap* m, uint32_t bar, int c0,
                                    int c1) {
  if constexpr (CTAS == 1)
    ptx::tma_load_2d(dst, m, bar, c0, c1);
  else
    ptx::tma_load_2d_pair(dst, m, bar, c0, c1);
}

// One 512-byte scale atom (FP8): atom `atom` of the scale tensor of map m.
template <int CTAS>
__device__ __forceinline__ void sf_atom(void* dst, const CUtensorMap* m, uint32_t bar,
                                        int64_t atom) {
  tma<CTAS>(dst, m, bar, 0, static_cast<int32_t>(atom * 4));
}

// The 128 K-major rows of A from row m0 at column k0 (grouped kinds).  MC: the two
// pairs of the cluster share them (same M tile); this CTA loads half of them, the
// half of its pair's parity, into its own and its counterpart's stage (the CTA of the
// other pair with the same place in its pair).
template <int CTAS, bool MC>
__device__ __forceinline__ void load_a(const GemmParams& p, uint8_t* sa, uint32_t bar, int k0,
                                       int m0, int rank) {
  if constexpr (MC) {
    const int half = rank >> 1;
    const uint16_t mask = static_cast<uint16_t>(0x5u << (rank & 1));
    ptx::tma_load_2d_pair_mc(sa + half * (BM / 2) * 128, &p.tmA_half, bar, k0,
                             m0 + half * (BM / 2), mask);
  } else {
    tma<CTAS>(sa, &p.tmA, bar, k0, m0);
  }
}

// This CTA's share of k block kb: its 128 rows of A and its B_ROWS rows (K-major)
// or columns (M/N-major) of B, completing on the barrier at cluster address `bar`;
// FP8: also the stage's scale atoms into sf (A's, then B's BN / 128).  `rank`: the
// CTA's cluster rank (its place in its pair is rank & 1).
template <int KIND, int BN, int CTAS, bool FP8, bool MC = false>
__device__ __forceinline__ void issue_loads(const GemmParams& p, const TileInfo& ti, int kb,
                                            uint8_t* sa, uint8_t* sb, uint8_t* sf, uint32_t bar,
                                            int rank) {
  using C = Cfg<KIND, BN, CTAS, FP8>;
  const int k0 = kb * C::KSTEP;
  const int prank = rank & 1;
  const int nb = ti.n0 + prank * C::B_ROWS;  // first B row / column of this CTA
  constexpr int NBOX = C::B_ROWS / C::MN_BOX;  // M/N-major boxes of B per stage
  constexpr int BOX_BYTES = 128 * C::KSTEP;  // bytes of one M/N-major box (128-byte rows)
  if constexpr (KIND == GEMM_GATEUP) {
    load_a<CTAS, MC>(p, sa, bar, k0, ti.m0, rank);
    if (CTAS == 1) {
      tma<CTAS>(sb, &p.tmB0, bar, k0, ti.e * p.I + ti.n0);
      tma<CTAS>(sb + (BN / 2) * 128, &p.tmB1, bar, k0, ti.e * p.I + ti.n0);
    } else {  // the pair's first CTA stages the gate rows, the second the up rows
      tma<CTAS>(sb, prank == 0 ? &p.tmB0 : &p.tmB1, bar, k0, ti.e * p.I + ti.n0);
    }
    if constexpr (FP8) {  // N = [gate rows | up rows] of the tile
      const int kg = k0 / 128;
      sf_atom<CTAS>(sf, &p.tmSA, bar, static_cast<int64_t>(kg) * p.sfa_mnb + ti.m0 / 128);
      const int64_t bb = static_cast<int64_t>(kg) * p.sfb_mnb + (ti.e * p.I + ti.n0) / 128;
      sf_atom<CTAS>(sf + 512, &p.tmSB0, bar, bb);
      sf_atom<CTAS>(sf + 1024, &p.tmSB1, bar, bb);
    }
  } else if constexpr (KIND == GEMM_DOWN) {
    load_a<CTAS, MC>(p, sa, bar, k0, ti.m0, rank);
    tma<CTAS>(sb, &p.tmB0, bar, k0, ti.e * p.H + nb);
    if constexpr (FP8) {
      const int kg = k0 / 128;
      sf_atom<CTAS>(sf, &p.tmSA, bar, static_cast<int64_t>(kg) * p.sfa_mnb + ti.m0 / 128);
#pragma unroll
      for (int j = 0; j < BN / 128; ++j)
        sf_atom<CTAS>(sf + 512 * (1 + j), &p.tmSB0, bar,
                      static_cast<int64_t>(kg) * p.sfb_mnb + (ti.e * p.H + ti.n0) / 128 + j);
    }
  } else if constexpr (KIND == GEMM_DGRAD_DOWN) {
    load_a<CTAS, MC>(p, sa, bar, k0, ti.m0, rank);
#pragma unroll
    for (int c = 0; c < NBOX; ++c)
      tma<CTAS>(sb + c * BOX_BYTES, &p.tmB0, bar, nb + c * C::MN_BOX, ti.e * p.H + k0);
    if constexpr (FP8) {  // B's scales: MN = I, K = the experts' stacked H rows
      sf_atom<CTAS>(sf, &p.tmSA, bar, static_cast<int64_t>(k0 / 128) * p.sfa_mnb + ti.m0 / 128);
      const int64_t kg = (static_cast<int64_t>(ti.e) * p.H + k0) / 128;
#pragma unroll
      for (int j = 0; j < BN / 128; ++j)
        sf_atom<CTAS>(sf + 512 * (1 + j), &p.tmSB0, bar, kg * p.sfb_mnb + ti.n0 / 128 + j);
    }
  } else if constexpr (KIND == GEMM_DGRAD_GATEUP) {
    load_a<CTAS, MC>(p, sa, bar, k0, ti.m0, rank);
    const bool gate = k0 < p.I;
    const CUtensorMap* m = gate ? &p.tmB0 : &p.tmB1;
    const int krow = ti.e * p.I + (gate ? k0 : k0 - p.I);
#pragma unroll
    for (int c = 0; c < NBOX; ++c)
      tma<CTAS>(sb + c * BOX_BYTES, m, bar, nb + c * C::MN_BOX, krow);
    if constexpr (FP8) {  // B's scales: MN = H, K = the experts' stacked I rows
      sf_atom<CTAS>(sf, &p.tmSA, bar, static_cast<int64_t>(k0 / 128) * p.sfa_mnb + ti.m0 / 128);
      const CUtensorMap* ms = gate ? &p.tmSB0 : &p.tmSB1;
#pragma unroll
      for (int j = 0; j < BN / 128; ++j)
        sf_atom<CTAS>(sf + 512 * (1 + j), ms, bar,
                      static_cast<int64_t>(krow / 128) * p.sfb_mnb + ti.n0 / 128 + j);
    }
  } else if constexpr (C::DENSE) {
    const int kd = k0 + ti.k_row0;  // (a split-K share starts at k_row0)
    if constexpr (KIND != GEMM_DENSE_TN) {
      tma<CTAS>(sa, &p.tmA, bar, kd, ti.m0);  // A [M, K]
    } else {
#pragma unroll
      for (int c = 0; c < BM / 64; ++c) tma<CTAS>(sa + c * 8192, &p.tmA, bar, ti.m0 + c * 64, kd);
    }
    if constexpr (KIND == GEMM_DENSE_NT) {
      tma<CTAS>(sb, &p.tmB0, bar, kd, ti.n0);  // B [N, K]
    } else {
#pragma unroll
      for (int c = 0; c < C::B_ROWS / 64; ++c)
        tma<CTAS>(sb + c * 8192, &p.tmB0, bar, ti.n0 + c * 64, kd);  // B [K, N]
    }
  } else {  // per-expert weight gradients: both operands M/N-major, K = routed rows
    const int krow = ti.k_row0 + k0;
    const bool second = KIND == GEMM_WGRAD_BOTH && ti.down;
    const CUtensorMap* ma = second ? &p.tmA2 : &p.tmA;
    const CUtensorMap* mb = second ? &p.tmB2 : &p.tmB0;
#pragma unroll
    for (int c = 0; c < BM / C::MN_BOX; ++c)
      tma<CTAS>(sa + c * BOX_BYTES, ma, bar, ti.m0 + c * C::MN_BOX, krow);
#pragma unroll
    for (int c = 0; c < NBOX; ++c)
      tma<CTAS>(sb + c * BOX_BYTES, mb, bar, nb + c * C::MN_BOX, krow);
    if constexpr (FP8) {  // scales of both: MN = the output's rows / columns, K = rows
      const int64_t kg = krow / 128;
      const int amnb = second ? p.sfa2_mnb : p.sfa_mnb;
      const int bmnb = second ? p.sfb2_mnb : p.sfb_mnb;
      sf_atom<CTAS>(sf, second ? &p.tmSA2 : &p.tmSA, bar, kg * amnb + ti.m0 / 128);
#pragma unroll
      for (int j = 0; j < BN / 128; ++j)
        sf_atom<CTAS>(sf + 512 * (1 + j), second ? &p.tmSB2 : &p.tmSB0, bar,
                      kg * bmnb + ti.n0 / 128 + j);
    }
  }
}

// ------------------------------------------------------------------ the kernel
// MC: A multicast between the two SM pairs of a four-CTA cluster (grouped bf16 kinds
// with an even number of N tiles): the pairs run N tiles 2j and 2j + 1 of the same M
// tile in step, each CTA loading half of its A rows for itself and its counterpart in
// the other pair, so a ring stage is refilled only once both pairs have consumed it
// (each stage's empty barrier takes one arrival from each pair's MMA issuer).
template <int KIND, int BN, int CTAS, bool FP8, bool MC = false>
__global__ void __launch_bounds__(Cfg<KIND, BN, CTAS, FP8>::THREADS, 1)
    moe_gemm_kernel(const __grid_constant__ GemmParams p) {
  using C = Cfg<KIND, BN, CTAS, FP8>;
  static_assert(!MC || (CTAS == 2 && !FP8 && !C::DENSE && !C::PER_EXPERT), "A multicast");
  constexpr int CL = MC ? 2 * CTAS : CTAS;  // CTAs per cluster
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::STAGES];
  __shared__ __align__(8) uint64_t empty_bar[C::STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ __align__(8) uint64_t epi_ld_bar[8];
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = CTAS == 1 ? 0 : static_cast<int>(ptx::cluster_rank());
  const int prank = rank & 1, leader = rank & ~1;  // place in the pair; the pair's first CTA
  // A^T.B with K split: clusters of p.ksplit CTAs, one tile a cluster, the CTA of rank
  // ks taking the ks-th share of K
  const bool splitk = KIND == GEMM_DENSE_TN && p.ksplit > 1;
  const int ks = splitk ? static_cast<int>(ptx::cluster_rank()) : 0;
  const int cl_size = splitk ? p.ksplit : CL;
  const int cluster = blockIdx.x / cl_size, n_clusters = gridDim.x / cl_size;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(&full_bar[s], 1);
      ptx::mbar_init(&empty_bar[s], MC ? 2 : 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull_bar[a], 1);
      ptx::mbar_init(&tempty_bar[a], C::EPI_WARPS * CTAS);
    }
    ptx::mbar_init(&drain_bar, 1);
    for (int q = 0; q < C::EPI_WARPS; ++q) ptx::mbar_init(&epi_ld_bar[q], 1);
    s_abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(MC ? &p.tmA_half : &p.tmA);
    ptx::prefetch_tmap(&p.tmB0);
    if (KIND == GEMM_GATEUP || KIND == GEMM_DGRAD_GATEUP) ptx::prefetch_tmap(&p.tmB1);
    if (KIND == GEMM_WGRAD_BOTH) {
      ptx::prefetch_tmap(&p.tmA2);
      ptx::prefetch_tmap(&p.tmB2);
    }
    if constexpr (FP8) {
      ptx::prefetch_tmap(&p.tmSA);
      ptx::prefetch_tmap(&p.tmSB0);
      if (KIND == GEMM_GATEUP || KIND == GEMM_DGRAD_GATEUP) ptx::prefetch_tmap(&p.tmSB1);
      if (KIND == GEMM_WGRAD_BOTH) {
        ptx::prefetch_tmap(&p.tmSA2);
        ptx::prefetch_tmap(&p.tmSB2);
      }
    }
  }
  if (warp == 2) {
    ptx::tmem_alloc<CTAS>(&s_tmem_base, C::TMEM_COLS);
    ptx::tmem_relinquish<CTAS>();
  }
  ptx::tc_fence_before();
  if constexpr (CTAS == 2) ptx::cluster_sync(); else __syncthreads();
  ptx::tc_fence_after();
  // the prologue above touched no global memory: it overlaps the previous kernel
  pdl_wait();
  pdl_trigger();
  const uint32_t tmem_base = s_tmem_base;
  volatile int* abort = &s_abort;
  Peers peers;
  for (int r = 1; r < CL; ++r)
    peers.a[peers.n++] = ptx::map_to_rank(ptx::smem_u32(&s_abort), static_cast<uint32_t>(rank ^ r));
  const int total = total_tiles<KIND, BN, CTAS, FP8, MC>(p);
  uint8_t* const sf_ring = smem + C::STAGES * C::STAGE_BYTES;  // FP8 scale atoms per stage
  // the pair's barriers that both CTAs signal live in its first CTA
  const uint32_t lead_full0 =
      CTAS == 1 ? ptx::smem_u32(&full_bar[0])
                : ptx::map_to_rank(ptx::smem_u32(&full_bar[0]), static_cast<uint32_t>(leader));

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- producer
    int stage = 0;
    uint32_t phase = 0;
    int last_parity[C::STAGES];
#pragma unroll
    for (int s = 0; s < C::STAGES; ++s) last_parity[s] = -1;
    bool ok = true;
    for (int t = cluster; t < total && ok; t += n_clusters) {
      const TileInfo ti = decode_tile<KIND, BN, CTAS, FP8, MC>(p, t, rank, ks);
      for (int kb = 0; kb < ti.k_iters; ++kb) {
        if (!ptx::mbar_wait_spin(&empty_bar[stage], phase ^ 1u, abort, WAIT_LIMIT_NS)) {
          record_timeout(p, abort, KIND * 16 + 1, peers);
          ok = false;
          break;
        }
        uint8_t* sa = smem + stage * C::STAGE_BYTES;
        if (prank == 0)
          ptx::mbar_arrive_expect_tx(&full_bar[stage], (C::STAGE_BYTES + C::SF_BYTES) * CTAS);
        // (with p.stall the first stage of CTA 0 never fills: the MMA issuer's bounded
        // wait runs out and every role unwinds, the path a lost copy would take)
        if (!(p.stall && blockIdx.x == 0 && t == cluster && kb == 0))
          issue_loads<KIND, BN, CTAS, FP8, MC>(p, ti, kb, sa, sa + C::A_BYTES,
                                           sf_ring + stage * C::SF_BYTES,
                                           lead_full0 + stage * 8u, rank);
        last_parity[stage] = static_cast<int>(phase);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // drain: every issued copy has landed before the CTA may exit (a pair's first CTA:
    // its full barriers; the other: consumption of its stages, which implies they
    // landed; with MC the stages' consumption by both pairs, and the first CTAs' full
    // barriers count the copies into their pairs from either pair).  After a failure
    // the stages may never complete: all waits share one time budget.
    const uint64_t deadline = ptx::globaltimer() + WAIT_LIMIT_NS;
    for (int s = 0; s < C::STAGES; ++s) {
      if (last_parity[s] < 0) continue;
      uint64_t* bar = prank == 0 ? &full_bar[s] : &empty_bar[s];
      if (!ptx::mbar_wait_until(bar, static_cast<uint32_t>(last_parity[s]), deadline)) {
        record_timeout(p, abort, KIND * 16 + 2);
        break;
      }
    }
  } else if (warp == 1 && lane == 0 && prank == 0) {
    // ---------------------------------------------------------------- MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    bool issued = false;
    for (int t = cluster; t < total && ok; t += n_clusters) {
      const TileInfo ti = decode_tile<KIND, BN, CTAS, FP8, MC>(p, t, rank, ks);
      if (ti.k_iters == 0) continue;
      if (!ptx::mbar_wait_spin(&tempty_bar[acc], acc_phase ^ 1u, abort, WAIT_LIMIT_NS)) {
        record_timeout(p, abort, KIND * 16 + 3, peers);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
      for (int kb = 0; kb < ti.k_iters; ++kb) {
        if (!ptx::mbar_wait_spin(&full_bar[stage], phase, abort, WAIT_LIMIT_NS)) {
          record_timeout(p, abort, KIND * 16 + 4, peers);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t a_base = ptx::smem_u32(smem + stage * C::STAGE_BYTES);
        const uint32_t b_base = a_base + C::A_BYTES;
        if constexpr (FP8) {
          // the stage's scales into TMEM, then four MMAs of K = 32: each advances 32
          // bytes along a K-major row, or 32 rows (4 KB) of an M/N-major box, and
          // reads byte kk of the scale words
          const uint32_t sf_base = ptx::smem_u32(sf_ring + stage * C::SF_BYTES);
          const uint32_t sfa_t = tmem_base + C::SF_COL0 + stage * C::SF_COLS_PER_STAGE;
          const uint32_t sfb_t = sfa_t + 4;
          ptx::tmem_cp_sf<CTAS>(sfa_t, ptx::smem_desc_sf(sf_base));
#pragma unroll
          for (int j = 0; j < BN / 128; ++j)
            ptx::tmem_cp_sf<CTAS>(sfb_t + 4 * j, ptx::smem_desc_sf(sf_base + 512 * (1 + j)));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t adesc = C::A_MN
                                       ? ptx::smem_desc_sw128(a_base + kk * 4096, 16384, 1024)
                                       : ptx::smem_desc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bdesc = C::B_MN
                                       ? ptx::smem_desc_sw128(b_base + kk * 4096, 16384, 1024)
                                       : ptx::smem_desc_sw128(b_base + kk * 32, 16, 1024);
            ptx::umma_mxf8<CTAS>(d_tmem, adesc, bdesc, C::IDESC | ptx::sf_ids(kk), sfa_t, sfb_t,
                                 (kb | kk) != 0 ? 1u : 0u);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t adesc = C::A_MN
                                       ? ptx::smem_desc_sw128(a_base + kk * 2048, 8192, 1024)
                                       : ptx::smem_desc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bdesc = C::B_MN
                                       ? ptx::smem_desc_sw128(b_base + kk * 2048, 8192, 1024)
                                       : ptx::smem_desc_sw128(b_base + kk * 32, 16, 1024);
            ptx::umma_bf16<CTAS>(d_tmem, adesc, bdesc, C::IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
        }
        issued = true;
        // the stage is free once this pair's MMAs have read it (MC: in every CTA of
        // the cluster, whose empty barriers also wait for the other pair's)
        ptx::umma_commit<CTAS>(&empty_bar[stage], MC ? 0xF : 0x3);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      ptx::umma_commit<CTAS>(&tfull_bar[acc], static_cast<uint16_t>(0x3u << leader));
      if (++acc == C::NACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (issued) {
      // drain: every issued MMA has completed before TMEM or the pair's shared memory
      // is released
      ptx::umma_commit<CTAS>(&drain_bar, static_cast<uint16_t>(0x1u << leader));
      int dummy = 0;
      if (!ptx::mbar_wait(&drain_bar, 0, &dummy, WAIT_LIMIT_NS))
        record_timeout(p, abort, KIND * 16 + 5);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue
    // warp 4 + ew: TMEM lane quadrant q = warp % 4 (the quadrant a warp may read),
    // column half hh (SPLIT tiles)
    const int ew = warp - 4, q = warp & 3, hh = ew >> 2;
    EpiWarp w;
    w.in = smem + C::STAGES * (C::STAGE_BYTES + C::SF_BYTES) + ew * C::EPI_WARP_BYTES;
    w.out = w.in + C::EPI_IN * 2048;
    w.ld_bar = &epi_ld_bar[ew];
    w.ld_phase = 0;
    w.ld_pending = false;
    w.ob = 0;
    w.lane = lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    const uint32_t lead_tempty0 =
        CTAS == 1
            ? ptx::smem_u32(&tempty_bar[0])
            : ptx::map_to_rank(ptx::smem_u32(&tempty_bar[0]), static_cast<uint32_t>(leader));
    for (int t = cluster; t < total; t += n_clusters) {
      const TileInfo ti = decode_tile<KIND, BN, CTAS, FP8, MC>(p, t, rank, ks);
      if (ti.k_iters == 0) {
        if constexpr (C::PER_EXPERT) zero_tile<KIND, BN, CTAS, FP8>(p, ti, q, hh, w);
        continue;
      }
      TileInfo nx;
      const bool has_next = t + n_clusters < total;
      if (has_next) nx = decode_tile<KIND, BN, CTAS, FP8, MC>(p, t + n_clusters, rank, ks);
      if (KIND == GEMM_DGRAD_DOWN && !w.ld_pending)
        load_inputs(w, p, ti.m0 + q * 32, ti.n0 + (C::SPLIT ? hh * (BN / 2) : 0));
      if (KIND == GEMM_DENSE_NN && !w.ld_pending) load_c_blocks<BN>(w, p, ti.m0 + q * 32, ti.n0);
      int ok = 1;
      if (lane == 0)
        ok = ptx::mbar_wait_spin(&tfull_bar[acc], acc_phase, abort, WAIT_LIMIT_NS) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) record_timeout(p, abort, KIND * 16 + 6, peers);
        break;
      }
      ptx::tc_fence_after();
      __syncwarp();
      const uint32_t tbase = tmem_base + static_cast<uint32_t>(acc * BN) +
                             (static_cast<uint32_t>(q * 32) << 16);
      // hand the accumulator back to the MMA issuer (every epilogue warp of the pair
      // arrives once per tile).  The warp's TMEM reads have completed (tcgen05.wait::ld)
      // before it arrives, so the arrive needs no release of its memory writes: a
      // relaxed arrive, which does not wait for the previous tile's global stores to
      // become visible (with a release arrive the tensor cores sat idle about a
      // microsecond per tile while they drained)
      auto release = [&]() {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0)
          ptx::mbar_arrive_cluster_relaxed(CTAS == 1 ? ptx::smem_u32(&tempty_bar[acc])
                                                     : lead_tempty0 + acc * 8u);
      };
      bool done;
      if constexpr (C::SPLIT)
        done = epilogue_tile_split<KIND, BN, CTAS, FP8>(p, ti, has_next ? &nx : nullptr, q, hh,
                                                        tbase, w, abort, release);
      else
        done = epilogue_tile<KIND, BN, CTAS, FP8>(p, ti, has_next ? &nx : nullptr, q, tbase, w,
                                                  abort);
      if (!done) {
        if (lane == 0) record_timeout(p, abort, KIND * 16 + 7, peers);
        break;
      }
      if (!C::EARLY_RELEASE) release();
      if (++acc == C::NACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // drain: outstanding input loads and output stores complete before the CTA exits
    if (w.ld_pending && lane == 0) {
      int dummy = 0;
      if (!ptx::mbar_wait(w.ld_bar, w.ld_phase, &dummy, WAIT_LIMIT_NS))
        record_timeout(p, abort, KIND * 16 + 8);
    }
    if (lane == 0) ptx::bulk_wait_all();
    __syncwarp();
  }

  ptx::tc_fence_before();
  if (CTAS == 2 || splitk) ptx::cluster_sync(); else __syncthreads();
  ptx::tc_fence_after();
  if constexpr (KIND == GEMM_DENSE_TN) {
    if (splitk) {
      // every CTA's partial tile is in its staging: CTA ks sums rows ks*BM/ksplit .. of
      // all of them in rank order (epilogue warp ew: columns 16 ew .. 16 ew + 15, one row
      // a lane) and stores the bf16 result; the second barrier keeps each CTA's shared
      // memory until the others have read it
      if (warp >= 4 && warp < 4 + C::EPI_WARPS && cluster < total) {
        const int ew = warp - 4;
        const TileInfo ti = decode_tile<KIND, BN, CTAS, FP8, MC>(p, cluster, rank, ks);
        const int rows = BM / p.ksplit;
        const uint32_t base = ptx::smem_u32(smem + C::STAGES * (C::STAGE_BYTES + C::SF_BYTES) +
                                            C::EPI_IN * 2048);
#pragma unroll 1
        for (int rr = 0; rr < rows; rr += 32) {
          const int r = ks * rows + rr + lane;  // row of the tile
          if (rr + lane >= rows) continue;
          const uint32_t row_off = static_cast<uint32_t>((r >> 5) * C::EPI_WARP_BYTES +
                                                         (r & 31) * (BN * 4));
          float acc[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[i] = 0.f;
          for (int s = 0; s < p.ksplit; ++s) {
            const uint32_t src = ptx::map_to_rank(base + row_off, static_cast<uint32_t>(s));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int piece = (4 * ew + j) ^ (r & 15);
              const float4 v = ptx::ld_cluster_f4(src + piece * 16);
              acc[4 * j] += v.x;
              acc[4 * j + 1] += v.y;
              acc[4 * j + 2] += v.z;
              acc[4 * j + 3] += v.w;
            }
          }
          const int orow = ti.m0 + r, ocol = ti.n0 + 16 * ew;
          if (orow < p.dm && ocol < p.dn) {
            uint16_t* o = p.out0 + static_cast<int64_t>(orow) * p.dn + ocol;
            if (ocol + 16 <= p.dn) {
              uint4* o4 = reinterpret_cast<uint4*>(o);
              o4[0] = make_uint4(pack2(acc[0], acc[1]), pack2(acc[2], acc[3]),
                                 pack2(acc[4], acc[5]), pack2(acc[6], acc[7]));
              o4[1] = make_uint4(pack2(acc[8], acc[9]), pack2(acc[10], acc[11]),
                                 pack2(acc[12], acc[13]), pack2(acc[14], acc[15]));
            } else {
              for (int i = 0; ocol + i < p.dn; ++i) {
                const __nv_bfloat16 b = __float2bfloat16_rn(acc[i]);
                o[i] = *reinterpret_cast<const uint16_t*>(&b);
              }
            }
          }
        }
      }
      ptx::cluster_sync();
    }
  }
  if (warp == 2) ptx::tmem_dealloc<CTAS>(tmem_base, C::TMEM_COLS);
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Row-major matrix [outer, inner] of bf16 (or, with fp8, of bytes: e4m3 codes) -> 2-D
// tensor map with a box of box_inner x box_outer elements and the given shared-memory
// swizzle.
static bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                     uint32_t box_inner, uint32_t box_outer,
                     CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B, bool fp8 = false) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * (fp8 ? 1 : 2)};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// e4m3 operand [outer, inner] bytes, boxes of 128 bytes x box_outer rows, 128B swizzle.
static bool make_fp8_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                         uint32_t box_outer) {
  return make_map(m, base, inner, outer, 128, box_outer, CU_TENSOR_MAP_SWIZZLE_128B, true);
}

// Scale tensor of `bytes` bytes (a whole number of 512-byte atoms) seen as rows of 128
// bytes; one box is one atom (4 rows), landing unswizzled in shared memory.
static bool make_sf_map(CUtensorMap* m, const void* base, uint64_t bytes) {
  return make_map(m, base, 128, bytes / 128, 128, 4, CU_TENSOR_MAP_SWIZZLE_NONE, true);
}

// 32 x 32 epilogue blocks (64-byte rows, 64-byte swizzle).
static bool make_epi_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer) {
  return make_map(m, base, inner, outer, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

template <int KIND, int BN, int CTAS, bool FP8, bool MC = false>
static cudaError_t run(const Ctx& c, const GemmParams& p, int64_t max_clusters) {
  using C = Cfg<KIND, BN, CTAS, FP8>;
  constexpr int CL = MC ? 2 * CTAS : CTAS;  // CTAs per cluster
  auto kern = moe_gemm_kernel<KIND, BN, CTAS, FP8, MC>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = c.stream;
  cfg.attrs = attr;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // (see pdl_wait)
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 1;
  int64_t clusters = c.num_sms / CL;
  if constexpr (CL > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CL;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
    static int active = 0;  // clusters resident at once (the same for every launch)
    if (active == 0) {
      cfg.gridDim = dim3(static_cast<unsigned>(CL * clusters), 1, 1);
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) active = n;
      else active = static_cast<int>(clusters);
    }
    clusters = active;
  }
  clusters = std::max<int64_t>(1, std::min<int64_t>(clusters, max_clusters));
  int cl_size = CL;
  if (KIND == GEMM_DENSE_TN && p.ksplit > 1) {
    // split K: one tile per cluster of ksplit CTAs, as many clusters as tiles (in
    // waves if they exceed the GPU; no cluster waits for another)
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(p.ksplit);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
    clusters = max_clusters;
    cl_size = p.ksplit;
  }
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * cl_size), 1, 1);
  static constexpr int kId[10] = {K_GEMM_GATEUP,       K_GEMM_DOWN,       K_GEMM_DGRAD_DOWN,
                                  K_GEMM_DGRAD_GATEUP, K_GEMM_WGRAD_DOWN, K_GEMM_WGRAD_GATEUP,
                                  K_GEMM_WGRAD,        K_DENSE_NT,        K_DENSE_NN,
                                  K_DENSE_TN};
  prof_begin(c, kId[KIND]);
  e = cudaLaunchKernelEx(&cfg, kern, p);
  prof_end(c, kId[KIND]);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Launch of the instantiation (kind, bn, ctas) for bf16 (gemm.cu) or MXFP8
// (gemm_fp8.cu) operands; cudaErrorInvalidValue when none exists.  mc: the bf16
// A-multicast form (SM pairs, grouped kinds; p.tmA_half set, max_units in clusters
// of two pairs).
cudaError_t run_bf16(const Ctx& c, const GemmParams& p, int kind, int bn, int ctas,
                     int64_t max_units, bool mc = false);
cudaError_t run_fp8(const Ctx& c, const GemmParams& p, int kind, int bn, int ctas,
                    int64_t max_units);

}  // namespace gemm
}  // namespace mmmoe

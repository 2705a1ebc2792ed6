// gemm.cu -- the expert GEMMs of the layer as one persistent, warp-specialised
// tcgen05 kernel template for sm_103a (TMA -> 128B-swizzled shared memory ring ->
// tcgen05.mma with fp32 accumulators in TMEM, double-buffered -> epilogue warps).
//
// Prime Mega MoE pages, "How does the fused kernel work?": the two expert linear
// layers with SwiGLU between them and the combine in the forward, and the
// matching backward.  Six variants share the main loop:
//   GATEUP       [g|u] = x_perm . [W_gate;W_up]^T  per expert M block, SwiGLU epilogue
//   DOWN         o = a . W_down^T                   epilogue w*o -> token-major slot
//   DGRAD_DOWN   g' = dy_perm . W_down               dSwiGLU epilogue (dh, w*a, <a,g'>)
//   DGRAD_GATEUP dx = dh . [W_gate;W_up]             epilogue -> token-major slot
//   WGRAD_DOWN   dW_down[e] = dy_perm^T . (w*a)      K = the expert's rows
//   WGRAD_GATEUP [dW_gate;dW_up][e] = dh^T . x_perm   K = the expert's rows
//
// Roles (256 threads): warp 0 lane 0 = TMA producer, warp 1 lane 0 = MMA issuer,
// warp 2 = TMEM allocator, warps 4..7 = epilogue (warp 4+q reads TMEM lanes
// 32q..32q+31, i.e. tile rows 32q..32q+31).  Every wait is bounded: on expiry the
// kernel records MM_MOE_ETIMEOUT in the status word and every role unwinds.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace mmmoe {

constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s

struct GemmParams {
  CUtensorMap tmA;
  CUtensorMap tmB0;
  CUtensorMap tmB1;
  int H, I, E;
  int n_tiles;  // N tiles per M block (grouped kinds) or per expert M row (per-expert kinds)
  int m_tiles;  // M tiles per expert (per-expert kinds)
  int k_iters;  // K iterations per tile (grouped kinds)
  int n_pw;
  int max_tiles;
  const int* meta;
  const int* tile_expert;
  const int* tile_rows;
  const int* pad_off;
  const int* expert_order;
  const int* rowflat;
  const float* w_row;
  uint16_t* out0;
  uint16_t* out1;
  float* outf;
  const uint16_t* aux;
  const uint16_t* aux2;
  DevStatus* status;
};

template <int KIND, int BN_>
struct Cfg {
  static constexpr int BN = BN_;
  static constexpr bool A_MN = KIND >= GEMM_WGRAD_DOWN;
  static constexpr bool B_MN = KIND >= GEMM_DGRAD_DOWN;
  static constexpr bool PER_EXPERT = KIND >= GEMM_WGRAD_DOWN;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN == 256 ? 4 : (BN == 128 ? 6 : 8);
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, BN, A_MN, B_MN);
  static_assert(BN == 64 || BN == 128 || BN == 256, "BN");
};

struct TileInfo {
  int e, mb, m0, n0, k_iters, k_row0;
};

// Decode tile t.  Grouped kinds: t -> (M block of padded routed rows, N tile), N
// fastest.  Per-expert kinds: experts in descending row count, then (M, N) tiles.
template <int KIND, int BN>
__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, int t) {
  TileInfo ti;
  if constexpr (Cfg<KIND, BN>::PER_EXPERT) {
    const int per_e = p.m_tiles * p.n_tiles;
    const int ei = t / per_e;
    const int rem = t - ei * per_e;
    const int mt = rem / p.n_tiles;
    const int nt = rem - mt * p.n_tiles;
    ti.e = __ldg(p.expert_order + ei);
    ti.mb = 0;
    ti.m0 = mt * BM;
    ti.n0 = nt * BN;
    ti.k_row0 = __ldg(p.pad_off + ti.e);
    ti.k_iters = (__ldg(p.pad_off + ti.e + 1) - ti.k_row0) / BK;
  } else {
    const int mb = t / p.n_tiles;
    const int nt = t - mb * p.n_tiles;
    ti.mb = mb;
    ti.e = __ldg(p.tile_expert + mb);
    ti.m0 = mb * BM;
    ti.n0 = nt * (KIND == GEMM_GATEUP ? BN / 2 : BN);
    ti.k_iters = p.k_iters;
    ti.k_row0 = 0;
  }
  return ti;
}

template <int KIND, int BN>
__device__ __forceinline__ int total_tiles(const GemmParams& p) {
  if constexpr (Cfg<KIND, BN>::PER_EXPERT) {
    return p.E * p.m_tiles * p.n_tiles;
  } else {
    int nt = __ldg(p.meta + META_NUM_TILES);
    nt = min(nt, p.max_tiles);
    return nt * p.n_tiles;
  }
}

__device__ __forceinline__ void record_timeout(GemmParams const& p, volatile int* abort,
                                               int detail) {
  *abort = 1;
  if (atomicCAS(&p.status->code, 0, MM_MOE_ETIMEOUT) == 0) p.status->detail = detail;
}

// ------------------------------------------------------------------ epilogue helpers
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void store32(uint16_t* dst, const float (&v)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    d[q] = make_uint4(pack2(v[8 * q], v[8 * q + 1]), pack2(v[8 * q + 2], v[8 * q + 3]),
                      pack2(v[8 * q + 4], v[8 * q + 5]), pack2(v[8 * q + 6], v[8 * q + 7]));
}

__device__ __forceinline__ void store32_zero(uint16_t* dst) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) d[q] = make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ void load32_bf16(const uint16_t* src, float (&v)[32]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 w = __ldg(s + q);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[8 * q + 2 * i] = __uint_as_float(ww[i] << 16);
      v[8 * q + 2 * i + 1] = __uint_as_float(ww[i] & 0xFFFF0000u);
    }
  }
}

__device__ __forceinline__ void as_float(const uint32_t (&r)[32], float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ float sigmoidf_(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }

// Epilogue of one tile for one thread = one accumulator row.
template <int KIND, int BN>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, const TileInfo& ti, int row,
                                              uint32_t tbase) {
  const int64_t I = p.I, H = p.H;
  if constexpr (KIND == GEMM_GATEUP) {
    constexpr int HALF = BN / 2;
    const int64_t pr = ti.m0 + row;
    uint16_t* hrow = p.out0 + pr * 2 * I + ti.n0;
    uint16_t* arow = p.out1 + pr * I + ti.n0;
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
      store32(hrow + c, g);
      store32(hrow + I + c, u);
      store32(arow + c, a);
    }
  } else if constexpr (KIND == GEMM_DOWN || KIND == GEMM_DGRAD_GATEUP) {
    const int pr = ti.m0 + row;
    const bool valid = row < __ldg(p.tile_rows + ti.mb);
    uint16_t* dst = nullptr;
    float w = 1.0f;
    if (valid) {
      const int64_t f = __ldg(p.rowflat + pr);
      dst = p.out0 + f * H + ti.n0;
      if (KIND == GEMM_DOWN) w = __ldg(p.w_row + pr);
    }
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t r[32];
      ptx::tmem_ld32(tbase + c, r);
      ptx::tmem_wait_ld(r);
      float v[32];
      as_float(r, v);
      if (KIND == GEMM_DOWN) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= w;
      }
      if (valid) store32(dst + c, v);
    }
  } else if constexpr (KIND == GEMM_DGRAD_DOWN) {
    const int64_t pr = ti.m0 + row;
    const float w = __ldg(p.w_row + pr);
    const uint16_t* hrow = p.aux + pr * 2 * I + ti.n0;
    const uint16_t* arow = p.aux2 + pr * I + ti.n0;
    uint16_t* dhrow = p.out0 + pr * 2 * I + ti.n0;
    uint16_t* awrow = p.out1 + pr * I + ti.n0;
    float dot = 0.f;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t r[32];
      ptx::tmem_ld32(tbase + c, r);
      float g[32], u[32], av[32];
      load32_bf16(hrow + c, g);
      load32_bf16(hrow + I + c, u);
      load32_bf16(arow + c, av);
      ptx::tmem_wait_ld(r);
      float gp[32];
      as_float(r, gp);
      float dg[32], du[32], aw[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float s = sigmoidf_(g[i]);
        const float sg = g[i] * s;               // silu(g)
        const float a = av[i];                   // the forward's a (from fp32 g, u)
        dot += a * gp[i];
        const float da = w * gp[i];
        dg[i] = da * u[i] * s * (1.0f + g[i] * (1.0f - s));
        du[i] = da * sg;
        aw[i] = w * a;
      }
      store32(dhrow + c, dg);
      store32(dhrow + I + c, du);
      store32(awrow + c, aw);
    }
    p.outf[pr * p.n_pw + ti.n0 / BN] = dot;
  } else if constexpr (KIND == GEMM_WGRAD_DOWN) {
    uint16_t* dst = p.out0 + (static_cast<int64_t>(ti.e) * H + ti.m0 + row) * I + ti.n0;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t r[32];
      ptx::tmem_ld32(tbase + c, r);
      ptx::tmem_wait_ld(r);
      float v[32];
      as_float(r, v);
      store32(dst + c, v);
    }
  } else {  // GEMM_WGRAD_GATEUP
    const int m = ti.m0 + row;
    uint16_t* dst = (m < I ? p.out0 + (static_cast<int64_t>(ti.e) * I + m) * H
                           : p.out1 + (static_cast<int64_t>(ti.e) * I + (m - I)) * H) + ti.n0;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t r[32];
      ptx::tmem_ld32(tbase + c, r);
      ptx::tmem_wait_ld(r);
      float v[32];
      as_float(r, v);
      store32(dst + c, v);
    }
  }
}

// Zero tile of a per-expert GEMM whose expert has no rows (K = 0).
template <int KIND, int BN>
__device__ __forceinline__ void zero_tile(const GemmParams& p, const TileInfo& ti, int row) {
  const int64_t I = p.I, H = p.H;
  uint16_t* dst;
  if constexpr (KIND == GEMM_WGRAD_DOWN) {
    dst = p.out0 + (static_cast<int64_t>(ti.e) * H + ti.m0 + row) * I + ti.n0;
  } else {
    const int m = ti.m0 + row;
    dst = (m < I ? p.out0 + (static_cast<int64_t>(ti.e) * I + m) * H
                 : p.out1 + (static_cast<int64_t>(ti.e) * I + (m - I)) * H) + ti.n0;
  }
#pragma unroll 1
  for (int c = 0; c < BN; c += 32) store32_zero(dst + c);
}

// ------------------------------------------------------------------ producer loads
template <int KIND, int BN>
__device__ __forceinline__ void issue_loads(const GemmParams& p, const TileInfo& ti, int kb,
                                            uint8_t* sa, uint8_t* sb, uint64_t* bar) {
  const int k0 = kb * BK;
  if constexpr (KIND == GEMM_GATEUP) {
    ptx::tma_load_2d(sa, &p.tmA, bar, k0, ti.m0);
    ptx::tma_load_2d(sb, &p.tmB0, bar, k0, ti.e * p.I + ti.n0);
    ptx::tma_load_2d(sb + (BN / 2) * 128, &p.tmB1, bar, k0, ti.e * p.I + ti.n0);
  } else if constexpr (KIND == GEMM_DOWN) {
    ptx::tma_load_2d(sa, &p.tmA, bar, k0, ti.m0);
    ptx::tma_load_2d(sb, &p.tmB0, bar, k0, ti.e * p.H + ti.n0);
  } else if constexpr (KIND == GEMM_DGRAD_DOWN) {
    ptx::tma_load_2d(sa, &p.tmA, bar, k0, ti.m0);
#pragma unroll
    for (int c = 0; c < BN / 64; ++c)
      ptx::tma_load_2d(sb + c * 8192, &p.tmB0, bar, ti.n0 + c * 64, ti.e * p.H + k0);
  } else if constexpr (KIND == GEMM_DGRAD_GATEUP) {
    ptx::tma_load_2d(sa, &p.tmA, bar, k0, ti.m0);
    const bool gate = k0 < p.I;
    const CUtensorMap* m = gate ? &p.tmB0 : &p.tmB1;
    const int krow = ti.e * p.I + (gate ? k0 : k0 - p.I);
#pragma unroll
    for (int c = 0; c < BN / 64; ++c) ptx::tma_load_2d(sb + c * 8192, m, bar, ti.n0 + c * 64, krow);
  } else {  // per-expert weight gradients: both operands M/N-major, K = routed rows
    const int krow = ti.k_row0 + k0;
#pragma unroll
    for (int c = 0; c < BM / 64; ++c)
      ptx::tma_load_2d(sa + c * 8192, &p.tmA, bar, ti.m0 + c * 64, krow);
#pragma unroll
    for (int c = 0; c < BN / 64; ++c)
      ptx::tma_load_2d(sb + c * 8192, &p.tmB0, bar, ti.n0 + c * 64, krow);
  }
}

// ------------------------------------------------------------------ the kernel
template <int KIND, int BN>
__global__ void __launch_bounds__(256, 1) moe_gemm_kernel(const __grid_constant__ GemmParams p) {
  using C = Cfg<KIND, BN>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::STAGES];
  __shared__ __align__(8) uint64_t empty_bar[C::STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(&full_bar[s], 1);
      ptx::mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull_bar[a], 1);
      ptx::mbar_init(&tempty_bar[a], 4);
    }
    ptx::mbar_init(&drain_bar, 1);
    s_abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&p.tmA);
    ptx::prefetch_tmap(&p.tmB0);
    if (KIND == GEMM_GATEUP || KIND == GEMM_DGRAD_GATEUP) ptx::prefetch_tmap(&p.tmB1);
  }
  if (warp == 2) {
    ptx::tmem_alloc(&s_tmem_base, C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  volatile int* abort = &s_abort;
  const int total = total_tiles<KIND, BN>(p);

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- producer
    int stage = 0;
    uint32_t phase = 0;
    int last_parity[C::STAGES];
#pragma unroll
    for (int s = 0; s < C::STAGES; ++s) last_parity[s] = -1;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const TileInfo ti = decode_tile<KIND, BN>(p, t);
      for (int kb = 0; kb < ti.k_iters; ++kb) {
        if (!ptx::mbar_wait(&empty_bar[stage], phase ^ 1u, abort, WAIT_LIMIT_NS)) {
          record_timeout(p, abort, KIND * 16 + 1);
          ok = false;
          break;
        }
        uint8_t* sa = smem + stage * C::STAGE_BYTES;
        ptx::mbar_arrive_expect_tx(&full_bar[stage], C::STAGE_BYTES);
        issue_loads<KIND, BN>(p, ti, kb, sa, sa + C::A_BYTES, &full_bar[stage]);
        last_parity[stage] = static_cast<int>(phase);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // drain: every issued copy has landed before the CTA may exit
    for (int s = 0; s < C::STAGES; ++s) {
      if (last_parity[s] < 0) continue;
      int dummy = 0;
      if (!ptx::mbar_wait(&full_bar[s], static_cast<uint32_t>(last_parity[s]), &dummy,
                          WAIT_LIMIT_NS))
        record_timeout(p, abort, KIND * 16 + 2);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    bool issued = false;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const TileInfo ti = decode_tile<KIND, BN>(p, t);
      if (ti.k_iters == 0) continue;
      if (!ptx::mbar_wait(&tempty_bar[acc], acc_phase ^ 1u, abort, WAIT_LIMIT_NS)) {
        record_timeout(p, abort, KIND * 16 + 3);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
      for (int kb = 0; kb < ti.k_iters; ++kb) {
        if (!ptx::mbar_wait(&full_bar[stage], phase, abort, WAIT_LIMIT_NS)) {
          record_timeout(p, abort, KIND * 16 + 4);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t a_base = ptx::smem_u32(smem + stage * C::STAGE_BYTES);
        const uint32_t b_base = a_base + C::A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t adesc = C::A_MN ? ptx::smem_desc_sw128(a_base + kk * 2048, 8192, 1024)
                                         : ptx::smem_desc_sw128(a_base + kk * 32, 16, 1024);
          const uint64_t bdesc = C::B_MN ? ptx::smem_desc_sw128(b_base + kk * 2048, 8192, 1024)
                                         : ptx::smem_desc_sw128(b_base + kk * 32, 16, 1024);
          ptx::umma_bf16(d_tmem, adesc, bdesc, C::IDESC, (kb | kk) != 0 ? 1u : 0u);
        }
        issued = true;
        ptx::umma_commit(&empty_bar[stage]);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      ptx::umma_commit(&tfull_bar[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (issued) {
      // drain: every issued MMA has completed before TMEM is released
      ptx::umma_commit(&drain_bar);
      int dummy = 0;
      if (!ptx::mbar_wait(&drain_bar, 0, &dummy, WAIT_LIMIT_NS))
        record_timeout(p, abort, KIND * 16 + 5);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp - 4;
    const int row = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const TileInfo ti = decode_tile<KIND, BN>(p, t);
      if (ti.k_iters == 0) {
        if constexpr (C::PER_EXPERT) zero_tile<KIND, BN>(p, ti, row);
        continue;
      }
      int ok = 1;
      if (lane == 0) ok = ptx::mbar_wait(&tfull_bar[acc], acc_phase, abort, WAIT_LIMIT_NS) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) record_timeout(p, abort, KIND * 16 + 6);
        break;
      }
      ptx::tc_fence_after();
      __syncwarp();
      const uint32_t tbase = tmem_base + static_cast<uint32_t>(acc * BN) +
                             (static_cast<uint32_t>(q * 32) << 16);
      epilogue_tile<KIND, BN>(p, ti, row, tbase);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tempty_bar[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 2) ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
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

// Row-major bf16 matrix [outer, inner] -> 2-D tensor map with a box of
// box_inner x box_outer elements and the 128-byte swizzle.
static bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                     uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int pick_bn(int64_t n) {
  if (n % 256 == 0) return 256;
  if (n % 128 == 0) return 128;
  return 64;
}

template <int KIND, int BN>
static cudaError_t run(const Ctx& c, const GemmParams& p, int grid) {
  using C = Cfg<KIND, BN>;
  cudaError_t e = cudaFuncSetAttribute(moe_gemm_kernel<KIND, BN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  static constexpr int kId[6] = {K_GEMM_GATEUP, K_GEMM_DOWN, K_GEMM_DGRAD_DOWN,
                                 K_GEMM_DGRAD_GATEUP, K_GEMM_WGRAD_DOWN, K_GEMM_WGRAD_GATEUP};
  prof_begin(c, kId[KIND]);
  moe_gemm_kernel<KIND, BN><<<grid, 256, C::SMEM_BYTES, c.stream>>>(p);
  prof_end(c, kId[KIND]);
  return cudaGetLastError();
}

cudaError_t launch_gemm(const Ctx& c, const Layout& L, const GemmArgs& g) {
  GemmParams p;
  memset(&p, 0, sizeof(p));
  const char* saved = g.saved;
  p.H = static_cast<int>(L.H);
  p.I = static_cast<int>(L.I);
  p.E = static_cast<int>(L.E);
  p.n_pw = static_cast<int>(L.n_pw);
  p.max_tiles = static_cast<int>(L.NT);
  p.meta = reinterpret_cast<const int*>(saved + L.meta);
  p.tile_expert = reinterpret_cast<const int*>(saved + L.tile_expert);
  p.tile_rows = reinterpret_cast<const int*>(saved + L.tile_rows);
  p.pad_off = reinterpret_cast<const int*>(saved + L.pad_off);
  p.expert_order = reinterpret_cast<const int*>(saved + L.expert_order);
  p.rowflat = reinterpret_cast<const int*>(saved + L.rowflat);
  p.w_row = reinterpret_cast<const float*>(saved + L.w_row);
  p.out0 = g.out0;
  p.out1 = g.out1;
  p.outf = g.outf;
  p.aux = g.aux;
  p.aux2 = g.aux2;
  p.status = reinterpret_cast<DevStatus*>(g.scratch + L.status);
  const uint64_t Rp = static_cast<uint64_t>(L.Rp), H = L.H, I = L.I, E = L.E;
  bool ok = true;
  int bn = 0;
  int64_t max_total = 0;
  switch (g.kind) {
    case GEMM_GATEUP:
      bn = (L.I % 128 == 0) ? 256 : 128;
      ok = make_map(&p.tmA, g.A, H, Rp, 64, BM) && make_map(&p.tmB0, g.B0, H, E * I, 64, bn / 2) &&
           make_map(&p.tmB1, g.B1, H, E * I, 64, bn / 2);
      p.n_tiles = static_cast<int>(L.I / (bn / 2));
      p.k_iters = static_cast<int>(L.H / BK);
      max_total = L.NT * p.n_tiles;
      break;
    case GEMM_DOWN:
      bn = pick_bn(L.H);
      ok = make_map(&p.tmA, g.A, I, Rp, 64, BM) && make_map(&p.tmB0, g.B0, I, E * H, 64, bn);
      p.n_tiles = static_cast<int>(L.H / bn);
      p.k_iters = static_cast<int>(L.I / BK);
      max_total = L.NT * p.n_tiles;
      break;
    case GEMM_DGRAD_DOWN:
      bn = pick_bn(L.I);
      ok = make_map(&p.tmA, g.A, H, Rp, 64, BM) && make_map(&p.tmB0, g.B0, I, E * H, 64, 64);
      p.n_tiles = static_cast<int>(L.I / bn);
      p.k_iters = static_cast<int>(L.H / BK);
      max_total = L.NT * p.n_tiles;
      break;
    case GEMM_DGRAD_GATEUP:
      bn = pick_bn(L.H);
      ok = make_map(&p.tmA, g.A, 2 * I, Rp, 64, BM) && make_map(&p.tmB0, g.B0, H, E * I, 64, 64) &&
           make_map(&p.tmB1, g.B1, H, E * I, 64, 64);
      p.n_tiles = static_cast<int>(L.H / bn);
      p.k_iters = static_cast<int>(2 * L.I / BK);
      max_total = L.NT * p.n_tiles;
      break;
    case GEMM_WGRAD_DOWN:
      bn = pick_bn(L.I);
      ok = make_map(&p.tmA, g.A, H, Rp, 64, 64) && make_map(&p.tmB0, g.B0, I, Rp, 64, 64);
      p.m_tiles = static_cast<int>(L.H / BM);
      p.n_tiles = static_cast<int>(L.I / bn);
      max_total = L.E * p.m_tiles * p.n_tiles;
      break;
    case GEMM_WGRAD_GATEUP:
      bn = pick_bn(L.H);
      ok = make_map(&p.tmA, g.A, 2 * I, Rp, 64, 64) && make_map(&p.tmB0, g.B0, H, Rp, 64, 64);
      p.m_tiles = static_cast<int>(2 * L.I / BM);
      p.n_tiles = static_cast<int>(L.H / bn);
      max_total = L.E * p.m_tiles * p.n_tiles;
      break;
    default:
      return cudaErrorInvalidValue;
  }
  if (!ok) return cudaErrorInvalidValue;
  const int grid = static_cast<int>(std::min<int64_t>(c.num_sms, std::max<int64_t>(max_total, 1)));
#define MMMOE_RUN(K, B) \
  if (g.kind == K && bn == B) return run<K, B>(c, p, grid);
  MMMOE_RUN(GEMM_GATEUP, 256)
  MMMOE_RUN(GEMM_GATEUP, 128)
  MMMOE_RUN(GEMM_DOWN, 256)
  MMMOE_RUN(GEMM_DOWN, 128)
  MMMOE_RUN(GEMM_DGRAD_DOWN, 256)
  MMMOE_RUN(GEMM_DGRAD_DOWN, 128)
  MMMOE_RUN(GEMM_DGRAD_DOWN, 64)
  MMMOE_RUN(GEMM_DGRAD_GATEUP, 256)
  MMMOE_RUN(GEMM_DGRAD_GATEUP, 128)
  MMMOE_RUN(GEMM_WGRAD_DOWN, 256)
  MMMOE_RUN(GEMM_WGRAD_DOWN, 128)
  MMMOE_RUN(GEMM_WGRAD_DOWN, 64)
  MMMOE_RUN(GEMM_WGRAD_GATEUP, 256)
  MMMOE_RUN(GEMM_WGRAD_GATEUP, 128)
#undef MMMOE_RUN
  return cudaErrorInvalidValue;
}

}  // namespace mmmoe

// internal.h -- types shared by the translation units of the library (not part of
// the public ABI): the workspace layout and the host-side kernel launchers.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/mm_moe.h"

namespace mmmoe {

constexpr int BM = 128;            // rows of an M tile (routed rows or output rows)
constexpr int BK = 64;             // K elements per pipeline stage (128 bytes of bf16)
constexpr int ROUTE_CHUNK = 2048;  // flat (token, slot) indices per routing block
constexpr int ROUTE_THREADS = 256;
constexpr int MAX_E = 1024;

// Device status word (first bytes of scratch).
struct DevStatus {
  int code;    // mm_moe_status
  int detail;  // first bad flat index / id of the kernel whose wait ran out
};

// Byte offsets of every region inside `saved` and `scratch`.  Every region starts
// on a 1024-byte boundary.  "Padded rows": each expert's routed rows start on a
// multiple of `pad` and its tail up to the next multiple is zero, so that M tiles
// (of one SM or of an SM pair) never straddle two experts and the token-axis K loop
// of the weight-gradient GEMMs reads zeros past an expert's last row.
struct Layout {
  int64_t T, H, I, E, k, R;
  int64_t pad;     // each expert's rows are padded to a multiple of this: BM, or 2*BM
                   // when the GEMMs run on SM pairs
  int64_t Rp;      // capacity of the padded row space: (ceil(R/pad) + E) * pad
  int64_t NT;      // capacity in M tiles: Rp / BM
  int64_t nblk;    // routing blocks: ceil(R / ROUTE_CHUNK)
  int64_t n_pw;    // partial dot products per row for dtopk_w (I / BN of the dgrad-down GEMM)
  bool recompute;  // MM_MOE_RECOMPUTE: x_perm, h, a live in scratch, not saved
  bool multicast;  // MM_MOE_MULTICAST: A-multicast clusters of two SM pairs
  // saved (x_perm, h, a: offsets into scratch instead when recompute)
  size_t counts, offsets, pad_off, expert_order, meta, perm, inv, prow, rowflat, tile_expert,
      tile_rows, w_row, x_perm, h, a, saved_bytes;
  // scratch
  size_t status, blk_counts, ys, dy_perm, dh, a_w, pw, dxs, scratch_bytes;
  // scratch, quantised operand copies (set only for the precisions that use them):
  // e4m3 codes [rows, cols] followed by their E8M0 scales, rows * cols / 32 bytes in
  // the mx::sf_offset arrangement (blockwise FP8 weights: the scales in both
  // arrangements, rows as the MMA rows first):
  // forward, blocks along K: x_perm, a, W_gate, W_up, W_down
  size_t q_x, q_a, q_wg, q_wu, q_wd;
  // backward: W_down along H and W_gate, W_up along I (q_wdc, q_wgc, q_wuc; blockwise
  // FP8: the one copy of each weight, read by every GEMM), dy_perm, dh, x_perm along
  // the token axis (q_dyc, q_dhc, q_xc), dh along I (q_dhr) and a_w along tokens
  // (q_awc); the permutation writes dy along H into dy_perm's place.
  // Under a quantised forward that keeps its activations the forward writes the weight
  // copies into `saved` (w_in_saved) and x's token-axis copy over x_perm, so q_xc is
  // unused.
  size_t q_wdc, q_wgc, q_wuc, q_dyc, q_dhc, q_xc, q_dhr, q_awc;
  bool w_in_saved;
  // quantisation of the forward's and the backward's GEMM operands: QS_NONE, QS_MX
  // (MXFP8) or QS_BLOCK (blockwise FP8, whose one 128 x 128-block copy of each weight
  // serves every GEMM: q_wgc, q_wuc, q_wdc, in saved when w_in_saved, else at the
  // front of scratch, w_common)
  int qf, qb;
  bool w_common;
};

enum { QS_NONE = 0, QS_MX = 1, QS_BLOCK = 2 };

// meta[] slots in `saved`
constexpr int META_NUM_TILES = 0;

mm_moe_status make_layout(const mm_moe_shape* s, Layout* L);

// Whether shapes that allow it run their GEMMs on SM pairs (environment variable
// MM_MOE_SM_PAIRS=0 selects single-SM tiles everywhere; default on).
bool sm_pairs_enabled();

// Width of the N tile each GEMM uses for an output dimension of n columns.
int pick_bn(int64_t n);

// ------------------------------------------------------------------ launchers
// Each returns cudaSuccess or the launch error; `launches` is incremented per kernel.
struct Ctx {
  cudaStream_t stream;
  int num_sms;
  int* launches;
};

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation (launch_k; the GEMMs in gemm.cuh), so that it may
// start, and run the part of its prologue that touches no global memory, while the
// kernel before it in the stream drains.  Each kernel calls pdl_wait() before its
// first global access, which returns once the kernel before it has completed and
// its writes are visible, and then pdl_trigger(), which lets the next kernel start
// launching.  (A kernel launched without the attribute passes both at once.)
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_k(cudaStream_t st, void (*kern)(KArgs...), dim3 grid, dim3 block,
                     size_t smem, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}
#endif

// Kernel ids (per-kernel timing and launch accounting).
enum KernelId {
  K_ROUTE_COUNT = 0,
  K_ROUTE_SCAN,
  K_ROUTE_PLACE,
  K_PERMUTE_X,
  K_GEMM_GATEUP,
  K_GEMM_DOWN,
  K_COMBINE,
  K_PERMUTE_DY,
  K_GEMM_DGRAD_DOWN,
  K_GEMM_DGRAD_GATEUP,
  K_UNPERMUTE,
  K_GEMM_WGRAD_DOWN,
  K_GEMM_WGRAD_GATEUP,
  K_GEMM_WGRAD,
  K_MX_QDQ_ROWS,
  K_MX_QDQ_COLS,
  K_FB_ROWS,
  K_FB_COLS,
  K_FB_TILES,
  K_FBQ_ROWS,
  K_FBQ_COLS,
  K_FBQ_TILES,
  K_MXQ_ROWS,
  K_MXQ_COLS,
  K_DENSE_NT,
  K_DENSE_NN,
  K_DENSE_TN,
  K_ROUTER_TOPK,
  K_ROUTER_DLOGITS,
  K_COUNT
};

// Bracket one kernel launch: optional timing events, and the launch counter.
void prof_begin(const Ctx& c, int id);
void prof_end(const Ctx& c, int id);

cudaError_t launch_route(const Ctx& c, const Layout& L, const int32_t* topk_idx,
                         const float* topk_w, char* saved, char* scratch);
// Every buffer the three routing kernels touch, as explicit device pointers.
struct RouteBufs {
  DevStatus* status;
  int* blk_counts;  // [ceil(R / ROUTE_CHUNK) * E]
  int* counts;      // [E]
  int* offsets;     // [E + 1]
  int* pad_off;     // [E + 1]
  int* expert_order;  // [E]
  int* tile_expert;   // [NT]
  int* tile_rows;     // [NT]
  int* meta;          // [16]
  int* perm;          // [R]
  int* inv;           // [R]
  int* prow;          // [R]
  int* rowflat;       // [Rp]
  float* w_row;       // [Rp]
};
cudaError_t launch_route_to(const Ctx& c, int R, int E, int pad, const int32_t* topk_idx,
                            const float* topk_w, const RouteBufs& b);
// dst = src's token rows in the padded expert-grouped order, padding rows zero; with
// quant = QS_MX / QS_BLOCK each row is quantised along its columns on the way (32- /
// 128-element blocks), once per token before its k copies are stored: dst receives
// the rows' e4m3 codes ([Rp, H] bytes) and `sf` their scale codes (mx::sf_offset over
// the Rp padded rows).
cudaError_t launch_permute(const Ctx& c, const Layout& L, const uint16_t* src, void* dst,
                           const char* saved, float* w_row_out, int kernel_id, char* scratch,
                           int quant = 0, uint8_t* sf = nullptr);
cudaError_t launch_combine(const Ctx& c, const Layout& L, const uint16_t* slots,
                           const char* saved, uint16_t* out);
cudaError_t launch_unpermute(const Ctx& c, const Layout& L, const uint16_t* slots,
                             const char* saved, const float* pw, uint16_t* dx, float* dtopk_w);

// Rows of the padded expert-grouped space read straight from a token-major [T, cols]
// tensor: padded row pr is token rowflat[pr] / k, or a zero row when pr is padding (its
// place in its BM-row block at or past tile_rows[pr / BM]).
struct RowGather {
  const int* rowflat;
  const int* tile_rows;
  int k;
};

// Source row of padded row pr: its index in `in`, or -1 for a zero row.  Both loads
// are issued together; rowflat of a padding row (never written) is read and dropped.
__device__ __forceinline__ int gather_src(int64_t pr, const RowGather& g) {
  if (g.rowflat == nullptr) return static_cast<int>(pr);
  const int64_t mb = pr / BM;
  const int f = __ldg(g.rowflat + pr);
  const int valid = __ldg(g.tile_rows + mb);
  return pr - mb * BM < valid ? f / g.k : -1;
}

// MXFP8 quantise-dequantise of a bf16 [rows, cols] tensor in blocks of 32 elements,
// along each row (along_rows) or down each column; the result is written as bf16.
// With `meta` (device) non-null only the first meta[META_NUM_TILES] * BM rows are
// processed (the padded routed rows that are in use).  Down columns, a non-null
// out_rows also receives the blocks along rows from the same read, and a gather with a
// non-null rowflat reads the rows from a token-major `in` instead.  out and out_rows
// may each equal in (every element is read once, by the thread that writes it).
cudaError_t launch_mx_qdq(const Ctx& c, const uint16_t* in, uint16_t* out, int64_t rows,
                          int64_t cols, bool along_rows, const int* meta,
                          uint16_t* out_rows = nullptr, RowGather gather = RowGather{});

// MXFP8 quantisation into e4m3 codes and E8M0 scales (the block-scaled tensor-core
// operand format; scale arrangement mx::sf_offset).  in: bf16 [rows, cols], rows and
// cols multiples of 128.  along_rows: blocks of 32 along each row (the MMA rows are
// the tensor's rows, mn_blocks = rows / 128); else blocks of 32 rows down each column
// (the MMA rows are the columns, mn_blocks = cols / 128), optionally with the row
// blocks of the same read too (codes_rows / sf_rows), and with a gather the rows come
// from a token-major `in`.  `meta` (device, may be null) limits the rows processed to
// meta[META_NUM_TILES] * BM (the padded routed rows in use); the scale arrangement
// still spans all `rows`.
struct MxqArgs {
  const uint16_t* in;
  uint8_t* codes;
  uint8_t* sf;
  int64_t rows, cols;
  bool along_rows;
  const int* meta;
  uint8_t* codes_rows;
  uint8_t* sf_rows;
  RowGather gather;
  DevStatus* status;  // device status word for a copy that never lands (may be null)
};
cudaError_t launch_mxq(const Ctx& c, const MxqArgs& a);

// Blockwise FP8 quantise-dequantise of a bf16 [rows, cols] tensor (power-of-two scale
// 2^ceil(log2(amax / 448)) per block), written as bf16: 128-element blocks along each
// row (FB_ROWS), down each column (FB_COLS; a non-null out_rows also receives the row
// blocks of the same read; `meta` and `gather` as for launch_mx_qdq), or 128 x 128
// tiles (FB_TILES).  out / out_rows may equal in.
enum { FB_ROWS = 0, FB_COLS = 1, FB_TILES = 2 };
// Blockwise FP8 in the form the block-scaled tensor cores read: e4m3 codes ([rows, cols]
// bytes) and E8M0 scale codes (mx::sf_offset), each 128-element block's scale repeated
// over its four 32-element scale blocks.  FB_ROWS: 128-blocks along each row (scales
// over rows / 128 row blocks); FB_COLS: 128-row blocks down each column (scales over
// cols / 128 column blocks), with codes_rows non-null also the row blocks (scales over
// rows / 128 row blocks to sf_rows), rows optionally gathered; FB_TILES: 128 x 128 weight
// tiles, one copy of the codes and the scales in both arrangements (sf: the MMA rows
// are the matrix rows; sf_mn: the MMA rows are the columns).  `meta` (device, optional)
// limits FB_ROWS / FB_COLS to the padded rows in use.
struct FbqArgs {
  const uint16_t* in;
  uint8_t* codes;
  uint8_t* sf;
  uint8_t* sf_mn;
  uint8_t* codes_rows;
  uint8_t* sf_rows;
  int64_t rows, cols;
  int layout;
  const int* meta;
  RowGather gather;
};
cudaError_t launch_fbq(const Ctx& c, const FbqArgs& a);
cudaError_t launch_fb_qdq(const Ctx& c, const uint16_t* in, uint16_t* out, int64_t rows,
                          int64_t cols, int layout, const int* meta, uint16_t* out_rows,
                          RowGather gather = RowGather{});

enum GemmKind {
  GEMM_GATEUP = 0,        // x_perm . [W_gate|W_up]^T  -> SwiGLU epilogue (h, a)
  GEMM_DOWN = 1,          // a . W_down^T              -> w * o, expert-grouped rows
  GEMM_DGRAD_DOWN = 2,    // dy_perm . W_down          -> dSwiGLU epilogue (dh, a_w, pw)
  GEMM_DGRAD_GATEUP = 3,  // dh . [W_gate;W_up]        -> dx, expert-grouped rows
  GEMM_WGRAD_DOWN = 4,    // dy_perm^T . a_w per expert -> dW_down
  GEMM_WGRAD_GATEUP = 5,  // dh^T . x_perm per expert   -> dW_gate, dW_up
  GEMM_WGRAD_BOTH = 6,    // both weight gradients in one launch, tiles ordered by expert
  // dense products (the router's; single-SM tiles, bf16 operands, any M, N, K):
  GEMM_DENSE_NT = 7,      // C [M, N] fp32  = A [M, K] . B [N, K]^T
  GEMM_DENSE_NN = 8,      // C [M, N] bf16 += A [M, K] . B [K, N]   (read-modify-write)
  GEMM_DENSE_TN = 9,      // C [M, N] bf16  = A [K, M]^T . B [K, N]
};

// A dense product of kind GEMM_DENSE_* (row-major bf16 operands; every inner dimension
// a multiple of 8, so that rows are 16-byte multiples).  Returns cudaErrorInvalidValue
// for unsupported sizes.
cudaError_t launch_dense(const Ctx& c, int kind, const uint16_t* A, const uint16_t* B, void* C,
                         int64_t M, int64_t N, int64_t K);

struct GemmArgs {
  int kind;
  // MXFP8 operands: e4m3 codes and E8M0 scales (mx::sf_offset) on the block-scaled
  // tensor cores; else bf16 operands
  bool fp8;
  // operands (device): bf16 tensors, or with fp8 their codes
  const void* A;    // base of the A operand tensor
  const void* B0;   // first B tensor
  const void* B1;   // second B tensor (W_up) or nullptr
  const uint8_t* sA;   // fp8: scales of A, B0, B1
  const uint8_t* sB0;
  const uint8_t* sB1;
  // epilogue (device)
  uint16_t* out0;
  uint16_t* out1;
  float* outf;
  const uint16_t* aux;   // h = [g | u] for the dSwiGLU epilogue
  const uint16_t* aux2;  // a = silu(g) * u saved by the forward
  // GEMM_WGRAD_BOTH: A, B0, out0, out1 as GEMM_WGRAD_GATEUP; A2, B2 (sA2, sB2), out2 as
  // the A, B0, out0 of GEMM_WGRAD_DOWN
  const void* A2;
  const void* B2;
  const uint8_t* sA2;
  const uint8_t* sB2;
  uint16_t* out2;
  const char* saved;
  char* scratch;
  // fp8 gate/up: the epilogue also writes a in MXFP8 along I (codes [Rp, I] and
  // scales) for the down projection; null: not written
  uint8_t* q_codes;
  uint8_t* q_sf;
};

cudaError_t launch_gemm(const Ctx& c, const Layout& L, const GemmArgs& g);
// whether GEMM_WGRAD_BOTH serves this layout (both weight gradients tile N alike)
bool wgrad_both_ok(const Layout& L);

}  // namespace mmmoe

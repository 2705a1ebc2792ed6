// mm_moe.cu -- the C ABI: argument validation, workspace layout and the launch
// sequences of the forward and backward passes (declared in include/mm_moe.h).
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "internal.h"

namespace mmmoe {

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool sm_pairs_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("MM_MOE_SM_PAIRS");
    return !(v != nullptr && v[0] == '0');
  }();
  return on;
}

// Bytes of one quantised copy of a [rows, cols] operand: e4m3 codes (rows * cols bytes)
// followed by the E8M0 scales (one per 32 elements; blockwise FP8 repeats each
// 128-block's scale four times) -- the form the block-scaled tensor cores read.
static size_t qcopy_bytes(size_t rows, size_t cols) { return rows * cols + rows * cols / 32; }

// Bytes of the backward's (blockwise: the only) copy of a weight: MXFP8 quantises it
// along its other axis (one copy); blockwise FP8's 128 x 128 blocks give the same codes
// either way, followed by the scales in both arrangements (rows, then columns as the
// MMA rows).
static size_t wcopy_bytes(int qs, size_t rows, size_t cols) {
  return qs == QS_BLOCK ? rows * cols + 2 * (rows * cols / 32) : qcopy_bytes(rows, cols);
}

mm_moe_status make_layout(const mm_moe_shape* s, Layout* L) {
  if (s == nullptr || L == nullptr) return MM_MOE_EINVAL;
  *L = Layout{};  // offsets a mode does not use stay 0
  if (s->T < 1 || s->H < 1 || s->I < 1 || s->E < 1 || s->k < 1) return MM_MOE_EINVAL;
  if (s->k > s->E || s->E > MAX_E) return MM_MOE_EINVAL;
  if (s->H % 128 != 0 || s->I % 64 != 0) return MM_MOE_EINVAL;
  if ((s->flags & ~(MM_MOE_RECOMPUTE | MM_MOE_MULTICAST)) != 0) return MM_MOE_EINVAL;
  if (s->prec < MM_MOE_BF16 || s->prec > MM_MOE_FP8_BLOCK) return MM_MOE_EINVAL;
  // blockwise FP8: 128 x 128 weight blocks; MXFP8 (both modes): 128-element K steps of
  // the block-scaled tensor cores over I and 2I
  if (s->prec != MM_MOE_BF16 && s->I % 128 != 0) return MM_MOE_EINVAL;
  if (s->T > (int64_t{1} << 31) / s->k) return MM_MOE_EINVAL;
  L->T = s->T;
  L->H = s->H;
  L->I = s->I;
  L->E = s->E;
  L->k = s->k;
  L->R = s->T * s->k;
  // SM-pair GEMM tiles (M = 256, N = 256) need H % 256 == 0 and I % 128 == 0
  L->pad = (s->H % 256 == 0 && s->I % 128 == 0 && sm_pairs_enabled()) ? 2 * BM : BM;
  L->Rp = ((L->R + L->pad - 1) / L->pad + L->E) * L->pad;
  L->NT = L->Rp / BM;
  if (L->Rp >= (int64_t{1} << 31)) return MM_MOE_EINVAL;
  L->recompute = (s->flags & MM_MOE_RECOMPUTE) != 0;
  L->multicast = (s->flags & MM_MOE_MULTICAST) != 0;
  L->qf = s->prec == MM_MOE_MXFP8 ? QS_MX : s->prec == MM_MOE_FP8_BLOCK ? QS_BLOCK : QS_NONE;
  L->qb = s->prec == MM_MOE_BF16 ? QS_NONE : s->prec == MM_MOE_FP8_BLOCK ? QS_BLOCK : QS_MX;
  L->nblk = (L->R + ROUTE_CHUNK - 1) / ROUTE_CHUNK;
  // partial sums of dtopk_w per row: one per N tile of the dgrad-down GEMM, two when
  // its FP8 tiles (256 wide) split their columns between two epilogue warps
  L->n_pw = L->I / pick_bn(L->I) * ((L->qb != QS_NONE && pick_bn(L->I) == 256) ? 2 : 1);
  const size_t A = 1024;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, A);
    return at;
  };
  const size_t E = static_cast<size_t>(L->E), R = static_cast<size_t>(L->R),
               Rp = static_cast<size_t>(L->Rp), NT = static_cast<size_t>(L->NT),
               H = static_cast<size_t>(L->H), I = static_cast<size_t>(L->I);
  // saved
  L->counts = take(4 * E);
  L->offsets = take(4 * (E + 1));
  L->pad_off = take(4 * (E + 1));
  L->expert_order = take(4 * E);
  L->meta = take(4 * 16);
  L->perm = take(4 * R);
  L->inv = take(4 * R);
  L->prow = take(4 * R);
  L->rowflat = take(4 * Rp);
  L->tile_expert = take(4 * NT);
  L->tile_rows = take(4 * NT);
  L->w_row = take(4 * Rp);
  if (!L->recompute) {
    L->x_perm = take(2 * Rp * H);  // (a quantised forward keeps x along tokens here)
    L->h = take(2 * Rp * 2 * I);
    L->a = take(2 * Rp * I);
  }
  // a quantised forward that keeps its activations also makes the backward's
  // weight copies (MXFP8: the forward's two-way passes; blockwise: the one copy)
  L->w_in_saved = L->qf != QS_NONE && !L->recompute;
  L->w_common = L->qf == QS_BLOCK && L->recompute;
  L->q_wdc = L->q_wgc = L->q_wuc = 0;
  if (L->w_in_saved) {
    const size_t W = wcopy_bytes(L->qf, E * I, H);
    L->q_wdc = take(W);
    L->q_wgc = take(W);
    L->q_wuc = take(W);
  }
  L->saved_bytes = o;
  // scratch: status and routing blocks, then the forward and backward regions overlaid
  o = 0;
  L->status = take(256);
  L->blk_counts = take(4 * static_cast<size_t>(L->nblk) * E);
  if (L->recompute) {  // live through the forward and the backward's recompute
    // (a quantised forward permutes x straight into its quantised copy q_x and the
    // backward gathers x's token-axis blocks from x: no x_perm; its offset is then
    // never dereferenced)
    if (L->qf == QS_NONE) L->x_perm = take(2 * Rp * H);
    L->h = take(2 * Rp * 2 * I);
    L->a = take(2 * Rp * I);
  }
  if (L->w_common) {  // blockwise weights under recompute: made by each pass, used by all
    const size_t W = wcopy_bytes(QS_BLOCK, E * I, H);
    L->q_wdc = take(W);
    L->q_wgc = take(W);
    L->q_wuc = take(W);
  }
  const size_t common = o;
  L->ys = take(2 * Rp * H);
  // quantised operand copies of the forward
  L->q_x = L->q_a = L->q_wg = L->q_wu = L->q_wd = 0;
  if (L->qf != QS_NONE) {
    L->q_x = take(qcopy_bytes(Rp, H));
    L->q_a = take(qcopy_bytes(Rp, I));
  }
  if (L->qf == QS_MX) {  // the forward's MXFP8 weights (blocks along their forward K)
    const size_t W = qcopy_bytes(E * I, H);
    L->q_wg = take(W);
    L->q_wu = take(W);
    L->q_wd = take(W);
  }
  const size_t fwd_end = o;
  o = common;
  L->dy_perm = take(2 * Rp * H);  // (MXFP8: dy along H, codes and scales)
  L->dh = take(2 * Rp * 2 * I);
  L->a_w = take(2 * Rp * I);
  L->pw = take(4 * Rp * static_cast<size_t>(L->n_pw));
  L->dxs = take(2 * Rp * H);
  L->q_dyc = L->q_dhc = L->q_xc = L->q_dhr = L->q_awc = 0;
  if (L->qb != QS_NONE && !L->w_in_saved) {  // left to the backward
    if (!L->w_common) {
      const size_t W = wcopy_bytes(L->qb, E * I, H);
      L->q_wdc = take(W);
      L->q_wgc = take(W);
      L->q_wuc = take(W);
    }
    L->q_xc = take(qcopy_bytes(Rp, H));
  }
  if (L->qb != QS_NONE) {
    L->q_dyc = take(qcopy_bytes(Rp, H));
    L->q_dhc = take(qcopy_bytes(Rp, 2 * I));
    L->q_dhr = take(qcopy_bytes(Rp, 2 * I));
    L->q_awc = take(qcopy_bytes(Rp, I));
  }
  L->scratch_bytes = o > fwd_end ? o : fwd_end;
  return MM_MOE_OK;
}

struct DevInfo {
  int sms = 0;
  mm_moe_status st = MM_MOE_ECUDA;
};

static mm_moe_status device_info(DevInfo* out) {
  static std::mutex mu;
  static DevInfo cache[64];
  static bool have[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MM_MOE_ECUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!have[dev]) {
    DevInfo d;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      return MM_MOE_ECUDA;
    }
    d.st = (major == 10 && minor == 3) ? MM_MOE_OK : MM_MOE_ENOTSUP;
    cache[dev] = d;
    have[dev] = true;
  }
  *out = cache[dev];
  return out->st;
}

static bool aligned(const void* p, uintptr_t a) {
  return p != nullptr && (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

static thread_local int g_last_launches = 0;

// A second stream (and a fork/join event pair) per device and host thread, so that
// bandwidth-bound kernels can run beside independent tensor-core kernels of the same
// call.  Created on first use; never destroyed (they live as long as the thread).
constexpr int SIDE_MARKS = 4;  // points of the side stream the caller's stream can wait for
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  cudaEvent_t mark[SIDE_MARKS] = {};
};

static bool side_stream(SideStream* out) {
  static thread_local SideStream per_dev[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  SideStream& ss = per_dev[dev];
  if (ss.s == nullptr) {
    if (cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess)
      return false;
    for (int i = 0; i < SIDE_MARKS; ++i)
      if (cudaEventCreateWithFlags(&ss.mark[i], cudaEventDisableTiming) != cudaSuccess)
        return false;
  }
  *out = ss;
  return true;
}

// A fork of the caller's stream onto the side stream that is joined back on every
// return: join() on the normal path, the destructor on an error return after the
// fork, so that no path leaves forked work unordered before later work on the
// caller's stream (or an unjoined fork in a stream capture).  In between, the side
// stream can be made to wait for the caller's stream so far (after_main), and the
// caller's stream for a marked point of the side stream (mark, main_waits).
class Fork {
 public:
  Fork() = default;
  Fork(const Fork&) = delete;
  Fork& operator=(const Fork&) = delete;
  ~Fork() { (void)join(); }
  // Returns false when the side stream or the fork could not be made.
  bool open(cudaStream_t main) {
    if (!side_stream(&ss_)) return false;
    main_ = main;
    if (cudaEventRecord(ss_.fork, main) != cudaSuccess) return false;
    if (cudaStreamWaitEvent(ss_.s, ss_.fork, 0) != cudaSuccess) return false;
    open_ = true;
    return true;
  }
  cudaStream_t side() const { return ss_.s; }
  // later side work runs after the caller's stream's work enqueued so far
  cudaError_t after_main() {
    cudaError_t e = cudaEventRecord(ss_.fork, main_);
    return e == cudaSuccess ? cudaStreamWaitEvent(ss_.s, ss_.fork, 0) : e;
  }
  // the side stream's work enqueued so far, as a mark for main_waits (-1: none left)
  int mark() {
    if (n_marks_ == SIDE_MARKS || cudaEventRecord(ss_.mark[n_marks_], ss_.s) != cudaSuccess)
      return -1;
    return n_marks_++;
  }
  cudaError_t main_waits(int m) {
    if (m < 0 || m >= n_marks_) return cudaErrorInvalidValue;
    return cudaStreamWaitEvent(main_, ss_.mark[m], 0);
  }
  cudaError_t join() {
    if (!open_) return cudaSuccess;
    open_ = false;
    cudaError_t e = cudaEventRecord(ss_.join, ss_.s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(main_, ss_.join, 0);
    return e;
  }

 private:
  SideStream ss_;
  cudaStream_t main_ = nullptr;
  bool open_ = false;
  int n_marks_ = 0;
};

#define MM_MOE_TRY(expr)                         \
  do {                                           \
    if ((expr) != cudaSuccess) return MM_MOE_ECUDA; \
  } while (0)


// A GEMM operand: a bf16 tensor, or (MXFP8) e4m3 codes and their scales.
struct Opnd {
  const void* p;
  const uint8_t* sf;
};

// The MXFP8 copy at byte offset `off` of `base` of a [rows, cols] operand: its codes,
// then its scales.
struct MxCopy {
  uint8_t* codes;
  uint8_t* sf;
  operator Opnd() const { return Opnd{codes, sf}; }
};
static MxCopy mx_copy(const char* base, size_t off, int64_t rows, int64_t cols) {
  uint8_t* c = reinterpret_cast<uint8_t*>(const_cast<char*>(base) + off);
  return MxCopy{c, c + rows * cols};
}

// MXFP8 quantisation of a bf16 [rows, cols] operand: blocks along its rows, or down
// its columns (with rows_out non-null the same read also yields the row blocks; a
// gather reads the rows from a token-major tensor).
static cudaError_t mx_rows(const Ctx& c, const uint16_t* in, MxCopy out, int64_t rows,
                           int64_t cols, const int* meta) {
  MxqArgs a{};
  a.in = in;
  a.codes = out.codes;
  a.sf = out.sf;
  a.rows = rows;
  a.cols = cols;
  a.along_rows = true;
  a.meta = meta;
  return launch_mxq(c, a);
}

static cudaError_t mx_cols(const Ctx& c, DevStatus* st, const uint16_t* in, MxCopy out,
                           int64_t rows, int64_t cols, const int* meta,
                           const MxCopy* rows_out = nullptr, RowGather gather = RowGather{}) {
  MxqArgs a{};
  a.status = st;
  a.in = in;
  a.codes = out.codes;
  a.sf = out.sf;
  a.rows = rows;
  a.cols = cols;
  a.along_rows = false;
  a.meta = meta;
  if (rows_out != nullptr) {
    a.codes_rows = rows_out->codes;
    a.sf_rows = rows_out->sf;
  }
  a.gather = gather;
  return launch_mxq(c, a);
}

// The quantised copy of an activation operand under scheme qs (MXFP8: 32-element
// blocks; blockwise FP8: 128-element blocks): along its rows, or down its columns (with
// rows_out non-null the same read also yields the row blocks; a gather reads the rows
// from a token-major tensor).
static cudaError_t q_rows(const Ctx& c, int qs, const uint16_t* in, MxCopy out, int64_t rows,
                          int64_t cols, const int* meta) {
  if (qs == QS_MX) return mx_rows(c, in, out, rows, cols, meta);
  FbqArgs a{};
  a.in = in;
  a.codes = out.codes;
  a.sf = out.sf;
  a.rows = rows;
  a.cols = cols;
  a.layout = FB_ROWS;
  a.meta = meta;
  return launch_fbq(c, a);
}

static cudaError_t q_cols(const Ctx& c, int qs, DevStatus* st, const uint16_t* in, MxCopy out,
                          int64_t rows, int64_t cols, const int* meta,
                          const MxCopy* rows_out = nullptr, RowGather gather = RowGather{}) {
  if (qs == QS_MX) return mx_cols(c, st, in, out, rows, cols, meta, rows_out, gather);
  FbqArgs a{};
  a.in = in;
  a.codes = out.codes;
  a.sf = out.sf;
  a.rows = rows;
  a.cols = cols;
  a.layout = FB_COLS;
  a.meta = meta;
  if (rows_out != nullptr) {
    a.codes_rows = rows_out->codes;
    a.sf_rows = rows_out->sf;
  }
  a.gather = gather;
  return launch_fbq(c, a);
}

// A weight's quantised copy at byte offset `off` of `base`, [rows, cols]: MXFP8's
// copies (each quantised along the K of the GEMMs that read it), or blockwise FP8's one
// copy, read with the scales of the arrangement the GEMM needs (mn: the weight's
// columns are the MMA rows, i.e. the GEMM contracts its rows).
static MxCopy w_copy(int qs, const char* base, size_t off, int64_t rows, int64_t cols, bool mn) {
  MxCopy m = mx_copy(base, off, rows, cols);
  if (qs == QS_BLOCK && mn) m.sf += rows * cols / 32;
  return m;
}

// Blockwise FP8's copy of a weight: 128 x 128 blocks, the codes and both scale
// arrangements, at offset `off` of `base`.
static cudaError_t fbq_weight(const Ctx& c, const uint16_t* W, char* base, size_t off,
                              int64_t rows, int64_t cols) {
  const MxCopy k = w_copy(QS_BLOCK, base, off, rows, cols, false);
  FbqArgs a{};
  a.in = W;
  a.codes = k.codes;
  a.sf = k.sf;
  a.sf_mn = k.sf + rows * cols / 32;
  a.rows = rows;
  a.cols = cols;
  a.layout = FB_TILES;
  return launch_fbq(c, a);
}

// The padded expert-grouped rows of a token-major tensor, for the column passes.
static RowGather routed_rows(const Layout& L, const char* sv) {
  return RowGather{reinterpret_cast<const int*>(sv + L.rowflat),
                   reinterpret_cast<const int*>(sv + L.tile_rows), static_cast<int>(L.k)};
}

// The permutation of x, and gate/up's A operand.  Under a quantised forward it writes
// x's blocks along H (the gate/up operand) straight to q_x, quantising each token row
// once (MXFP8: codes and scales; blockwise: bf16 values); no bf16 copy of the
// permuted rows is made.  Otherwise x_perm is the bf16 permuted copy.
static Opnd permute_x(const Ctx& c, const Layout& L, const uint16_t* x, uint16_t* x_perm,
                      const char* sv, float* w_row_out, char* sc, cudaError_t* err) {
  if (L.qf == QS_NONE) {
    *err = launch_permute(c, L, x, x_perm, sv, w_row_out, K_PERMUTE_X, sc);
    return Opnd{x_perm, nullptr};
  }
  const MxCopy q = mx_copy(sc, L.q_x, L.Rp, L.H);
  *err = launch_permute(c, L, x, q.codes, sv, w_row_out, K_PERMUTE_X, sc, L.qf, q.sf);
  return q;
}

// x's blocks along tokens (the dW_gate / dW_up operand), gathered from x in routed
// order into `dst` (saved's x_perm place, or q_xc), under scheme qs.
static cudaError_t x_tokens(const Ctx& c, const Layout& L, int qs, const uint16_t* x, char* dst,
                            const char* sv, char* sc) {
  const int* meta = reinterpret_cast<const int*>(sv + L.meta);
  DevStatus* sw = reinterpret_cast<DevStatus*>(sc + L.status);  // the status word
  return q_cols(c, qs, sw, x, mx_copy(dst, 0, L.Rp, L.H), L.Rp, L.H, meta, nullptr,
                routed_rows(L, sv));
}

// The weight copies of a quantised forward; they read only the weights, so the
// forward runs them on its side stream beside the routing (gate/up's first, then
// W_down's, which only the down projection waits for).  MXFP8: with `keep` (the
// forward of a layer that keeps its activations) one two-way pass per weight writes
// its blocks along the forward's K to scratch and along the backward's K to `wbase`
// (saved); otherwise row passes write the forward's copies only.  Blockwise FP8: the
// one 128 x 128-block copy of each weight (codes and both scale arrangements), which
// every GEMM reads, to `wbase` (saved, or the front of scratch under recompute).
static cudaError_t weights_gateup(const Ctx& c, const Layout& L, bool keep,
                                  const uint16_t* W_gate, const uint16_t* W_up, char* wbase,
                                  char* sc) {
  const int64_t EI = L.E * L.I;
  DevStatus* sw = reinterpret_cast<DevStatus*>(sc + L.status);  // the status word
  cudaError_t e = cudaSuccess;
  if (L.qf == QS_MX) {
    const MxCopy wg = mx_copy(sc, L.q_wg, EI, L.H), wu = mx_copy(sc, L.q_wu, EI, L.H);
    if (keep) {  // one read each, both axes
      e = mx_cols(c, sw, W_gate, mx_copy(wbase, L.q_wgc, EI, L.H), EI, L.H, nullptr, &wg);
      if (e == cudaSuccess)
        e = mx_cols(c, sw, W_up, mx_copy(wbase, L.q_wuc, EI, L.H), EI, L.H, nullptr, &wu);
    } else {
      e = mx_rows(c, W_gate, wg, EI, L.H, nullptr);
      if (e == cudaSuccess) e = mx_rows(c, W_up, wu, EI, L.H, nullptr);
    }
  } else if (L.qf == QS_BLOCK) {
    e = fbq_weight(c, W_gate, wbase, L.q_wgc, EI, L.H);
    if (e == cudaSuccess) e = fbq_weight(c, W_up, wbase, L.q_wuc, EI, L.H);
  }
  return e;
}

static cudaError_t weights_down(const Ctx& c, const Layout& L, bool keep,
                                const uint16_t* W_down, char* wbase, char* sc) {
  const int64_t EH = L.E * L.H;
  DevStatus* sw = reinterpret_cast<DevStatus*>(sc + L.status);  // the status word
  if (L.qf == QS_MX) {
    const MxCopy wd = mx_copy(sc, L.q_wd, EH, L.I);
    return keep ? mx_cols(c, sw, W_down, mx_copy(wbase, L.q_wdc, EH, L.I), EH, L.I, nullptr, &wd)
                : mx_rows(c, W_down, wd, EH, L.I, nullptr);
  }
  if (L.qf == QS_BLOCK) return fbq_weight(c, W_down, wbase, L.q_wdc, EH, L.I);
  return cudaSuccess;
}

// The forward's gate/up stage on A (from permute_x): h = [g | u] and a = silu(g) * u,
// from the weights (or, in a quantised forward, their copies made by weights_gateup,
// which the caller has made or ordered before).  `emit_qa` makes it also produce the
// down projection's operand: a in MXFP8 along I from the GEMM's epilogue, or
// (blockwise FP8) a row pass over a.  The backward under MM_MOE_RECOMPUTE calls it
// with the forward's arguments and gets h and a bit for bit (the same kernels on the
// same inputs).
static mm_moe_status gateup_stage(const Ctx& c, const Layout& L, bool emit_qa, Opnd A,
                                  const uint16_t* W_gate, const uint16_t* W_up, uint16_t* h,
                                  uint16_t* a, const char* sv, char* wbase, char* sc) {
  const int* meta = reinterpret_cast<const int*>(sv + L.meta);
  GemmArgs g{};
  g.saved = sv;
  g.scratch = sc;
  g.kind = GEMM_GATEUP;
  g.A = A.p;
  g.sA = A.sf;
  g.B0 = W_gate;
  g.B1 = W_up;
  g.out0 = h;
  g.out1 = a;
  if (L.qf == QS_MX) {
    const MxCopy wg = mx_copy(sc, L.q_wg, L.E * L.I, L.H), wu = mx_copy(sc, L.q_wu, L.E * L.I, L.H);
    g.fp8 = true;
    g.B0 = wg.codes;
    g.sB0 = wg.sf;
    g.B1 = wu.codes;
    g.sB1 = wu.sf;
    if (emit_qa) {
      const MxCopy qa = mx_copy(sc, L.q_a, L.Rp, L.I);
      g.q_codes = qa.codes;
      g.q_sf = qa.sf;
    }
  } else if (L.qf == QS_BLOCK) {
    const MxCopy wg = w_copy(QS_BLOCK, wbase, L.q_wgc, L.E * L.I, L.H, false),
                 wu = w_copy(QS_BLOCK, wbase, L.q_wuc, L.E * L.I, L.H, false);
    g.fp8 = true;
    g.B0 = wg.codes;
    g.sB0 = wg.sf;
    g.B1 = wu.codes;
    g.sB1 = wu.sf;
  }
  MM_MOE_TRY(launch_gemm(c, L, g));
  if (L.qf == QS_BLOCK && emit_qa)
    MM_MOE_TRY(q_rows(c, QS_BLOCK, a, mx_copy(sc, L.q_a, L.Rp, L.I), L.Rp, L.I, meta));
  return MM_MOE_OK;
}

}  // namespace mmmoe

using namespace mmmoe;

extern "C" MM_MOE_API mm_moe_status mm_moe_workspace_size(const mm_moe_shape* shape,
                                                          size_t* scratch_bytes,
                                                          size_t* saved_bytes) {
  Layout L;
  const mm_moe_status st = make_layout(shape, &L);
  if (st != MM_MOE_OK) return st;
  if (scratch_bytes) *scratch_bytes = L.scratch_bytes;
  if (saved_bytes) *saved_bytes = L.saved_bytes;
  return MM_MOE_OK;
}

extern "C" MM_MOE_API mm_moe_status mm_moe_forward(const mm_moe_shape* shape, const uint16_t* x,
                                                   const int32_t* topk_idx, const float* topk_w,
                                                   const uint16_t* W_gate, const uint16_t* W_up,
                                                   const uint16_t* W_down, uint16_t* y,
                                                   void* scratch, void* saved, void* stream) {
  Layout L;
  mm_moe_status st = make_layout(shape, &L);
  if (st != MM_MOE_OK) return st;
  if (!aligned(x, 16) || !aligned(W_gate, 16) || !aligned(W_up, 16) || !aligned(W_down, 16) ||
      !aligned(y, 16) || !aligned(topk_idx, 4) || !aligned(topk_w, 4) || !aligned(scratch, 256) ||
      !aligned(saved, 256))
    return MM_MOE_EINVAL;
  DevInfo d;
  st = device_info(&d);
  if (st != MM_MOE_OK) return st;
  int launches = 0;
  Ctx c{static_cast<cudaStream_t>(stream), d.sms, &launches};
  char* sc = static_cast<char*>(scratch);
  char* sv = static_cast<char*>(saved);
  MM_MOE_TRY(cudaMemsetAsync(sc + L.status, 0, sizeof(DevStatus), c.stream));
  // A quantised forward's weight copies read only the weights: they run on the side
  // stream beside the routing and the permutation (which write none of the buffers
  // they write); gate/up waits for its two weights only, the down projection for
  // W_down's copy.  The side stream then gathers x's blocks along tokens (the
  // backward's operand) beside the two GEMMs.
  char* wbase = L.w_common ? sc : sv;  // where the backward's (blockwise: all) weight copies go
  Fork fork;
  int m_gateup = -1, m_down = -1;
  const Ctx cs{nullptr, d.sms, &launches};
  Ctx side = cs;
  if (L.qf != QS_NONE) {
    if (!fork.open(c.stream)) return MM_MOE_ECUDA;
    side.stream = fork.side();
    MM_MOE_TRY(weights_gateup(side, L, L.w_in_saved, W_gate, W_up, wbase, sc));
    m_gateup = fork.mark();
    MM_MOE_TRY(weights_down(side, L, L.w_in_saved, W_down, wbase, sc));
    m_down = fork.mark();
    if (m_gateup < 0 || m_down < 0) return MM_MOE_ECUDA;
  }
  MM_MOE_TRY(launch_route(c, L, topk_idx, topk_w, sv, sc));
  // x_perm, h, a: kept in saved, or in scratch under MM_MOE_RECOMPUTE
  char* act = L.recompute ? sc : sv;
  uint16_t* x_perm = reinterpret_cast<uint16_t*>(act + L.x_perm);
  uint16_t* h = reinterpret_cast<uint16_t*>(act + L.h);
  uint16_t* a = reinterpret_cast<uint16_t*>(act + L.a);
  uint16_t* ys = reinterpret_cast<uint16_t*>(sc + L.ys);
  if (L.w_in_saved) {  // x along tokens into x_perm's place, once the routing exists
    MM_MOE_TRY(fork.after_main());
    MM_MOE_TRY(x_tokens(side, L, L.qf, x, act + L.x_perm, sv, sc));
  }
  // Operands of the two GEMMs: the bf16 tensors, or in a quantised forward their
  // copies quantised along each GEMM's K (H for gate/up, I for down)
  cudaError_t err = cudaSuccess;
  const Opnd A1 = permute_x(c, L, x, x_perm, sv, reinterpret_cast<float*>(sv + L.w_row), sc, &err);
  MM_MOE_TRY(err);
  if (m_gateup >= 0) MM_MOE_TRY(fork.main_waits(m_gateup));
  st = gateup_stage(c, L, true, A1, W_gate, W_up, h, a, sv, wbase, sc);
  if (st != MM_MOE_OK) return st;
  GemmArgs g{};
  g.saved = sv;
  g.scratch = sc;
  g.kind = GEMM_DOWN;
  g.A = a;
  g.B0 = W_down;
  g.out0 = ys;
  if (L.qf != QS_NONE) {
    const MxCopy qa = mx_copy(sc, L.q_a, L.Rp, L.I);
    const MxCopy wd = L.qf == QS_MX ? mx_copy(sc, L.q_wd, L.E * L.H, L.I)
                                    : w_copy(QS_BLOCK, wbase, L.q_wdc, L.E * L.H, L.I, false);
    g.fp8 = true;
    g.A = qa.codes;
    g.sA = qa.sf;
    g.B0 = wd.codes;
    g.sB0 = wd.sf;
  }
  if (m_down >= 0) MM_MOE_TRY(fork.main_waits(m_down));
  MM_MOE_TRY(launch_gemm(c, L, g));
  MM_MOE_TRY(launch_combine(c, L, ys, sv, y));
  MM_MOE_TRY(fork.join());
  g_last_launches = launches;
  return MM_MOE_OK;
}

extern "C" MM_MOE_API mm_moe_status mm_moe_backward(const mm_moe_shape* shape, const uint16_t* dy,
                                                    const void* saved, const uint16_t* W_gate,
                                                    const uint16_t* W_up, const uint16_t* W_down,
                                                    const uint16_t* x, uint16_t* dx,
                                                    uint16_t* dW_gate,
                                                    uint16_t* dW_up, uint16_t* dW_down,
                                                    float* dtopk_w, void* scratch, void* stream) {
  Layout L;
  mm_moe_status st = make_layout(shape, &L);
  if (st != MM_MOE_OK) return st;
  if (!aligned(dy, 16) || !aligned(W_gate, 16) || !aligned(W_up, 16) || !aligned(W_down, 16) ||
      !aligned(dx, 16) || !aligned(dW_gate, 16) || !aligned(dW_up, 16) || !aligned(dW_down, 16) ||
      !aligned(dtopk_w, 4) || !aligned(scratch, 256) || !aligned(saved, 256) ||
      (L.recompute && !aligned(x, 16)))
    return MM_MOE_EINVAL;
  DevInfo d;
  st = device_info(&d);
  if (st != MM_MOE_OK) return st;
  int launches = 0;
  Ctx c{static_cast<cudaStream_t>(stream), d.sms, &launches};
  char* sc = static_cast<char*>(scratch);
  const char* sv = static_cast<const char*>(saved);
  uint16_t* dy_perm = reinterpret_cast<uint16_t*>(sc + L.dy_perm);
  uint16_t* dh = reinterpret_cast<uint16_t*>(sc + L.dh);
  uint16_t* a_w = reinterpret_cast<uint16_t*>(sc + L.a_w);
  float* pw = reinterpret_cast<float*>(sc + L.pw);
  uint16_t* dxs = reinterpret_cast<uint16_t*>(sc + L.dxs);
  const char* act = L.recompute ? sc : sv;  // where x_perm, h and a are
  const uint16_t* x_perm = reinterpret_cast<const uint16_t*>(act + L.x_perm);
  const uint16_t* h = reinterpret_cast<const uint16_t*>(act + L.h);
  const uint16_t* a = reinterpret_cast<const uint16_t*>(act + L.a);
  const int* meta = reinterpret_cast<const int*>(sv + L.meta);
  const int64_t EI = L.E * L.I, EH = L.E * L.H, Rp = L.Rp, H = L.H, I = L.I;
  DevStatus* sw = reinterpret_cast<DevStatus*>(sc + L.status);  // the status word
  MM_MOE_TRY(cudaMemsetAsync(sc + L.status, 0, sizeof(DevStatus), c.stream));
  if (L.recompute) {
    // activation checkpointing: gate/up's operand (x_perm, or q_x under a quantised
    // forward), h and a again, as the forward made them
    uint16_t* xp = reinterpret_cast<uint16_t*>(sc + L.x_perm);
    MM_MOE_TRY(weights_gateup(c, L, false, W_gate, W_up, sc, sc));
    cudaError_t err = cudaSuccess;
    const Opnd A0 = permute_x(c, L, x, xp, sv, nullptr, sc, &err);
    MM_MOE_TRY(err);
    if (L.qf == QS_BLOCK) MM_MOE_TRY(weights_down(c, L, false, W_down, sc, sc));
    st = gateup_stage(c, L, false, A0, W_gate, W_up, reinterpret_cast<uint16_t*>(sc + L.h),
                      reinterpret_cast<uint16_t*>(sc + L.a), sv, sc, sc);
    if (st != MM_MOE_OK) return st;
  }
  // A quantised backward (MXFP8 for full MXFP8 and fp8_bwd, blockwise FP8): every
  // GEMM runs on the block-scaled tensor cores and reads copies of its operands
  // quantised along its own K (codes and scales).  The permutation of dy writes dy's
  // blocks along H (the first GEMM's operand) into dy_perm's place; dy's blocks along
  // tokens (the dW_down operand) are gathered from dy on the side stream beside the
  // first two GEMMs, as are (MXFP8 without the forward's copies) the weights along I
  // for dgrad-gate/up.  The backward's weight copies were otherwise made by the forward
  // (saved) or by the recompute (blockwise, front of scratch); blockwise FP8 reads its
  // one weight copy with the scales of the other arrangement here.  (The side stream
  // starts after the recompute, whose buffers overlap these.)
  const int qb = L.qb;
  const char* wsrc = L.w_in_saved ? sv : sc;
  const bool make_w = qb == QS_MX && !L.w_in_saved;
  Fork fork;
  if (!fork.open(c.stream)) return MM_MOE_ECUDA;
  Ctx side{fork.side(), d.sms, &launches};
  int m_dy = -1, m_w = -1;
  if (qb != QS_NONE) {
    MM_MOE_TRY(q_cols(side, qb, sw, dy, mx_copy(sc, L.q_dyc, Rp, H), Rp, H, meta, nullptr,
                      routed_rows(L, sv)));
    m_dy = fork.mark();
    if (make_w) {
      MM_MOE_TRY(mx_cols(side, sw, W_gate, mx_copy(sc, L.q_wgc, EI, H), EI, H, nullptr));
      MM_MOE_TRY(mx_cols(side, sw, W_up, mx_copy(sc, L.q_wuc, EI, H), EI, H, nullptr));
      m_w = fork.mark();
    }
  }
  GemmArgs g{};
  g.saved = sv;
  g.scratch = sc;
  g.kind = GEMM_DGRAD_DOWN;
  g.A = dy_perm;
  g.B0 = W_down;
  g.aux = h;
  g.aux2 = a;
  g.out0 = dh;
  g.out1 = a_w;
  g.outf = pw;
  if (qb != QS_NONE) {
    const MxCopy dyr = mx_copy(sc, L.dy_perm, Rp, H), wdc = w_copy(qb, wsrc, L.q_wdc, EH, I, true);
    MM_MOE_TRY(launch_permute(c, L, dy, dyr.codes, sv, nullptr, K_PERMUTE_DY, sc, qb, dyr.sf));
    if (make_w) MM_MOE_TRY(mx_cols(c, sw, W_down, wdc, EH, I, nullptr));
    g.fp8 = true;
    g.A = dyr.codes;
    g.sA = dyr.sf;
    g.B0 = wdc.codes;
    g.sB0 = wdc.sf;
  } else {
    MM_MOE_TRY(launch_permute(c, L, dy, dy_perm, sv, nullptr, K_PERMUTE_DY, sc, qb));
  }
  MM_MOE_TRY(launch_gemm(c, L, g));
  g = GemmArgs{};
  g.saved = sv;
  g.scratch = sc;
  g.kind = GEMM_DGRAD_GATEUP;
  g.A = dh;
  g.B0 = W_gate;
  g.B1 = W_up;
  g.out0 = dxs;
  if (qb != QS_NONE) {
    // one read of dh: blocks along tokens (dW_gate, dW_up) and along I (this GEMM)
    const MxCopy dhc = mx_copy(sc, L.q_dhc, Rp, 2 * I), dhr = mx_copy(sc, L.q_dhr, Rp, 2 * I);
    const MxCopy wgc = w_copy(qb, wsrc, L.q_wgc, EI, H, true),
                 wuc = w_copy(qb, wsrc, L.q_wuc, EI, H, true);
    MM_MOE_TRY(q_cols(c, qb, sw, dh, dhc, Rp, 2 * I, meta, &dhr));
    if (m_w >= 0) MM_MOE_TRY(fork.main_waits(m_w));
    g.fp8 = true;
    g.A = dhr.codes;
    g.sA = dhr.sf;
    g.B0 = wgc.codes;
    g.sB0 = wgc.sf;
    g.B1 = wuc.codes;
    g.sB1 = wuc.sf;
  }
  MM_MOE_TRY(launch_gemm(c, L, g));
  // the un-permute (bandwidth-bound) runs on the side stream beside the
  // weight-gradient GEMMs, which read none of its inputs and write none of its outputs
  MM_MOE_TRY(fork.after_main());
  MM_MOE_TRY(launch_unpermute(side, L, dxs, sv, pw, dx, dtopk_w));
  // token-axis blocks of the weight-gradient operands: each expert's rows start on a
  // multiple of 128 and its padding rows are zero, so 32- or 128-row blocks of the
  // padded row space are the per-expert blocks with a zero-padded tail
  g = GemmArgs{};
  g.saved = sv;
  g.scratch = sc;
  g.A = dh;              // dW_gate / dW_up = dh^T x
  g.B0 = x_perm;
  g.A2 = dy_perm;        // dW_down = dy^T (w a)
  g.B2 = a_w;
  g.out0 = dW_gate;
  g.out1 = dW_up;
  g.out2 = dW_down;
  if (qb != QS_NONE) {
    const MxCopy awc = mx_copy(sc, L.q_awc, Rp, I);
    MM_MOE_TRY(q_cols(c, qb, sw, a_w, awc, Rp, I, meta));
    MxCopy xc = mx_copy(sv, L.x_perm, Rp, H);  // the forward's gather (kept activations)
    if (!L.w_in_saved) {
      xc = mx_copy(sc, L.q_xc, Rp, H);
      if (L.qf == QS_NONE)  // fp8_bwd: from the forward's bf16 x_perm
        MM_MOE_TRY(mx_cols(c, sw, x_perm, xc, Rp, H, meta));
      else                  // recompute under a quantised forward: from x itself
        MM_MOE_TRY(x_tokens(c, L, qb, x, reinterpret_cast<char*>(xc.codes), sv, sc));
    }
    const MxCopy dyc = mx_copy(sc, L.q_dyc, Rp, H), dhc = mx_copy(sc, L.q_dhc, Rp, 2 * I);
    g.fp8 = true;
    g.A = dhc.codes;
    g.sA = dhc.sf;
    g.B0 = xc.codes;
    g.sB0 = xc.sf;
    g.A2 = dyc.codes;
    g.sA2 = dyc.sf;
    g.B2 = awc.codes;
    g.sB2 = awc.sf;
  }
  if (m_dy >= 0) MM_MOE_TRY(fork.main_waits(m_dy));
  // both weight gradients in one launch where they tile N alike (one list of tiles,
  // experts by descending row count, balances the clusters' loads far better than
  // two lists); otherwise one launch each
  const bool both = wgrad_both_ok(L);
  if (!both) {
    GemmArgs gd = g;
    gd.kind = GEMM_WGRAD_DOWN;
    gd.A = g.A2;
    gd.sA = g.sA2;
    gd.B0 = g.B2;
    gd.sB0 = g.sB2;
    gd.out0 = dW_down;
    MM_MOE_TRY(launch_gemm(c, L, gd));
  }
  g.kind = both ? GEMM_WGRAD_BOTH : GEMM_WGRAD_GATEUP;
  MM_MOE_TRY(launch_gemm(c, L, g));
  MM_MOE_TRY(fork.join());  // the call ends on `stream`
  g_last_launches = launches;
  return MM_MOE_OK;
}

extern "C" MM_MOE_API mm_moe_status mm_moe_get_routing(const mm_moe_shape* shape,
                                                       const void* saved,
                                                       const int32_t** offsets,
                                                       const int32_t** perm,
                                                       const int32_t** inv) {
  Layout L;
  const mm_moe_status st = make_layout(shape, &L);
  if (st != MM_MOE_OK) return st;
  if (saved == nullptr) return MM_MOE_EINVAL;
  const char* sv = static_cast<const char*>(saved);
  if (offsets) *offsets = reinterpret_cast<const int32_t*>(sv + L.offsets);
  if (perm) *perm = reinterpret_cast<const int32_t*>(sv + L.perm);
  if (inv) *inv = reinterpret_cast<const int32_t*>(sv + L.inv);
  return MM_MOE_OK;
}

extern "C" MM_MOE_API mm_moe_status mm_moe_read_status(const void* scratch, void* stream) {
  if (scratch == nullptr) return MM_MOE_EINVAL;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MM_MOE_ECUDA;
  DevStatus s{};
  if (cudaMemcpy(&s, scratch, sizeof(s), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MM_MOE_ECUDA;
  return static_cast<mm_moe_status>(s.code);
}

extern "C" MM_MOE_API int mm_moe_last_launch_count(void) { return g_last_launches; }

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

mm_moe_status make_layout(const mm_moe_shape* s, Layout* L) {
  if (s == nullptr || L == nullptr) return MM_MOE_EINVAL;
  *L = Layout{};  // offsets a mode does not use stay 0
  if (s->T < 1 || s->H < 1 || s->I < 1 || s->E < 1 || s->k < 1) return MM_MOE_EINVAL;
  if (s->k > s->E || s->E > MAX_E) return MM_MOE_EINVAL;
  if (s->H % 128 != 0 || s->I % 64 != 0) return MM_MOE_EINVAL;
  if ((s->flags & ~MM_MOE_RECOMPUTE) != 0) return MM_MOE_EINVAL;
  if (s->prec < MM_MOE_BF16 || s->prec > MM_MOE_FP8_BLOCK) return MM_MOE_EINVAL;
  if (s->prec == MM_MOE_FP8_BLOCK && s->I % 128 != 0) return MM_MOE_EINVAL;  // 128 x 128 blocks
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
  L->qf = s->prec == MM_MOE_MXFP8 ? QS_MX : s->prec == MM_MOE_FP8_BLOCK ? QS_BLOCK : QS_NONE;
  L->qb = s->prec == MM_MOE_BF16 ? QS_NONE : s->prec == MM_MOE_FP8_BLOCK ? QS_BLOCK : QS_MX;
  L->nblk = (L->R + ROUTE_CHUNK - 1) / ROUTE_CHUNK;
  L->n_pw = L->I / pick_bn(L->I);
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
    L->x_perm = take(2 * Rp * H);
    L->h = take(2 * Rp * 2 * I);
    L->a = take(2 * Rp * I);
  }
  // a quantised forward that keeps its activations also makes the backward's
  // weight copies (MXFP8: the forward's two-way passes; blockwise: the one copy)
  const size_t W = 2 * E * I * H;  // bytes of one expert weight tensor
  L->w_in_saved = L->qf != QS_NONE && !L->recompute;
  L->w_common = L->qf == QS_BLOCK && L->recompute;
  L->q_wdc = L->q_wgc = L->q_wuc = 0;
  if (L->w_in_saved) {
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
    L->q_wdc = take(W);
    L->q_wgc = take(W);
    L->q_wuc = take(W);
  }
  const size_t common = o;
  L->ys = take(2 * Rp * H);
  // quantised operand copies of the forward (bf16 holding the dequantised values)
  L->q_x = L->q_a = L->q_wg = L->q_wu = L->q_wd = 0;
  if (L->qf != QS_NONE) {
    L->q_x = take(2 * Rp * H);
    L->q_a = take(2 * Rp * I);
  }
  if (L->qf == QS_MX) {  // the forward's MXFP8 weights (blocks along their forward K)
    L->q_wg = take(W);
    L->q_wu = take(W);
    L->q_wd = take(W);
  }
  const size_t fwd_end = o;
  o = common;
  L->dy_perm = take(2 * Rp * H);
  L->dh = take(2 * Rp * 2 * I);
  L->a_w = take(2 * Rp * I);
  L->pw = take(4 * Rp * static_cast<size_t>(L->n_pw));
  L->dxs = take(2 * Rp * H);
  L->q_dyc = L->q_dhc = L->q_xc = 0;
  if (L->qb != QS_NONE && !L->w_in_saved) {  // left to the backward
    if (!L->w_common) {
      L->q_wdc = take(W);
      L->q_wgc = take(W);
      L->q_wuc = take(W);
    }
    L->q_xc = take(2 * Rp * H);
  }
  if (L->qb != QS_NONE) {
    L->q_dyc = take(2 * Rp * H);
    L->q_dhc = take(2 * Rp * 2 * I);
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
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
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
  }
  *out = ss;
  return true;
}

// A fork of the caller's stream onto the side stream that is joined back on every
// return: join() on the normal path, the destructor on an error return after the
// fork, so that no path leaves forked work unordered before later work on the
// caller's stream (or an unjoined fork in a stream capture).
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
};

#define MM_MOE_TRY(expr)                         \
  do {                                           \
    if ((expr) != cudaSuccess) return MM_MOE_ECUDA; \
  } while (0)

// Quantisation of an activation operand under scheme qs (QS_MX: 32-element blocks,
// QS_BLOCK: 128-element blocks): along rows, or down columns (with out_rows non-null
// the same read also writes the row blocks there).
static cudaError_t act_rows(const Ctx& c, int qs, const uint16_t* in, uint16_t* out,
                            int64_t rows, int64_t cols, const int* meta) {
  return qs == QS_BLOCK ? launch_fb_qdq(c, in, out, rows, cols, FB_ROWS, meta, nullptr)
                        : launch_mx_qdq(c, in, out, rows, cols, true, meta);
}

static cudaError_t act_cols(const Ctx& c, int qs, const uint16_t* in, uint16_t* out,
                            int64_t rows, int64_t cols, const int* meta,
                            uint16_t* out_rows = nullptr, RowGather gather = RowGather{}) {
  return qs == QS_BLOCK ? launch_fb_qdq(c, in, out, rows, cols, FB_COLS, meta, out_rows, gather)
                        : launch_mx_qdq(c, in, out, rows, cols, false, meta, out_rows, gather);
}

// The padded expert-grouped rows of a token-major tensor, for act_cols.
static RowGather routed_rows(const Layout& L, const char* sv) {
  return RowGather{reinterpret_cast<const int*>(sv + L.rowflat),
                   reinterpret_cast<const int*>(sv + L.tile_rows), static_cast<int>(L.k)};
}

// Under a quantised forward the permutation of x writes x's blocks along H (the
// gate/up operand) straight to q_x, quantising each token row once; the blocks along
// tokens (the dW_gate / dW_up operand), when wanted, are gathered from x into
// `x_cols`.  No bf16 copy of the permuted rows is made.  Otherwise x_perm is the
// bf16 permuted copy.  Returns gate/up's A operand.
static const uint16_t* permute_x(const Ctx& c, const Layout& L, const uint16_t* x,
                                 uint16_t* x_perm, uint16_t* x_cols, const char* sv,
                                 float* w_row_out, char* sc, cudaError_t* err) {
  if (L.qf == QS_NONE) {
    *err = launch_permute(c, L, x, x_perm, sv, w_row_out, K_PERMUTE_X, sc);
    return x_perm;
  }
  uint16_t* q_x = reinterpret_cast<uint16_t*>(sc + L.q_x);
  *err = launch_permute(c, L, x, q_x, sv, w_row_out, K_PERMUTE_X, sc, L.qf);
  if (*err == cudaSuccess && x_cols != nullptr)
    *err = act_cols(c, L.qf, x, x_cols, L.Rp, L.H, reinterpret_cast<const int*>(sv + L.meta),
                    nullptr, routed_rows(L, sv));
  return q_x;
}

// The forward's gate/up stage on A (from permute_x): h = [g | u] and a = silu(g) * u.
// Under a quantised forward (L.qf) the weights are first quantised along H.  MXFP8:
// with `keep` (the forward of a layer that keeps its activations) by two-way passes
// that also write the weights along their backward K to `wbase` (saved); otherwise by
// row passes; `emit_qa` makes the epilogue also write a quantised along I for the down
// projection.  Blockwise FP8: the one 128 x 128-block copy of each of the three
// weights goes to `wbase` (saved, or the front of scratch under recompute); `emit_qa`
// adds a row pass over a.  The backward under MM_MOE_RECOMPUTE calls it with the
// forward's arguments and gets h and a bit for bit (the same kernels on the same
// inputs).
// The weight copies of a quantised forward (see gateup_stage); they read only the
// weights, so the forward runs them on its side stream beside the routing.
static cudaError_t weight_copies(const Ctx& c, const Layout& L, bool keep, bool emit_qa,
                                 const uint16_t* W_gate, const uint16_t* W_up,
                                 const uint16_t* W_down, char* wbase, char* sc) {
  const int64_t EI = L.E * L.I, EH = L.E * L.H;
  auto sq = [&](size_t off) { return reinterpret_cast<uint16_t*>(sc + off); };
  auto wq = [&](size_t off) { return reinterpret_cast<uint16_t*>(wbase + off); };
  cudaError_t e = cudaSuccess;
  if (L.qf == QS_MX) {
    if (keep) {  // one read each, both axes
      e = launch_mx_qdq(c, W_gate, wq(L.q_wgc), EI, L.H, false, nullptr, sq(L.q_wg));
      if (e == cudaSuccess)
        e = launch_mx_qdq(c, W_up, wq(L.q_wuc), EI, L.H, false, nullptr, sq(L.q_wu));
      if (e == cudaSuccess && emit_qa)
        e = launch_mx_qdq(c, W_down, wq(L.q_wdc), EH, L.I, false, nullptr, sq(L.q_wd));
    } else {
      e = launch_mx_qdq(c, W_gate, sq(L.q_wg), EI, L.H, true, nullptr);
      if (e == cudaSuccess) e = launch_mx_qdq(c, W_up, sq(L.q_wu), EI, L.H, true, nullptr);
      if (e == cudaSuccess && emit_qa)
        e = launch_mx_qdq(c, W_down, sq(L.q_wd), EH, L.I, true, nullptr);
    }
  } else if (L.qf == QS_BLOCK) {  // the copies every GEMM of the layer reads
    e = launch_fb_qdq(c, W_gate, wq(L.q_wgc), EI, L.H, FB_TILES, nullptr, nullptr);
    if (e == cudaSuccess)
      e = launch_fb_qdq(c, W_up, wq(L.q_wuc), EI, L.H, FB_TILES, nullptr, nullptr);
    if (e == cudaSuccess)
      e = launch_fb_qdq(c, W_down, wq(L.q_wdc), EH, L.I, FB_TILES, nullptr, nullptr);
  }
  return e;
}

static mm_moe_status gateup_stage(const Ctx& c, const Layout& L, bool keep, bool emit_qa,
                                  const uint16_t* A, const uint16_t* W_gate,
                                  const uint16_t* W_up, const uint16_t* W_down, uint16_t* h,
                                  uint16_t* a, const char* sv, char* wbase, char* sc,
                                  bool weights_ready = false) {
  const int* meta = reinterpret_cast<const int*>(sv + L.meta);
  auto sq = [&](size_t off) { return reinterpret_cast<uint16_t*>(sc + off); };
  auto wq = [&](size_t off) { return reinterpret_cast<uint16_t*>(wbase + off); };
  if (!weights_ready)
    MM_MOE_TRY(weight_copies(c, L, keep, emit_qa, W_gate, W_up, W_down, wbase, sc));
  const uint16_t *Bg = W_gate, *Bu = W_up;
  if (L.qf == QS_MX) {
    Bg = sq(L.q_wg);
    Bu = sq(L.q_wu);
  } else if (L.qf == QS_BLOCK) {
    Bg = wq(L.q_wgc);
    Bu = wq(L.q_wuc);
  }
  GemmArgs g{};
  g.saved = sv;
  g.scratch = sc;
  g.kind = GEMM_GATEUP;
  g.A = A;
  g.B0 = Bg;
  g.B1 = Bu;
  g.out0 = h;
  g.out1 = a;
  g.mx = (L.qf == QS_MX && emit_qa) ? 1 : 0;
  g.q0 = g.mx ? sq(L.q_a) : nullptr;
  MM_MOE_TRY(launch_gemm(c, L, g));
  if (L.qf == QS_BLOCK && emit_qa) MM_MOE_TRY(act_rows(c, QS_BLOCK, a, sq(L.q_a), L.Rp, L.I, meta));
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
  // stream beside the routing, the permutation and the token-axis gather, which write
  // none of the buffers they write, and gate/up waits for them
  char* wbase = L.w_common ? sc : sv;  // where the backward's (blockwise: all) weight copies go
  const bool side = L.qf != QS_NONE;
  Fork fork;
  if (side) {
    if (!fork.open(c.stream)) return MM_MOE_ECUDA;
    const Ctx cs{fork.side(), d.sms, &launches};
    MM_MOE_TRY(weight_copies(cs, L, L.w_in_saved, true, W_gate, W_up, W_down, wbase, sc));
  }
  MM_MOE_TRY(launch_route(c, L, topk_idx, topk_w, sv, sc));
  // x_perm, h, a: kept in saved, or in scratch under MM_MOE_RECOMPUTE
  char* act = L.recompute ? sc : sv;
  uint16_t* x_perm = reinterpret_cast<uint16_t*>(act + L.x_perm);
  uint16_t* h = reinterpret_cast<uint16_t*>(act + L.h);
  uint16_t* a = reinterpret_cast<uint16_t*>(act + L.a);
  uint16_t* ys = reinterpret_cast<uint16_t*>(sc + L.ys);
  // Operands of the two GEMMs: the bf16 tensors, or in a quantised forward their
  // copies quantised along each GEMM's K (H for gate/up, I for down).  A forward that
  // keeps its activations also leaves x's blocks along tokens in x_perm's place.
  cudaError_t err = cudaSuccess;
  const uint16_t* A1 = permute_x(c, L, x, x_perm, L.w_in_saved ? x_perm : nullptr, sv,
                                 reinterpret_cast<float*>(sv + L.w_row), sc, &err);
  MM_MOE_TRY(err);
  MM_MOE_TRY(fork.join());
  st = gateup_stage(c, L, L.w_in_saved, true, A1, W_gate, W_up, W_down, h, a, sv, wbase, sc,
                    side);
  if (st != MM_MOE_OK) return st;
  const uint16_t* A2 = L.qf != QS_NONE ? reinterpret_cast<uint16_t*>(sc + L.q_a) : a;
  const uint16_t* Bd = L.qf == QS_MX      ? reinterpret_cast<uint16_t*>(sc + L.q_wd)
                       : L.qf == QS_BLOCK ? reinterpret_cast<uint16_t*>(wbase + L.q_wdc)
                                          : W_down;
  GemmArgs g{};
  g.saved = sv;
  g.scratch = sc;
  g.kind = GEMM_DOWN;
  g.A = A2;
  g.B0 = Bd;
  g.out0 = ys;
  MM_MOE_TRY(launch_gemm(c, L, g));
  MM_MOE_TRY(launch_combine(c, L, ys, sv, y));
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
  MM_MOE_TRY(cudaMemsetAsync(sc + L.status, 0, sizeof(DevStatus), c.stream));
  if (L.recompute) {
    // activation checkpointing: gate/up's operand (x_perm, or q_x under a quantised
    // forward), h and a again, as the forward made them
    uint16_t* xp = reinterpret_cast<uint16_t*>(sc + L.x_perm);
    cudaError_t err = cudaSuccess;
    const uint16_t* A0 = permute_x(c, L, x, xp, nullptr, sv, nullptr, sc, &err);
    MM_MOE_TRY(err);
    st = gateup_stage(c, L, false, false, A0, W_gate, W_up, W_down,
                      reinterpret_cast<uint16_t*>(sc + L.h),
                      reinterpret_cast<uint16_t*>(sc + L.a), sv, sc, sc);
    if (st != MM_MOE_OK) return st;
  }
  // A quantised backward (MXFP8 for full MXFP8 and fp8_bwd, blockwise FP8): every
  // GEMM reads copies of its operands quantised along its own K.  The permutation of
  // dy then writes dy's blocks along H (this GEMM's operand) to dy_perm, and dy's
  // blocks along tokens (the dW_down operand) are gathered from dy.
  const int qb = L.qb;
  MM_MOE_TRY(launch_permute(c, L, dy, dy_perm, sv, nullptr, K_PERMUTE_DY, sc, qb));
  const int* meta = reinterpret_cast<const int*>(sv + L.meta);
  const int64_t EI = L.E * L.I, EH = L.E * L.H;
  auto q = [&](size_t off) { return reinterpret_cast<uint16_t*>(sc + off); };
  // the backward's quantised weights: made by the forward (saved), by the recompute
  // (blockwise, front of scratch), or here (MXFP8 along their backward K)
  auto qw = [&](size_t off) -> const uint16_t* {
    return L.w_in_saved ? reinterpret_cast<const uint16_t*>(sv + off) : q(off);
  };
  const bool make_w = qb == QS_MX && !L.w_in_saved;
  const uint16_t* A1 = dy_perm;
  const uint16_t* Bd = W_down;
  if (qb != QS_NONE) {
    MM_MOE_TRY(act_cols(c, qb, dy, q(L.q_dyc), L.Rp, L.H, meta, nullptr, routed_rows(L, sv)));
    if (make_w) MM_MOE_TRY(launch_mx_qdq(c, W_down, q(L.q_wdc), EH, L.I, false, nullptr));
    Bd = qw(L.q_wdc);
  }
  GemmArgs g{};
  g.saved = sv;
  g.scratch = sc;
  g.kind = GEMM_DGRAD_DOWN;
  g.A = A1;
  g.B0 = Bd;
  g.aux = h;
  g.aux2 = a;
  g.out0 = dh;
  g.out1 = a_w;
  g.outf = pw;
  MM_MOE_TRY(launch_gemm(c, L, g));
  const uint16_t *A2 = dh, *Bg = W_gate, *Bu = W_up;
  if (qb != QS_NONE) {
    // one read of dh: blocks along tokens (dW_gate, dW_up) to q_dhc, blocks along I
    // (the next GEMM) in place
    MM_MOE_TRY(act_cols(c, qb, dh, q(L.q_dhc), L.Rp, 2 * L.I, meta, dh));
    if (make_w) {
      MM_MOE_TRY(launch_mx_qdq(c, W_gate, q(L.q_wgc), EI, L.H, false, nullptr));
      MM_MOE_TRY(launch_mx_qdq(c, W_up, q(L.q_wuc), EI, L.H, false, nullptr));
    }
    Bg = qw(L.q_wgc);
    Bu = qw(L.q_wuc);
  }
  g = GemmArgs{};
  g.saved = sv;
  g.scratch = sc;
  g.kind = GEMM_DGRAD_GATEUP;
  g.A = A2;
  g.B0 = Bg;
  g.B1 = Bu;
  g.out0 = dxs;
  MM_MOE_TRY(launch_gemm(c, L, g));
  // the un-permute (bandwidth-bound) runs on the side stream beside the
  // weight-gradient GEMMs, which read none of its inputs and write none of its outputs
  Fork fork;
  if (!fork.open(c.stream)) return MM_MOE_ECUDA;
  const Ctx cs{fork.side(), d.sms, &launches};
  MM_MOE_TRY(launch_unpermute(cs, L, dxs, sv, pw, dx, dtopk_w));
  // token-axis blocks of the weight-gradient operands: each expert's rows start on a
  // multiple of 128 and its padding rows are zero, so 32- or 128-row blocks of the
  // padded row space are the per-expert blocks with a zero-padded tail
  const uint16_t *A3 = dy_perm, *B3 = a_w, *A4 = dh, *B4 = x_perm;
  if (qb != QS_NONE) {
    MM_MOE_TRY(act_cols(c, qb, a_w, a_w, L.Rp, L.I, meta));
    if (!L.w_in_saved) {  // (a quantised forward that keeps its activations left x's
                          // blocks along tokens in x_perm's place)
      if (L.qf == QS_NONE)  // fp8_bwd: x_perm is the forward's bf16 copy
        MM_MOE_TRY(act_cols(c, qb, x_perm, q(L.q_xc), L.Rp, L.H, meta));
      else  // recompute under a quantised forward: from x itself
        MM_MOE_TRY(act_cols(c, qb, x, q(L.q_xc), L.Rp, L.H, meta, nullptr, routed_rows(L, sv)));
      B4 = q(L.q_xc);
    }
    A3 = q(L.q_dyc);
    A4 = q(L.q_dhc);
  }
  // both weight gradients in one launch where they tile N alike (one list of tiles,
  // experts by descending row count, balances the clusters' loads far better than
  // two lists); otherwise one launch each
  const bool both = wgrad_both_ok(L);
  g = GemmArgs{};
  g.saved = sv;
  g.scratch = sc;
  g.kind = both ? GEMM_WGRAD_BOTH : GEMM_WGRAD_GATEUP;
  g.A = A4;
  g.B0 = B4;
  g.out0 = dW_gate;
  g.out1 = dW_up;
  g.A2 = A3;
  g.B2 = B3;
  g.out2 = dW_down;
  if (!both) {
    GemmArgs gd{};
    gd.saved = sv;
    gd.scratch = sc;
    gd.kind = GEMM_WGRAD_DOWN;
    gd.A = A3;
    gd.B0 = B3;
    gd.out0 = dW_down;
    MM_MOE_TRY(launch_gemm(c, L, gd));
  }
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

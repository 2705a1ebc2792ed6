/*
 * mm_moe.h -- C ABI of a fused mixture-of-experts layer (forward + backward)
 * for one NVIDIA GB300 (sm_103a).
 *
 * What it computes.  The layer of the Prime Mega MoE pages ("Prime Intellect
 * releases Prime Mega MoE"; section "Why is MoE training communication-bound?":
 * each token goes to a few experts and the GPU sorts tokens by expert before
 * sending them; section "How does the fused kernel work?": dispatch, the two
 * expert linear layers, SwiGLU and combine in one call, intermediates kept in
 * GPU-only scratch buffers, and a backward pass added for training).  On one
 * GPU the dispatch is a permutation of rows:
 *
 *   route     stable sort of the flat (token, slot) indices f = t*k + j by
 *             expert topk_idx[t][j]  ->  offsets[E+1], perm[R], inv[R], R = T*k
 *   forward   g = W_gate[e] x_t,  u = W_up[e] x_t,  a = silu(g) * u,
 *             o = W_down[e] a,    y_t = sum_j topk_w[t][j] * o_(t,j)  (j ascending)
 *   backward  of L = <y, dy>: dx, dW_gate, dW_up, dW_down, dtopk_w
 *
 * Conventions shared by every entry point.
 *   - Every pointer argument except `shape` and the out-parameters of the size
 *     and routing queries is a DEVICE pointer on the current CUDA device, 16-byte
 *     aligned.  bf16 tensors are passed as their 16-bit patterns (uint16_t).
 *   - Every tensor is dense and row-major in the shape written beside it.
 *   - The library allocates and frees nothing.  The caller owns every buffer,
 *     sized by mm_moe_workspace_size, and may reuse scratch between calls.
 *   - Calls only enqueue work on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and return; none blocks the host except
 *     mm_moe_read_status.  Calls on one stream are ordered; calls that share a
 *     scratch or saved buffer on different streams race.  The backward forks part
 *     of its work onto an internal stream of the calling host thread and joins it
 *     back before returning, so all its work is ordered before later work on
 *     `stream`.
 *   - Argument errors are returned before anything is enqueued.  Errors found
 *     on the device (an expert index outside [0, E), a wait that ran out of
 *     time) are written to a status word at the start of `scratch`, which every
 *     forward/backward call clears first; read it with mm_moe_read_status.  No
 *     kernel traps or asserts.
 */
#ifndef MM_MOE_H
#define MM_MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MM_MOE_API __attribute__((visibility("default")))
#else
#define MM_MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Arithmetic of the expert GEMMs.  The pages list BF16, MXFP8 (Blackwell) and
 * an fp8_bwd mode (BF16 forward, FP8 backward) -- section "How does the fused
 * kernel work?".
 *   MM_MOE_BF16     bf16 operands, fp32 accumulation.
 *   MM_MOE_MXFP8    every GEMM operand of the forward and the backward is
 *                   quantised to MXFP8 (OCP Microscaling v1.0: e4m3 elements,
 *                   one power-of-two e8m0 scale 2^(floor(log2 amax) - 8) per 32
 *                   elements along that GEMM's K; token-axis blocks of the
 *                   weight-gradient GEMMs start at each expert's first row, the
 *                   last one zero-padded) and multiplied on the block-scaled FP8
 *                   tensor cores; fp32 accumulation.  Needs I % 128 == 0.
 *   MM_MOE_FP8_BWD  the BF16 forward and the MXFP8 backward (I % 128 == 0).
 *   MM_MOE_FP8_BLOCK blockwise FP8 (the pages' Hopper precision, in the form
 *                   Blackwell tensor cores take) in the forward and the backward:
 *                   activations in 128-element blocks along each GEMM's K (128-row
 *                   token blocks for the weight gradients), weights in 128 x 128
 *                   blocks, one power-of-two scale 2^ceil(log2(amax / 448)) per
 *                   block, e4m3 elements, multiplied on the block-scaled FP8 tensor
 *                   cores like MXFP8 (each block's scale repeated over its 32-element
 *                   scale blocks); fp32 accumulation; needs I % 128 == 0.
 * Stored tensors (h, a, the outputs and the gradients) stay bf16 in every mode,
 * and the quantised operand copies live in `scratch` (which is larger for the
 * quantised modes). */
typedef enum {
  MM_MOE_BF16 = 0,
  MM_MOE_MXFP8 = 1,
  MM_MOE_FP8_BWD = 2,
  MM_MOE_FP8_BLOCK = 3
} mm_moe_precision;

typedef enum {
  MM_MOE_OK = 0,
  MM_MOE_EINVAL = 1,    /* bad shape, NULL or misaligned pointer, undersized call */
  MM_MOE_ENOTSUP = 2,   /* precision or device not supported (needs sm_103) */
  MM_MOE_EBADIDX = 3,   /* device: an expert index outside [0, E); that pair is dropped */
  MM_MOE_ETIMEOUT = 4,  /* device: a pipeline wait ran out of time; outputs undefined */
  MM_MOE_ECUDA = 5      /* a CUDA runtime call or launch failed */
} mm_moe_status;

/* Options of a layer (bits of mm_moe_shape.flags).
 *   MM_MOE_RECOMPUTE  activation checkpointing, as in the pages' training runs
 *                     (section "How fast is Prime Mega MoE?": full activation
 *                     checkpointing): `saved` keeps only the routing; the backward
 *                     takes x again, re-permutes it and re-runs the gate/up GEMM
 *                     (bit-identical to the forward's) before the backward proper.
 *                     Less memory held between the passes, one more GEMM. */
#define MM_MOE_RECOMPUTE 1
/*   MM_MOE_MULTICAST  the bf16 grouped GEMMs (gate/up, down, dgrad-down, dgrad-gate/up)
 *                     run on clusters of two SM pairs where their 256-wide N tiles come
 *                     in an even number: the pairs take N tiles 2j and 2j + 1 of one M
 *                     tile in step and share its A rows by TMA multicast, each CTA
 *                     loading half of them for itself and the other pair (half the A
 *                     reads from L2).  The same results bit for bit.  Off by default:
 *                     a GB300 holds 36 four-CTA clusters (144 of its 152 SMs), which
 *                     costs about what the halved A reads gain (benchmark layer 3.10 ->
 *                     3.11 ms, 235B shape 6.23 -> 6.23 ms on one box).  Single-GPU only:
 *                     the copies read this GPU's own memory. */
#define MM_MOE_MULTICAST 2

/* Problem shape.  T tokens, H hidden, I expert intermediate, E experts, top-k.
 * Limits: T, H, I, E, k >= 1; k <= E <= 1024; H % 128 == 0; I % 64 == 0 (I % 128
 * == 0 in the quantised precisions); T * k < 2^31. */
typedef struct {
  int64_t T, H, I, E, k;
  int32_t prec;   /* mm_moe_precision */
  int32_t flags;  /* MM_MOE_RECOMPUTE | MM_MOE_MULTICAST, or 0; other bits must be 0 */
} mm_moe_shape;

/* Bytes of the two caller-owned device buffers.
 *   scratch : per-call working memory (forward and backward both use it; its
 *             first 256 bytes hold the device status word).
 *   saved   : written by mm_moe_forward, read by mm_moe_backward; holds the
 *             routing (offsets, perm, inv), the routing weights in routed order,
 *             the expert-grouped copy of x, h = [g | u] and a = silu(g) * u in
 *             bf16.  Under MM_MOE_MXFP8 and MM_MOE_FP8_BLOCK the copy of x is kept
 *             quantised along the token axis and `saved` also holds quantised copies
 *             of the weights (MXFP8: along their backward contraction axis;
 *             blockwise: the one copy every GEMM reads), so the backward's weight
 *             arguments must be the forward's, as in every mode.  With MM_MOE_RECOMPUTE it holds
 *             only the routing and the routing weights in routed order; the
 *             expert-grouped x (under a quantised forward only its quantised copy), h
 *             and a live in `scratch`.  It must not change between the forward and
 *             its backward.
 * Returns MM_MOE_EINVAL for an invalid shape. */
MM_MOE_API mm_moe_status mm_moe_workspace_size(const mm_moe_shape* shape,
                                    size_t* scratch_bytes, size_t* saved_bytes);

/* Forward pass.
 *   x        [T, H]    bf16   input tokens
 *   topk_idx [T, k]    int32  expert of each (token, slot)
 *   topk_w   [T, k]    fp32   routing weight of each (token, slot), used as given
 *   W_gate   [E, I, H] bf16   gate projection of every expert
 *   W_up     [E, I, H] bf16   up projection
 *   W_down   [E, H, I] bf16   down projection
 *   y        [T, H]    bf16   output (overwritten)
 *   scratch, saved            caller buffers of the sizes above
 *   stream                    cudaStream_t
 * Internally fp32 accumulation; h, the SwiGLU output a and the weighted expert
 * outputs are stored as bf16; the combine sums the k slots in fp32 in slot
 * order (no atomics, bitwise deterministic). */
MM_MOE_API mm_moe_status mm_moe_forward(const mm_moe_shape* shape,
                             const uint16_t* x, const int32_t* topk_idx, const float* topk_w,
                             const uint16_t* W_gate, const uint16_t* W_up,
                             const uint16_t* W_down, uint16_t* y,
                             void* scratch, void* saved, void* stream);

/* Backward pass of the forward that wrote `saved` (same shape and weights).
 *   dy       [T, H]    bf16   upstream gradient of y
 *   x        [T, H]    bf16   the forward's input; read only with MM_MOE_RECOMPUTE
 *                             (may be NULL otherwise)
 *   dx       [T, H]    bf16   gradient of x (overwritten)
 *   dW_gate  [E, I, H] bf16   gradients of the weights (overwritten, not
 *   dW_up    [E, I, H] bf16   accumulated; an expert with no routed token
 *   dW_down  [E, H, I] bf16   gets exact zeros)
 *   dtopk_w  [T, k]    fp32   gradient of the routing weights
 * dtopk_w[t][j] = <a, W_down[e]^T dy_t> (equal to <dy_t, o> in exact
 * arithmetic).  All sums have a fixed order: bitwise deterministic. */
MM_MOE_API mm_moe_status mm_moe_backward(const mm_moe_shape* shape, const uint16_t* dy,
                              const void* saved,
                              const uint16_t* W_gate, const uint16_t* W_up,
                              const uint16_t* W_down, const uint16_t* x,
                              uint16_t* dx, uint16_t* dW_gate, uint16_t* dW_up,
                              uint16_t* dW_down, float* dtopk_w,
                              void* scratch, void* stream);

/* Device pointers, inside `saved`, to the routing the last forward computed
 * (section "Why is MoE training communication-bound?": tokens sorted by
 * expert).  offsets [E+1] int32: rows of expert e are [offsets[e], offsets[e+1]);
 * perm [T*k] int32: flat index t*k+j of routed row r, ascending inside an
 * expert; inv [T*k] int32: routed row of flat index f.  Host call, no sync. */
MM_MOE_API mm_moe_status mm_moe_get_routing(const mm_moe_shape* shape, const void* saved,
                                 const int32_t** offsets, const int32_t** perm,
                                 const int32_t** inv);

/* The top-k router in front of the layer, and its backward.  The pages say each
 * token goes to a small subset of the experts (section "Why is MoE training
 * communication-bound?"; 8 of 128 in the tested models, "TL;DR") and do not
 * describe the router.  Readings: logits = x W_router^T (no bias); the k largest
 * logits per token in descending order, equal logits to the lower expert index;
 * topk_w = softmax over the chosen logits (the full softmax renormalised over them);
 * the gradient flows through topk_w only.
 *   shape    T, H, E, k as for the layer (I and prec ignored); k <= 32, E <= 1024,
 *            H % 8 == 0, E % 8 == 0
 *   x        [T, H] bf16;  W_router [E, H] bf16
 *   logits   [T, E] fp32 out (x W_router^T, fp32 accumulation)
 *   topk_idx [T, k] int32 out;  topk_w [T, k] fp32 out
 * The three matrix products run on the library's own tensor-core GEMM (bf16
 * operands, fp32 accumulation); like every call of the library these two allocate
 * nothing.  A GEMM wait that ran out of time is not reported (the router calls take
 * no scratch buffer, so they have no status word).  Non-finite logits give an
 * unspecified selection.  Errors as for the layer. */
MM_MOE_API mm_moe_status mm_moe_router_forward(const mm_moe_shape* shape, const uint16_t* x,
                                               const uint16_t* W_router, float* logits,
                                               int32_t* topk_idx, float* topk_w, void* stream);

/*   dtopk_w   [T, k] fp32: gradient of topk_w (mm_moe_backward's dtopk_w)
 *   dlogits   [T, E] bf16 out: the logit gradient w_j (g_j - sum_i w_i g_i) at the
 *             chosen experts, zero elsewhere (rounded to bf16 for the GEMMs)
 *   dx        [T, H] bf16 in/out: the router's input gradient dlogits W_router is
 *             ADDED (fp32 sum of the bf16 value and the product, rounded to bf16),
 *             so the layer's dx can be passed straight in
 *   dW_router [E, H] bf16 out: dlogits^T x */
MM_MOE_API mm_moe_status mm_moe_router_backward(const mm_moe_shape* shape, const uint16_t* x,
                                                const uint16_t* W_router,
                                                const int32_t* topk_idx, const float* topk_w,
                                                const float* dtopk_w, uint16_t* dlogits,
                                                uint16_t* dx, uint16_t* dW_router, void* stream);

/* MXFP8 quantise-dequantise of a bf16 matrix, the operation the MXFP8 modes apply
 * to every GEMM operand (OCP Microscaling v1.0 MXFP8: blocks of 32 elements share
 * the power-of-two scale 2^(floor(log2 amax) - 8), 2^-127 for an all-zero block;
 * each element is rounded to e4m3, nearest even, saturating at +-448).  The Prime
 * Mega MoE pages name MXFP8 as the Blackwell precision (section "How does the
 * fused kernel work?") but give no standalone quantiser; this one is exported
 * for callers that keep MXFP8 copies of their own tensors.
 *   in, out  [rows, cols] bf16, device, 16-byte aligned; out may equal in
 *   axis     1: blocks along each row (cols % 32 == 0);
 *            0: blocks down each column (rows % 32 == 0, cols % 8 == 0)
 * out holds e4m3 * scale, exact in bf16 while it is at least 2^-133 (smaller
 * values are rounded to bf16).  Returns MM_MOE_EINVAL for bad sizes or pointers
 * (before any work is enqueued), MM_MOE_ENOTSUP off sm_103, MM_MOE_ECUDA for a
 * failed launch. */
MM_MOE_API mm_moe_status mm_moe_mx_qdq(const uint16_t* in, uint16_t* out, int64_t rows,
                                       int64_t cols, int axis, void* stream);

/* MXFP8 quantisation of a bf16 matrix into the form the MXFP8 modes' GEMMs read on
 * the block-scaled tensor cores (tcgen05.mma kind::mxf8f6f4.block_scale): e4m3 codes
 * and E8M0 scale codes (2^e stored as e + 127), with the block rule of mm_moe_mx_qdq
 * (the Prime Mega MoE pages' Blackwell precision, section "How does the fused kernel
 * work?"); exported for callers that keep MXFP8 copies of their own tensors.
 *   in      [rows, cols] bf16 device; rows % 128 == 0, cols % 128 == 0
 *   codes   [rows, cols] uint8 device out: the e4m3 code of each element
 *   scales  rows * cols / 32 uint8 device out: the scale code of each block.  Call the
 *           rows of the GEMM operand mn (for axis 1 the matrix rows, for axis 0 its
 *           columns) and the 32-element blocks along K kb; the code of (mn, kb) is at
 *           byte ((kb / 4) * (MN / 128) + mn / 128) * 512 + (mn % 32) * 16
 *           + ((mn / 32) % 4) * 4 + kb % 4, MN being the number of operand rows
 *           (512-byte atoms of 128 rows x 4 blocks, as the tensor cores take them).
 *   axis    1: blocks along each row; 0: blocks of 32 rows down each column
 * All pointers 16-byte aligned.  Errors as for mm_moe_mx_qdq. */
MM_MOE_API mm_moe_status mm_moe_mx_quantize(const uint16_t* in, uint8_t* codes,
                                            uint8_t* scales, int64_t rows, int64_t cols,
                                            int axis, void* stream);

/* Blockwise FP8 quantise-dequantise of a bf16 matrix, the operation
 * MM_MOE_FP8_BLOCK applies to every GEMM operand: one power-of-two scale
 * 2^ceil(log2(amax / 448)) per block (2^-127 for an all-zero block), elements
 * rounded to e4m3 (nearest even); exported for callers that keep such copies of
 * their own tensors.
 *   in, out  [rows, cols] bf16, device, 16-byte aligned; out may equal in
 *   layout   0: 128-element blocks along each row (cols % 128 == 0);
 *            1: 128-element blocks down each column (rows % 128 == 0, cols % 8 == 0);
 *            2: 128 x 128 tiles (rows % 128 == 0, cols % 128 == 0)
 * Errors as for mm_moe_mx_qdq. */
MM_MOE_API mm_moe_status mm_moe_fp8_block_qdq(const uint16_t* in, uint16_t* out,
                                              int64_t rows, int64_t cols, int layout,
                                              void* stream);

/* Blockwise FP8 quantisation of a bf16 matrix into the form MM_MOE_FP8_BLOCK's GEMMs
 * read on the block-scaled tensor cores: e4m3 codes and E8M0 scale codes (2^e stored
 * as e + 127), with the block rule of mm_moe_fp8_block_qdq (the pages' Hopper
 * precision, section "How does the fused kernel work?"), each 128-element block's
 * scale code repeated over its four 32-element scale blocks; exported for callers
 * that keep such copies of their own tensors.
 *   in      [rows, cols] bf16 device; rows % 128 == 0, cols % 128 == 0
 *   codes   [rows, cols] uint8 device out: the e4m3 code of each element
 *   scales  uint8 device out, in the atom arrangement of mm_moe_mx_quantize: layout 0
 *           rows * cols / 32 bytes, the matrix rows as the operand rows; layout 1 the
 *           same size, the columns as the operand rows; layout 2 twice that, first the
 *           rows then the columns as the operand rows (the codes serve both)
 *   layout  0: 128-element blocks along each row; 1: blocks of 128 rows down each
 *           column; 2: 128 x 128 tiles
 * All pointers 16-byte aligned.  Errors as for mm_moe_mx_qdq. */
MM_MOE_API mm_moe_status mm_moe_fp8_block_quantize(const uint16_t* in, uint8_t* codes,
                                                   uint8_t* scales, int64_t rows, int64_t cols,
                                                   int layout, void* stream);

/* Synchronises `stream`, then returns the device status word of `scratch`
 * (MM_MOE_OK, MM_MOE_EBADIDX or MM_MOE_ETIMEOUT), or MM_MOE_ECUDA when the
 * synchronisation itself fails.  The only blocking call of the library. */
MM_MOE_API mm_moe_status mm_moe_read_status(const void* scratch, void* stream);

/* Token routing that allocates nothing and takes no scratch buffer.  The source
 * pages have no counterpart to this entry point: it exists for callers that cannot
 * allocate device memory when they route tokens (runtimes without a device
 * allocator, processes whose memory pool belongs to another component, code that
 * must not meet an out-of-memory failure on this path).
 *   shape->T, k, E   as for mm_moe_forward (H, I and prec are ignored);
 *                    limits: T * k <= 262144, E <= 256, k <= E
 *   topk_idx [T, k]  int32 device, topk_w [T, k] fp32 device (inputs)
 *   offsets [E+1], perm [T*k], inv [T*k]  int32 device outputs, the same values
 *                    mm_moe_get_routing returns after mm_moe_forward
 * Its working memory is one fixed 4 MiB array in the library's device image:
 * every GPU that loads the library holds it until the process exits, and every
 * call shares it, so calls that overlap on the GPU (other streams, other host
 * threads) race and must be serialised by the caller.  The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture.  Pairs whose expert
 * index is outside [0, E) are dropped: their inv is -1, offsets[E] (the routed
 * rows) is then below T * k and perm[offsets[E] .. T*k) is left unwritten.  This
 * is the only report of such pairs: the call has no status word a caller can read
 * (mm_moe_read_status reads a caller's scratch, which this call does not take).
 * Returns MM_MOE_EINVAL for sizes beyond the limits or NULL / misaligned
 * pointers, MM_MOE_ENOTSUP off sm_103, MM_MOE_ECUDA for a failed CUDA call.
 * Enqueues on `stream` and returns without synchronising. */
MM_MOE_API mm_moe_status mm_moe_route_noalloc(const mm_moe_shape* shape,
                                              const int32_t* topk_idx, const float* topk_w,
                                              int32_t* offsets, int32_t* perm, int32_t* inv,
                                              void* stream);

/* Number of kernels the last successful mm_moe_forward / mm_moe_backward call
 * on this host thread enqueued (for launch accounting). */
MM_MOE_API int mm_moe_last_launch_count(void);

/* Optional per-kernel timing (tracing aid; the pages describe none).
 * mm_moe_profile_start clears the totals and, until mm_moe_profile_stop, makes
 * every forward/backward call on this host thread record a CUDA event before and
 * after each kernel it enqueues (on the call's stream).  mm_moe_profile_stop
 * synchronises those events and writes, for kernel id i < n, the summed
 * milliseconds total_ms[i] and the number of launches launches[i] (either array
 * may be NULL).  Ids run from 0 to mm_moe_kernel_count()-1; mm_moe_kernel_name(i)
 * names them (static strings, NULL for an unknown id).  Returns MM_MOE_ECUDA if
 * an event could not be read. */
MM_MOE_API mm_moe_status mm_moe_profile_start(void);
MM_MOE_API mm_moe_status mm_moe_profile_stop(float* total_ms, int* launches, int n);
MM_MOE_API const char* mm_moe_kernel_name(int id);
MM_MOE_API int mm_moe_kernel_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MM_MOE_H */

// gemm_fp8.cu -- the MXFP8 instantiations of the expert GEMM template (gemm.cuh):
// e4m3 operands with E8M0 block scales on tcgen05.mma.kind::mxf8f6f4.block_scale.
// Tiles: gate/up 256 wide (its 128 gate and 128 up rows); the others 256 wide where
// the output dimension allows, else 128; SM pairs where the padded layout has them
// and, for M/N-major operands, where the tile is 256 wide (a CTA's 128 columns).
#include "gemm.cuh"

namespace mmmoe {
namespace gemm {

cudaError_t run_fp8(const Ctx& c, const GemmParams& p, int kind, int bn, int ctas,
                    int64_t max_units) {
#define MMMOE_RUN(K, B, N) \
  if (kind == K && bn == B && ctas == N) return run<K, B, N, true>(c, p, max_units);
  MMMOE_RUN(GEMM_GATEUP, 256, 2)
  MMMOE_RUN(GEMM_GATEUP, 256, 1)
  MMMOE_RUN(GEMM_DOWN, 256, 2)
  MMMOE_RUN(GEMM_DOWN, 128, 2)
  MMMOE_RUN(GEMM_DOWN, 256, 1)
  MMMOE_RUN(GEMM_DOWN, 128, 1)
  MMMOE_RUN(GEMM_DGRAD_DOWN, 256, 2)
  MMMOE_RUN(GEMM_DGRAD_DOWN, 256, 1)
  MMMOE_RUN(GEMM_DGRAD_DOWN, 128, 1)
  MMMOE_RUN(GEMM_DGRAD_GATEUP, 256, 2)
  MMMOE_RUN(GEMM_DGRAD_GATEUP, 256, 1)
  MMMOE_RUN(GEMM_DGRAD_GATEUP, 128, 1)
  MMMOE_RUN(GEMM_WGRAD_DOWN, 256, 2)
  MMMOE_RUN(GEMM_WGRAD_DOWN, 256, 1)
  MMMOE_RUN(GEMM_WGRAD_DOWN, 128, 1)
  MMMOE_RUN(GEMM_WGRAD_GATEUP, 256, 2)
  MMMOE_RUN(GEMM_WGRAD_GATEUP, 256, 1)
  MMMOE_RUN(GEMM_WGRAD_GATEUP, 128, 1)
  MMMOE_RUN(GEMM_WGRAD_BOTH, 256, 2)
  MMMOE_RUN(GEMM_WGRAD_BOTH, 256, 1)
  MMMOE_RUN(GEMM_WGRAD_BOTH, 128, 1)
#undef MMMOE_RUN
  return cudaErrorInvalidValue;
}

}  // namespace gemm
}  // namespace mmmoe

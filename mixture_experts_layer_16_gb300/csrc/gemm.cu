// gemm.cu -- host side of the expert GEMMs: the tensor maps and tile counts of each
// kind, the choice of tile width and of single SMs or SM pairs, and the bf16
// instantiations of the kernel template in gemm.cuh (the MXFP8 ones are in
// gemm_fp8.cu).
#include "gemm.cuh"

namespace mmmoe {

using gemm::GemmParams;

int pick_bn(int64_t n) {
  if (n % 256 == 0) return 256;
  if (n % 128 == 0) return 128;
  return 64;
}

bool wgrad_both_ok(const Layout& L) {
  const int bn = pick_bn(L.H);
  return bn >= 128 && pick_bn(L.I) == bn;
}

namespace gemm {

cudaError_t run_bf16(const Ctx& c, const GemmParams& p, int kind, int bn, int ctas,
                     int64_t max_units, bool mc) {
  if (mc) {
    if (ctas != 2 || bn != 256) return cudaErrorInvalidValue;
    switch (kind) {
      case GEMM_GATEUP: return run<GEMM_GATEUP, 256, 2, false, true>(c, p, max_units);
      case GEMM_DOWN: return run<GEMM_DOWN, 256, 2, false, true>(c, p, max_units);
      case GEMM_DGRAD_DOWN: return run<GEMM_DGRAD_DOWN, 256, 2, false, true>(c, p, max_units);
      case GEMM_DGRAD_GATEUP: return run<GEMM_DGRAD_GATEUP, 256, 2, false, true>(c, p, max_units);
      default: return cudaErrorInvalidValue;
    }
  }
#define MMMOE_RUN(K, B, N) \
  if (kind == K && bn == B && ctas == N) return run<K, B, N, false>(c, p, max_units);
  MMMOE_RUN(GEMM_GATEUP, 256, 2)
  MMMOE_RUN(GEMM_DOWN, 256, 2)
  MMMOE_RUN(GEMM_DGRAD_DOWN, 256, 2)
  MMMOE_RUN(GEMM_DGRAD_DOWN, 128, 2)
  MMMOE_RUN(GEMM_DGRAD_GATEUP, 256, 2)
  MMMOE_RUN(GEMM_WGRAD_DOWN, 256, 2)
  MMMOE_RUN(GEMM_WGRAD_DOWN, 128, 2)
  MMMOE_RUN(GEMM_WGRAD_GATEUP, 256, 2)
  MMMOE_RUN(GEMM_WGRAD_BOTH, 256, 2)
  MMMOE_RUN(GEMM_WGRAD_BOTH, 128, 2)
  MMMOE_RUN(GEMM_GATEUP, 256, 1)
  MMMOE_RUN(GEMM_GATEUP, 128, 1)
  MMMOE_RUN(GEMM_DOWN, 256, 1)
  MMMOE_RUN(GEMM_DOWN, 128, 1)
  MMMOE_RUN(GEMM_DGRAD_DOWN, 256, 1)
  MMMOE_RUN(GEMM_DGRAD_DOWN, 128, 1)
  MMMOE_RUN(GEMM_DGRAD_DOWN, 64, 1)
  MMMOE_RUN(GEMM_DGRAD_GATEUP, 256, 1)
  MMMOE_RUN(GEMM_DGRAD_GATEUP, 128, 1)
  MMMOE_RUN(GEMM_WGRAD_DOWN, 256, 1)
  MMMOE_RUN(GEMM_WGRAD_DOWN, 128, 1)
  MMMOE_RUN(GEMM_WGRAD_DOWN, 64, 1)
  MMMOE_RUN(GEMM_WGRAD_GATEUP, 256, 1)
  MMMOE_RUN(GEMM_WGRAD_GATEUP, 128, 1)
  MMMOE_RUN(GEMM_WGRAD_BOTH, 256, 1)
  MMMOE_RUN(GEMM_WGRAD_BOTH, 128, 1)
#undef MMMOE_RUN
  return cudaErrorInvalidValue;
}

}  // namespace gemm

// Dense products on single-SM 128 x 128 tiles, 128 x 64 for A^T.B (its output, E x H for
// the router's weight gradient, has few tiles and a long K: narrower tiles double the
// SMs at work), bf16 in, fp32 accumulation; the tensor maps cover exactly M, N, K, so
// ragged tiles read zeros past the edges and the bf16 stores are clipped there (the
// fp32 epilogue masks them).
cudaError_t launch_dense(const Ctx& c, int kind, const uint16_t* A, const uint16_t* B, void* C,
                         int64_t M, int64_t N, int64_t K) {
  using namespace gemm;
  // (the inner dimension of every operand and of the output: rows of 16-byte multiples)
  const bool inner_ok = kind == GEMM_DENSE_TN ? (M % 8 == 0 && N % 8 == 0)
                                              : (K % 8 == 0 && N % 8 == 0);
  if (M < 1 || N < 1 || K < 1 || !inner_ok || M >= (int64_t{1} << 31) ||
      N >= (int64_t{1} << 31) || K >= (int64_t{1} << 31))
    return cudaErrorInvalidValue;
  const int BN = kind == GEMM_DENSE_TN ? 64 : 128;
  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.dm = static_cast<int>(M);
  p.dn = static_cast<int>(N);
  p.m_tiles = static_cast<int>((M + BM - 1) / BM);
  p.n_tiles = static_cast<int>((N + BN - 1) / BN);
  p.k_iters = static_cast<int>((K + BK - 1) / BK);
  const uint64_t m = M, n = N, k = K;
  bool ok = false;
  switch (kind) {
    case GEMM_DENSE_NT:  // A [M, K], B [N, K], C [M, N] fp32
      ok = make_map(&p.tmA, A, k, m, 64, BM) && make_map(&p.tmB0, B, k, n, 64, 128);
      p.outf = static_cast<float*>(C);
      break;
    case GEMM_DENSE_NN:  // A [M, K], B [K, N], C [M, N] bf16 (read and written)
      ok = make_map(&p.tmA, A, k, m, 64, BM) && make_map(&p.tmB0, B, n, k, 64, 64) &&
           make_epi_map(&p.tmC0, C, n, m) && make_epi_map(&p.tmD0, C, n, m);
      break;
    case GEMM_DENSE_TN:  // A [K, M], B [K, N], C [M, N] bf16
      ok = make_map(&p.tmA, A, m, k, 64, 64) && make_map(&p.tmB0, B, n, k, 64, 64) &&
           make_epi_map(&p.tmC0, C, n, m);
      p.out0 = static_cast<uint16_t*>(C);
      {
        // few tiles and a long K (the router's E x H weight gradient, K = tokens): split
        // K over a cluster of 2, 4 or 8 CTAs, at least 8 K iterations each, to put about
        // every SM to work; the partial tiles are summed in the cluster's shared memory
        const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
        int ks = 1;
        while (ks < 8 && tiles * ks * 2 <= c.num_sms && p.k_iters >= 8 * ks * 2) ks *= 2;
        p.ksplit = ks;
        p.kper = (p.k_iters + ks - 1) / ks;
      }
      break;
    default:
      return cudaErrorInvalidValue;
  }
  if (!ok) return cudaErrorInvalidValue;
  const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
  switch (kind) {
    case GEMM_DENSE_NT: return run<GEMM_DENSE_NT, 128, 1, false>(c, p, tiles);
    case GEMM_DENSE_NN: return run<GEMM_DENSE_NN, 128, 1, false>(c, p, tiles);
    default: return run<GEMM_DENSE_TN, 64, 1, false>(c, p, tiles);
  }
}

cudaError_t launch_gemm(const Ctx& c, const Layout& L, const GemmArgs& g) {
  using namespace gemm;
  GemmParams p;
  memset(&p, 0, sizeof(p));
  const char* saved = g.saved;
  const bool f8 = g.fp8;
  // SM pairs where the layout allows them; the weight-gradient GEMMs (K = an
  // expert's rows) go back to single-SM tiles when experts average fewer than
  // WGRAD_PAIR_MIN_ROWS rows: their short main loops leave pair tiles waiting on
  // each other and on the epilogue (4k-token 30B-shape layer: 0.52 ms on pairs,
  // 0.42 ms on single SMs; 16k tokens: pairs 5 % faster)
  constexpr int64_t WGRAD_PAIR_MIN_ROWS = 512;
  const bool per_expert = g.kind >= GEMM_WGRAD_DOWN;
  int ctas = (L.pad == 2 * BM && !(per_expert && L.R < WGRAD_PAIR_MIN_ROWS * L.E)) ? 2 : 1;
  p.H = static_cast<int>(L.H);
  p.I = static_cast<int>(L.I);
  p.E = static_cast<int>(L.E);
  p.n_pw = static_cast<int>(L.n_pw);
  p.max_tiles = static_cast<int>(L.NT);
  p.meta = reinterpret_cast<const int*>(saved + L.meta);
  p.tile_expert = reinterpret_cast<const int*>(saved + L.tile_expert);
  p.tile_rows = reinterpret_cast<const int*>(saved + L.tile_rows);
  p.pad_off = reinterpret_cast<const int*>(saved + L.pad_off);
  p.counts = reinterpret_cast<const int*>(saved + L.counts);
  p.expert_order = reinterpret_cast<const int*>(saved + L.expert_order);
  p.rowflat = reinterpret_cast<const int*>(saved + L.rowflat);
  p.w_row = reinterpret_cast<const float*>(saved + L.w_row);
  p.out0 = g.out0;
  p.out1 = g.out1;
  p.outf = g.outf;
  p.status = reinterpret_cast<DevStatus*>(g.scratch + L.status);
  // Failure-path test hook: MM_MOE_TEST_STALL_GEMM=<kind> makes that GEMM's first
  // stage on CTA 0 never fill (read at every launch; unset, it does nothing)
  if (const char* v = std::getenv("MM_MOE_TEST_STALL_GEMM"))
    p.stall = (v[0] >= '0' && v[0] <= '6' && v[1] == '\0' && v[0] - '0' == g.kind) ? 1 : 0;
  const uint64_t Rp = static_cast<uint64_t>(L.Rp), H = L.H, I = L.I, E = L.E;
  // operand maps: bf16 (64-element K boxes, 64-wide M/N-major boxes) or e4m3 codes
  // (128-element K boxes, 128-wide M/N-major boxes); box_rows = rows of a K-major box
  auto kmaj = [&](CUtensorMap* m, const void* base, uint64_t K, uint64_t rows,
                  uint32_t box_rows) {
    return f8 ? make_fp8_map(m, base, K, rows, box_rows)
              : make_map(m, base, K, rows, 64, box_rows);
  };
  auto mnmaj = [&](CUtensorMap* m, const void* base, uint64_t MN, uint64_t krows) {
    return f8 ? make_fp8_map(m, base, MN, krows, 128) : make_map(m, base, MN, krows, 64, 64);
  };
  // scale map of an operand with MN rows and K columns (fp8 only)
  auto sfm = [&](CUtensorMap* m, const uint8_t* base, uint64_t MN, uint64_t K) {
    return !f8 || make_sf_map(m, base, MN * K / 32);
  };
  const int kstep = f8 ? 128 : BK;
  bool ok = true;
  int bn = 0;
  int64_t max_units = 0;  // tiles (of both CTAs of a pair) that exist at most
  switch (g.kind) {
    case GEMM_GATEUP:
      bn = (f8 || L.I % 128 == 0) ? 256 : 128;
      ok = kmaj(&p.tmA, g.A, H, Rp, BM) && kmaj(&p.tmB0, g.B0, H, E * I, bn / 2) &&
           kmaj(&p.tmB1, g.B1, H, E * I, bn / 2) && make_epi_map(&p.tmC0, g.out0, 2 * I, Rp) &&
           make_epi_map(&p.tmC1, g.out1, I, Rp) && sfm(&p.tmSA, g.sA, Rp, H) &&
           sfm(&p.tmSB0, g.sB0, E * I, H) && sfm(&p.tmSB1, g.sB1, E * I, H);
      p.sfa_mnb = static_cast<int>(Rp / 128);
      p.sfb_mnb = static_cast<int>(E * I / 128);
      p.q_codes = g.q_codes;
      p.q_sf = g.q_sf;
      p.q_mnb = static_cast<int>(Rp / 128);
      p.n_tiles = static_cast<int>(L.I / (bn / 2));
      p.k_iters = static_cast<int>(L.H / kstep);
      max_units = L.NT / ctas * p.n_tiles;
      break;
    case GEMM_DOWN:
      bn = pick_bn(L.H);
      ok = kmaj(&p.tmA, g.A, I, Rp, BM) && kmaj(&p.tmB0, g.B0, I, E * H, bn / ctas) &&
           make_epi_map(&p.tmC0, g.out0, H, Rp) && sfm(&p.tmSA, g.sA, Rp, I) &&
           sfm(&p.tmSB0, g.sB0, E * H, I);
      p.sfa_mnb = static_cast<int>(Rp / 128);
      p.sfb_mnb = static_cast<int>(E * H / 128);
      p.n_tiles = static_cast<int>(L.H / bn);
      p.k_iters = static_cast<int>(L.I / kstep);
      max_units = L.NT / ctas * p.n_tiles;
      break;
    case GEMM_DGRAD_DOWN:
      bn = pick_bn(L.I);
      if (f8 && bn != 256) ctas = 1;  // M/N-major e4m3 boxes are 128 wide per CTA
      ok = kmaj(&p.tmA, g.A, H, Rp, BM) && mnmaj(&p.tmB0, g.B0, I, E * H) &&
           make_epi_map(&p.tmC0, g.out0, 2 * I, Rp) && make_epi_map(&p.tmC1, g.out1, I, Rp) &&
           make_epi_map(&p.tmD0, g.aux, 2 * I, Rp) && make_epi_map(&p.tmD1, g.aux2, I, Rp) &&
           sfm(&p.tmSA, g.sA, Rp, H) && sfm(&p.tmSB0, g.sB0, I, E * H);
      p.sfa_mnb = static_cast<int>(Rp / 128);
      p.sfb_mnb = static_cast<int>(I / 128);
      p.n_tiles = static_cast<int>(L.I / bn);
      p.k_iters = static_cast<int>(L.H / kstep);
      max_units = L.NT / ctas * p.n_tiles;
      break;
    case GEMM_DGRAD_GATEUP:
      bn = pick_bn(L.H);
      if (f8 && bn != 256) ctas = 1;
      ok = kmaj(&p.tmA, g.A, 2 * I, Rp, BM) && mnmaj(&p.tmB0, g.B0, H, E * I) &&
           mnmaj(&p.tmB1, g.B1, H, E * I) && make_epi_map(&p.tmC0, g.out0, H, Rp) &&
           sfm(&p.tmSA, g.sA, Rp, 2 * I) && sfm(&p.tmSB0, g.sB0, H, E * I) &&
           sfm(&p.tmSB1, g.sB1, H, E * I);
      p.sfa_mnb = static_cast<int>(Rp / 128);
      p.sfb_mnb = static_cast<int>(H / 128);
      p.n_tiles = static_cast<int>(L.H / bn);
      p.k_iters = static_cast<int>(2 * L.I / kstep);
      max_units = L.NT / ctas * p.n_tiles;
      break;
    case GEMM_WGRAD_DOWN:
      bn = pick_bn(L.I);
      if (f8 && bn != 256) ctas = 1;
      ok = mnmaj(&p.tmA, g.A, H, Rp) && mnmaj(&p.tmB0, g.B0, I, Rp) &&
           make_epi_map(&p.tmC0, g.out0, I, E * H) && sfm(&p.tmSA, g.sA, H, Rp) &&
           sfm(&p.tmSB0, g.sB0, I, Rp);
      p.sfa_mnb = static_cast<int>(H / 128);
      p.sfb_mnb = static_cast<int>(I / 128);
      p.m_tiles = static_cast<int>(L.H / (BM * ctas));
      p.n_tiles = static_cast<int>(L.I / bn);
      max_units = L.E * p.m_tiles * p.n_tiles;
      break;
    case GEMM_WGRAD_GATEUP:
      bn = pick_bn(L.H);
      if (f8 && bn != 256) ctas = 1;
      ok = mnmaj(&p.tmA, g.A, 2 * I, Rp) && mnmaj(&p.tmB0, g.B0, H, Rp) &&
           make_epi_map(&p.tmC0, g.out0, H, E * I) && make_epi_map(&p.tmC1, g.out1, H, E * I) &&
           sfm(&p.tmSA, g.sA, 2 * I, Rp) && sfm(&p.tmSB0, g.sB0, H, Rp);
      p.sfa_mnb = static_cast<int>(2 * I / 128);
      p.sfb_mnb = static_cast<int>(H / 128);
      p.m_tiles = static_cast<int>(2 * L.I / (BM * ctas));
      p.n_tiles = static_cast<int>(L.H / bn);
      max_units = L.E * p.m_tiles * p.n_tiles;
      break;
    case GEMM_WGRAD_BOTH:
      if (!wgrad_both_ok(L)) return cudaErrorInvalidValue;
      bn = pick_bn(L.H);
      if (f8 && bn != 256) ctas = 1;
      ok = mnmaj(&p.tmA, g.A, 2 * I, Rp) && mnmaj(&p.tmB0, g.B0, H, Rp) &&
           make_epi_map(&p.tmC0, g.out0, H, E * I) && make_epi_map(&p.tmC1, g.out1, H, E * I) &&
           mnmaj(&p.tmA2, g.A2, H, Rp) && mnmaj(&p.tmB2, g.B2, I, Rp) &&
           make_epi_map(&p.tmC2, g.out2, I, E * H) && sfm(&p.tmSA, g.sA, 2 * I, Rp) &&
           sfm(&p.tmSB0, g.sB0, H, Rp) && sfm(&p.tmSA2, g.sA2, H, Rp) &&
           sfm(&p.tmSB2, g.sB2, I, Rp);
      p.sfa_mnb = static_cast<int>(2 * I / 128);
      p.sfb_mnb = static_cast<int>(H / 128);
      p.sfa2_mnb = static_cast<int>(H / 128);
      p.sfb2_mnb = static_cast<int>(I / 128);
      p.m_tiles = static_cast<int>(2 * L.I / (BM * ctas));
      p.n_tiles = static_cast<int>(L.H / bn);
      p.m_tiles2 = static_cast<int>(L.H / (BM * ctas));
      p.n_tiles2 = static_cast<int>(L.I / bn);
      max_units = L.E * (p.m_tiles * p.n_tiles + p.m_tiles2 * p.n_tiles2);
      {
        // bf16 pairs: when an expert's tiles nearly fill the resident clusters, launch
        // exactly that many clusters, so that cluster j takes tile j of every expert
        // (equal K, so equal work, and each expert's operands streamed once, by all of
        // its tiles at the same time); the joint launch of the 16k-token 30B-shape
        // layer: 72 tiles an expert, 0.873 -> 0.848 ms on 72 of 76 clusters (the MXFP8
        // one ran slower that way, 0.642 -> 0.660)
        const int64_t per_e = p.m_tiles * p.n_tiles + p.m_tiles2 * p.n_tiles2;
        const int64_t pairs = c.num_sms / 2;
        if (!f8 && ctas == 2 && per_e <= pairs && 10 * per_e >= 9 * pairs) max_units = per_e;
      }
      break;
    default:
      return cudaErrorInvalidValue;
  }
  if (!ok) return cudaErrorInvalidValue;
  // MM_MOE_MULTICAST: bf16 grouped GEMMs on SM pairs with 256-wide tiles and an even
  // number of N tiles run on clusters of two pairs that share each M tile's A rows by
  // multicast (half the A reads from L2)
  const bool mc = L.multicast && !f8 && ctas == 2 && bn == 256 &&
                  g.kind <= GEMM_DGRAD_GATEUP && p.n_tiles >= 2 && p.n_tiles % 2 == 0;
  if (mc) {
    const uint64_t ka = g.kind == GEMM_DOWN ? I : g.kind == GEMM_DGRAD_GATEUP ? 2 * I : H;
    if (!kmaj(&p.tmA_half, g.A, ka, Rp, BM / 2)) return cudaErrorInvalidValue;
    max_units /= 2;
  }
  return f8 ? run_fp8(c, p, g.kind, bn, ctas, max_units)
            : run_bf16(c, p, g.kind, bn, ctas, max_units, mc);
}

}  // namespace mmmoe

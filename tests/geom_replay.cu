// Host replay of the decode kernel's launch plan (test infrastructure).
//
// Includes the decode source itself so that the kernel's own plan functions
// (make_geom, layout) run on the host, for every M in 1..32 of one shape, and
// checks what the kernel's indexing relies on:
//   * the shared-memory plan fits the budget and its regions are ordered and
//     do not overlap where they are live at the same time;
//   * the CTAs' channel slices (COMBINE, down products) cover every
//     (stream, channel) exactly once, and their mix ranges every channel once;
//   * the exchange buffers the handle allocates hold the plan's words;
//   * tensor-memory columns and issuer counts stay within their limits.
// Usage: geom_replay HC HS r sms smem_optin   -> one line per M, then "DONE".
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "../hyper_connection_gated_gb300/csrc/decode.cu"

namespace {

int fails = 0;

void check(bool ok, int M, const char* what) {
  if (!ok) {
    std::printf("FAIL M=%d %s\n", M, what);
    ++fails;
  }
}

}  // namespace

int main(int argc, char** argv) {
  if (argc != 6) {
    std::fprintf(stderr, "usage: geom_replay HC HS r sms smem_optin\n");
    return 2;
  }
  const int HC = std::atoi(argv[1]), HS = std::atoi(argv[2]), r = std::atoi(argv[3]);
  hcgr::Device dev;
  dev.sms = std::atoi(argv[4]);
  dev.smem_optin = std::atoi(argv[5]);
  const int n_out = r + HC;
  for (int M = 1; M <= hcgr::DECODE_MAX_M; ++M) {
    const hcgr::Call c = hcgr::shape_call(M, HC, HS, r);
    hcgr::Geom g;
    if (!hcgr::make_geom(c, dev, g)) {
      std::printf("M=%d plan=none\n", M);
      continue;
    }
    std::printf("M=%d plan G=%d P=%d nkc=%d ntd=%d nsl_w=%d nsl_u=%d ncu=%d Qn=%d Jm=%d total=%d tmem=%d\n",
                M, g.G, g.P, g.nkc, g.ntd, g.nsl_w, g.nsl_u, g.ncu, g.Qn, g.Jm, g.total, g.tmem_cols);
    // grid and budget
    check(g.G <= dev.sms && g.G <= hcgr::MAX_GRID, M, "grid beyond the SMs");
    check(g.total <= hcgr::SMEM_BUDGET && g.total + 1024 <= dev.smem_optin, M, "shared memory");
    check(g.tmem_cols <= 512 && g.tmem_cols >= g.ntd * g.Nd &&
              g.tmem_cols >= g.ncu * g.ntu * g.Nu, M, "tensor-memory columns");
    check(g.ntd <= hcgr::DOWN_ISSUERS && g.nchunk_u <= hcgr::UP_ISSUERS, M, "issuers");
    // region order: header arrays, operands, up slots, then region A
    check(g.off_act % 1024 == 0 && g.off_u % 1024 == 0 && g.off_a % 1024 == 0, M, "alignment");
    check(g.off_act + g.nkc * g.Nd * 128 <= g.off_u, M, "operands overlap the up slots");
    check(g.off_u + g.nsl_u * g.slot_u <= g.off_a, M, "up slots overlap region A");
    check(g.off_a + g.nsl_w * hcgr::TILE <= g.total, M, "down slots beyond the plan");
    check(g.off_u + (g.nsl_u - 1) * g.slot_u + g.ntu * hcgr::TILE <= g.total, M,
          "the last up slot's tile reads beyond the plan");
    check(g.off_hb + g.nchunk_u * g.Nu * 128 <= g.off_g, M, "h operand overlaps the gates");
    check(g.off_g + M * g.rows_u * 4 <= g.total, M, "gates beyond the plan");
    check(g.off_red + HC * g.row * 4 <= g.total, M, "reducer scratch beyond the plan");
    // exchanges
    check(g.Qn % 4 == 0 && g.Jm * g.Qn >= n_out && (M * g.Jm <= g.G || g.Jm == 1), M,
          "reduce-scatter blocks");
    check(g.row == g.Qn + 4 && g.nquad * 4 == g.row && g.nquad <= hcgr::NT, M, "block rows");
    check(static_cast<size_t>(g.nred) * g.G * g.row ==
              hcgr::decode_xred_words(dev, M, HC, HS, r), M, "reduce-scatter words");
    check(static_cast<size_t>(M) * g.L2w <= hcgr::decode_xgat_words(n_out) &&
              hcgr::decode_xgat_words(n_out) % 4 == 0 && g.L2w >= r / 2 + HC, M,
          "all-gather words");
    // coverage: COMBINE / down slices, then the mix ranges
    std::vector<int> seen(static_cast<size_t>(HC) * HS, 0), seen_mix(HS, 0);
    for (int b = 0; b < g.G; ++b) {
      const int s = b / g.P;
      const int c0 = (b % g.P) * 64 * g.nkc;
      const int nkv = std::min(g.nkc, (HS - c0) / 64);
      check(s < HC && c0 < HS && nkv >= 1, M, "empty slice");
      for (int k = 0; k < nkv * 64; ++k) ++seen[static_cast<size_t>(s) * HS + c0 + k];
      const int cp0 = std::min(HS, b * g.nc_max);
      const int nc = std::min(HS, cp0 + g.nc_max) - cp0;
      check(nc >= 0 && nc <= g.nc_max && nc % 2 == 0, M, "mix range");
      for (int k = 0; k < nc; ++k) ++seen_mix[cp0 + k];
    }
    bool once = true;
    for (int v : seen) once = once && v == 1;
    check(once, M, "slices do not cover every (stream, channel) once");
    once = true;
    for (int v : seen_mix) once = once && v == 1;
    check(once, M, "mix ranges do not cover every channel once");
  }
  std::printf("DONE fails=%d\n", fails);
  return fails == 0 ? 0 : 1;
}

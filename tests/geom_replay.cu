// Host replay of the decode kernel's launch plan (test infrastructure).
//
// Includes the decode source itself so that the kernel's own plan functions
// (make_geom, layout) run on the host, for every M in 1..32 of one shape, and
// checks what the kernel's indexing relies on:
//   * the shared-memory plan fits the budget and its regions are ordered and
//     do not overlap where they are live at the same time;
//   * the down CTAs' channel slices (COMBINE, down products) cover every
//     (stream, channel) exactly once, and the up CTAs' mix ranges every
//     channel once;
//   * weight rings keep each slot with one MMA issuer;
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
    std::printf("M=%d plan G=%d Gd=%d Gu=%d P=%d nkc=%d ntd=%d nsl_w=%d nc=%d ntu=%d nsl_u=%d ncu=%d "
                "Qn=%d Jm=%d total=%d tmem=%d/%d\n",
                M, g.G, g.Gd, g.Gu, g.P, g.nkc, g.ntd, g.nsl_w, g.nc_max, g.ntu, g.nsl_u, g.ncu, g.Qn,
                g.Jm, g.total, g.tmem_d, g.tmem_u);
    // grid and budget
    check(g.G == g.Gd + g.Gu && g.G <= dev.sms && g.G <= hcgr::MAX_GRID, M, "grid beyond the SMs");
    check(g.d_total <= hcgr::SMEM_BUDGET && g.u_total <= hcgr::SMEM_BUDGET &&
              g.total >= g.d_total && g.total >= g.u_total && g.total + 1024 <= dev.smem_optin &&
              g.total + 1024 >= hcgr::SMEM_MIN,
          M, "shared memory");
    check(g.tmem_d <= 512 && g.tmem_d >= g.ntd * g.Nd && g.tmem_u <= 512 &&
              g.tmem_u >= g.ncu * g.ntu * g.Nu, M, "tensor-memory columns");
    check(g.ntd <= hcgr::DOWN_ISSUERS && g.nchunk_u <= hcgr::UP_ISSUERS && g.ncu >= 1 &&
              g.ncu <= g.nchunk_u, M, "issuers");
    // rings: every slot of the down ring serves one issuer (its slot count a
    // multiple of its row tiles); every up slot feeds one accumulator copy,
    // read by one issuer per row tile
    const int nbox = g.ntd * g.nkc;
    check(g.nsl_w >= 1 && g.nsl_w <= hcgr::MAX_SLOTS && (g.nsl_w >= nbox || g.nsl_w % g.ntd == 0),
          M, "down ring");
    check(g.nsl_u >= 1 && g.nsl_u <= hcgr::MAX_SLOTS &&
              g.ncu * g.ntu <= hcgr::UP_ISSUERS &&
              (g.nsl_u >= g.nchunk_u ? g.ncu >= 1 && g.ncu <= g.nchunk_u : g.ncu == g.nsl_u),
          M, "up ring");
    // down role regions: header arrays, operands, weight slots
    check(g.d_ss1 >= hcgr::HDR && g.d_ssum >= g.d_ss1 + g.Nt * g.nkc * 8 * 4, M, "down header arrays");
    check(g.d_act % 1024 == 0 && g.d_act >= g.d_ssum + g.Nt * 4, M, "down operand alignment");
    check(g.d_w % 1024 == 0 && g.d_w >= g.d_act + g.nkc * g.Nd * 128, M, "operands overlap the slots");
    check(g.d_w + g.nsl_w * hcgr::TILE <= g.d_total, M, "down slots beyond the plan");
    // up role regions
    check(g.u_rr >= hcgr::HDR && g.u_iw >= g.u_rr + g.Nt * HC * 4 &&
              g.u_x3r >= g.u_iw + g.Nt * HC * 4 && g.u_x3y >= g.u_x3r + M * HC * g.nc_max * 2 &&
              g.u_x3w >= g.u_x3y + M * g.nc_max * 2 && g.u_rl >= g.u_x3w + HC * g.nc_max * 2 &&
              g.u_red >= g.u_rl + HC * 4 && g.u_g >= g.u_red + HC * g.row * 4 &&
              g.u_hb >= g.u_g + M * g.rows_u * 4, M, "up header arrays");
    check(g.u_hb % 1024 == 0 && g.u_u % 1024 == 0 && g.slot_u % 1024 == 0, M, "up alignment");
    check(g.u_u >= g.u_hb + g.nchunk_u * g.Nu * 128, M, "h operand overlaps the up slots");
    check(g.u_u + (g.nsl_u - 1) * g.slot_u + g.ntu * hcgr::TILE <= g.u_total, M,
          "the last up slot's tile reads beyond the plan");
    check(g.rows_u == HC * g.nc_max && g.ntu * 128 >= g.rows_u && g.slot_u >= g.rows_u * 128, M,
          "up rows");
    // exchanges
    check(g.Qn % 4 == 0 && g.Jm * g.Qn >= n_out && (M * g.Jm <= g.Gu || g.Jm == 1) &&
              g.Qn >= std::min(hcgr::QN_MIN, (n_out + 3) / 4 * 4) && g.Qn < n_out + 4, M,
          "reduce-scatter blocks");
    check(g.row == g.Qn + 4 && g.nquad * 4 == g.row && g.nquad <= hcgr::NT, M, "block rows");
    // (items beyond NT loop; sub-ranges of one (stream, quad) stay in one warp)
    check(g.R >= 1 && g.R <= 32 && (g.R & (g.R - 1)) == 0 &&
              (g.R == 1 || g.R * HC * g.nquad <= hcgr::NT) && g.ppr * g.R >= g.P, M,
          "reducer sub-ranges");
    check(static_cast<size_t>(g.nred) * g.Gd * g.row ==
              hcgr::decode_xred_words(dev, M, HC, HS, r), M, "reduce-scatter words");
    check(static_cast<size_t>(M) * g.L2w <= hcgr::decode_xgat_words(n_out) &&
              hcgr::decode_xgat_words(n_out) % 4 == 0 && g.L2w >= r / 2 + HC && g.L2w % 4 == 0 &&
              (r / 2) % 4 == 0, M, "all-gather words");
    // coverage: COMBINE / down slices, then the up CTAs' mix ranges
    std::vector<int> seen(static_cast<size_t>(HC) * HS, 0), seen_mix(HS, 0);
    for (int b = 0; b < g.Gd; ++b) {
      const int s = b / g.P;
      const int c0 = (b % g.P) * 64 * g.nkc;
      const int nkv = std::min(g.nkc, (HS - c0) / 64);
      check(s < HC && c0 < HS && nkv >= 1, M, "empty slice");
      for (int k = 0; k < nkv * 64; ++k) ++seen[static_cast<size_t>(s) * HS + c0 + k];
    }
    for (int u = 0; u < g.Gu; ++u) {
      const int cp0 = std::min(HS, u * g.nc_max);
      const int nc = std::min(HS, cp0 + g.nc_max) - cp0;
      check(nc > 0 && nc <= g.nc_max && nc % 2 == 0, M, "mix range");
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

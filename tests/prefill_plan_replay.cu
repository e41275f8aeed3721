// Host replay of the prefill kernels' launch plan (test infrastructure).
//
// Includes the prefill source so that its own plan functions (K chunks per
// stream, K2's channel block, the scratch size) run on the host, for a sweep
// of token counts of one shape, and checks what the kernels rely on:
//   * K chunks: S >= 1; with S > 1 the (tile, stream, chunk) CTAs fit one
//     wave and every chunk of the kernel's split holds at least two K blocks,
//     the chunks covering the stream's K blocks once;
//   * the scratch a call carves (partials, sums of squares, hh, 1 + Wnorm)
//     fits the bytes a handle allocates for that M, the launch's capacity
//     check accepts the call, and the allocation never shrinks as max_M grows;
//   * K2's channel block divides HS, keeps N = HC * NCU <= 256 and is halved
//     (HC = 4) only where the halved units fit one round over the SMs.
// Usage: prefill_plan_replay HC HS r sms   -> one line per M, then "DONE".
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "../hyper_connection_gated_gb300/csrc/prefill.cu"

namespace {

int fails = 0;

void check(bool ok, long long M, const char* what) {
  if (!ok) {
    std::printf("FAIL M=%lld %s\n", M, what);
    ++fails;
  }
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

int main(int argc, char** argv) {
  if (argc != 5) {
    std::fprintf(stderr, "usage: prefill_plan_replay HC HS r sms\n");
    return 2;
  }
  const int HC = std::atoi(argv[1]), HS = std::atoi(argv[2]), r = std::atoi(argv[3]);
  const int sms = std::atoi(argv[4]);
  const int nkb = HS / hcgr::BK;
  const int np = hcgr::k1_np(r, HC);
  std::vector<long long> Ms;
  for (long long M = 1; M <= 300; ++M) Ms.push_back(M);
  for (long long M : {383LL, 384LL, 385LL, 511LL, 512LL, 513LL, 1000LL, 1024LL, 2047LL, 2048LL,
                      2049LL, 2432LL, 4096LL, 8191LL, 8192LL, 16384LL, 32768LL, 65535LL, 65536LL,
                      65537LL, 100000LL})
    Ms.push_back(M);
  size_t prev_ws = 0;
  for (long long M : Ms) {
    const int n_mt = static_cast<int>((M + hcgr::BM - 1) / hcgr::BM);
    const int S = hcgr::k1_chunks(n_mt, HC, nkb, sms);
    check(S >= 1, M, "no K chunk");
    if (S > 1) check(static_cast<long long>(HC) * S * n_mt <= sms, M, "K1 chunks beyond one wave");
    // the kernel's split of a stream's K blocks: chunk c takes [c nkb / S, (c + 1) nkb / S)
    int covered = 0;
    for (int c = 0; c < S; ++c) {
      const int kb0 = c * nkb / S, kb1 = (c + 1) * nkb / S;
      check(kb0 == covered, M, "K chunks not contiguous");
      check(S == 1 || kb1 - kb0 >= 2, M, "a K chunk with fewer than two K blocks");
      covered = kb1;
    }
    check(covered == nkb, M, "K chunks do not cover the stream");
    // scratch: the launch's capacity check, and its carve against the allocation
    const size_t Mp = static_cast<size_t>(n_mt) * hcgr::BM;
    const size_t part = static_cast<size_t>(HC) * S * Mp * np;
    const size_t part_cap = std::max(static_cast<size_t>(HC) * Mp * np,
                                     static_cast<size_t>(2 * hcgr::MAX_GRID) * hcgr::BM * np);
    check(part <= part_cap, M, "partials beyond the launch's capacity check");
    const size_t sumsq = static_cast<size_t>(HC) * S * Mp;
    const size_t carve = align256(part * 4) + align256(sumsq * 4) +
                         align256(static_cast<size_t>(M) * r * 2) + static_cast<size_t>(HC) * HS * 4;
    const size_t ws = hcgr::prefill_ws_bytes(M, HC, HS, r);
    check(carve <= ws, M, "the call's scratch beyond the handle's allocation");
    check(ws >= prev_ws, M, "allocation shrinks as max_M grows");
    prev_ws = ws;
    // K2's channel block
    const int ncu = hcgr::k2_block(HC, n_mt, HS, sms);
    check(HS % ncu == 0 && HC * ncu <= 256 && ncu % 8 == 0, M, "K2 channel block");
    check(ncu == hcgr::k2_ncu(HC) ||
              (HC == 4 && ncu == 32 && static_cast<long long>(n_mt) * (HS / 32) <= sms),
          M, "K2 block halved outside one round");
    std::printf("M=%lld n_mt=%d S=%d ncu=%d part=%zu ws=%zu\n", M, n_mt, S, ncu, part, ws);
  }
  std::printf("DONE fails=%d\n", fails);
  return fails == 0 ? 0 : 1;
}

// Decode path of the HC gated residual: one cooperative persistent kernel for
// small token counts (M <= 32), where the time goes into streaming the
// weights once (aiter PR #5913, "Technical Details"; the page's skinny decode
// with split-K partials and a last-stage reduce is the prior art).
//
// Grid: G = HC * P CTAs (at most one per SM), three phases separated by two
// bounded grid barriers:
//   1. CTA b owns a channel slice [c0, c0 + w) of one stream s (every slice
//      has the same width w; the stream end clips the last one).  It forms
//      R2 = bf16(R + y * iw) for the slice (stored), the partial sum of R2^2
//      per token and, on the tensor cores (mma.sync bf16, fp32 accumulate),
//        part[b][m][n] = sum_{c in slice} a[m, c] * W[n, s * HS + c]
//      for all r + HC rows of the down and inject weights, with a = R2 *
//      (1 + Wnorm) split into two bf16 terms (hi + lo, ~16 mantissa bits) or
//      a = R2 for a folded weight.  Because rrms_s is constant over stream s,
//      lora = sum_b rrms_{s(b)} part[b] is exact: the per-stream factor
//      commutes out of the K-sum.
//   2. One TMA box brings CTA b's share of the outputs from every partial
//      (and the partial sums of squares) into shared memory: rrms, then lora
//      and inj_next as rrms-weighted sums in a fixed order (deterministic).
//   3. One bulk copy brings lora; h = SiLU(lora / HC) in bf16; the gates
//      G[s, c] = sigmoid(h . Wu[s * HS + c]) for the CTA's channel range and
//      all streams on the tensor cores; xn is rebuilt from R2 (recomputed
//      from R, y and inj prefetched at kernel start, bit-identical to phase
//      1), rrms and Wnorm; x = (1 / HC) sum_s G * xn is stored.
// Weights move as TMA boxes issued at kernel start: the down/inject slice as
// 3-D boxes (the stream is its own tensor dimension, so a box never crosses
// a stream end), the up-weight rows of the channel range as 3-D boxes with
// 128-byte swizzle (bank-conflict-free fragment loads).  When everything
// fits in shared memory the whole weight stream is in flight before the
// first barrier; otherwise both stream through two-slot rings.
#include <algorithm>

#include "hc_gr_internal.cuh"
#include "tmap.h"

namespace hcgr {
namespace {

constexpr int NT = 512;            // threads per CTA
constexpr int NW = NT / 32;
constexpr int MAX_SLOTS = 8;
constexpr int MAXP = 8;            // (row tile, token tile) pairs per warp in phase 3
constexpr int BOX_CAP = 32 * 1024; // bytes per down/inject weight box
constexpr int SMEM_BUDGET = 216 * 1024;
constexpr int SMEM_ALLOC = SMEM_BUDGET + 1024;

struct Geom {
  int MB;                                   // M rounded up to 8 (MMA token tiles)
  int G, P, w, nch_max;                     // phase 1: P slices of w channels per stream
  int nbox, rows_box, slot_w, nslot_w;      // down weight boxes
  int nc_max, rows_u, rows_u16, nchunk_u, slot_u, nslot_u;   // up weight chunks (64 columns)
  int Q, part_ld, ss_bytes;                 // phase 2
  int hstride;                              // bf16 elements per h row in shared memory
  int off_rr, off_iw, off_x3r, off_x3y, off_x3w, off_wi, off_u, off_un;
  int off_w, off_ahi, off_alo, off_ss1;     // phase 1 (union region)
  int off_pbox, off_ss;                     // phase 2 (union region)
  int off_red;                              // phase 2 (union region)
  int off_h, off_g;                         // phase 3 (union region)
  int total;
};

__host__ __device__ inline int round_up(int v, int a) { return (v + a - 1) / a * a; }

struct Params {
  CUtensorMap tm_wd;    // Wd as [r][HC][HS] (inner HS), box {w, 1, rows_box}
  CUtensorMap tm_wi;    // Wi as [HC][HC][HS], box {w, 1, HC}
  CUtensorMap tm_wu;    // Wu as [HC][HS][r] (inner r), box {64, nc_max, HC}, 128B swizzle
  CUtensorMap tm_part;  // partials [G][part_ld] fp32, box {Q, G}
  Call c;
  Geom g;
  float* part;
  float* sumsq;
  bf16_t* hdec;              // h = bf16(SiLU(lora / HC)), written in phase 2
  unsigned long long* bar;   // this grid size's barrier counter
  int* err;
  uint64_t limit_ns;
};

bool layout(const Call& c, Geom& g) {
  int off = 256;                                       // mbarriers + flag
  const int MB = g.MB;
  g.off_rr = off;   off += round_up(MB * c.HC * 4, 128);
  g.off_iw = off;   off += round_up(MB * c.HC * 4, 128);
  g.off_x3r = off;  off += round_up(MB * c.HC * g.nc_max * 2, 128);
  g.off_x3y = off;  off += round_up(MB * g.nc_max * 2, 128);
  g.off_x3w = off;  off += round_up(c.HC * g.nc_max * 2, 128);
  g.off_wi = off;   off += round_up(16 * g.w * 2, 128);
  off = round_up(off, 1024);
  g.off_u = off;    off += g.nslot_u * g.slot_u;
  g.off_un = off;
  // phase 1
  int p1 = off;
  g.off_w = p1;     p1 += g.nslot_w * g.slot_w;
  g.off_ahi = p1;   p1 += round_up(MB * g.w * 2, 128);
  g.off_alo = p1;   p1 += round_up(MB * g.w * 2, 128);
  g.off_ss1 = p1;   p1 += round_up(MB * g.nch_max * 4, 128);
  // phase 2
  int p2 = off;
  g.off_pbox = p2;  p2 += round_up(g.G * g.Q * 4, 128);
  g.off_ss = p2;    p2 += round_up(g.ss_bytes, 128);
  g.off_red = p2;   p2 += round_up(g.Q * c.HC * 4, 128);
  // phase 3
  int p3 = off;
  g.off_h = p3;     p3 += round_up(MB * g.hstride * 2, 128);
  g.off_g = p3;     p3 += round_up(MB * g.rows_u * 4, 128);
  g.total = std::max(p1, std::max(p2, p3));
  return g.total <= SMEM_BUDGET;
}

bool make_geom(const Call& c, const Device& dev, Geom& g) {
  const int M = static_cast<int>(c.M);
  g.MB = round_up(M, 8);
  const int P0 = std::max(1, dev.sms / c.HC);
  int w = round_up((c.HS + P0 - 1) / P0, 8);
  if (((w / 8) & 1) == 0 && w + 8 <= c.HS) w += 8;   // odd 16-byte units: no bank conflicts
  w = std::min(w, c.HS);
  if (w > 256) return false;
  g.w = w;
  g.P = (c.HS + w - 1) / w;
  g.G = c.HC * g.P;
  if (g.G > dev.sms) return false;
  g.nch_max = w / 8;
  g.nc_max = (c.HS + g.G - 1) / g.G;
  g.rows_u = c.HC * g.nc_max;
  g.rows_u16 = round_up(g.rows_u, 16);
  if (g.rows_u16 > 256 || (g.rows_u16 / 16) * (g.MB / 8) > NW * MAXP) return false;
  g.nchunk_u = (c.r + 63) / 64;
  g.slot_u = round_up(g.rows_u16 * 128, 1024);
  const int n_out = c.n_out;
  g.Q = round_up((M * n_out + g.G - 1) / g.G, 4);
  if (g.Q > 256) return false;
  g.part_ld = round_up(M * n_out, 4);
  g.ss_bytes = round_up(g.G * M * 4, 16);
  g.hstride = round_up(c.r, 8) + 8;
  // down weight boxes: rows a multiple of 16 (one MMA row tile never spans boxes)
  g.nbox = std::max(1, (c.r * w * 2 + BOX_CAP - 1) / BOX_CAP);
  g.rows_box = round_up((c.r + g.nbox - 1) / g.nbox, 16);
  while (g.rows_box > 256) {
    ++g.nbox;
    g.rows_box = round_up((c.r + g.nbox - 1) / g.nbox, 16);
  }
  g.nbox = (c.r + g.rows_box - 1) / g.rows_box;
  g.slot_w = round_up(g.rows_box * w * 2, 128);
  // everything resident when it fits, else two-slot rings
  g.nslot_w = g.nbox;
  g.nslot_u = g.nchunk_u;
  if (g.nbox <= MAX_SLOTS && g.nchunk_u <= MAX_SLOTS && layout(c, g)) return true;
  g.nslot_u = std::min(g.nchunk_u, 2);
  for (int rows = std::min(256, round_up(c.r, 16)); rows >= 16; rows -= 16) {
    g.rows_box = rows;
    g.nbox = (c.r + rows - 1) / rows;
    g.slot_w = round_up(rows * w * 2, 128);
    g.nslot_w = std::min(g.nbox, 2);
    if (layout(c, g)) return true;
  }
  return false;
}

__device__ __forceinline__ uint32_t lds32(const unsigned char* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

// --------------------------------------------------------------- the kernel
__global__ void __launch_bounds__(NT, 1) decode_kernel(const __grid_constant__ Params p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Call& c = p.c;
  const Geom& g = p.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, tq = lane & 3;       // MMA fragment coordinates
  const int b = blockIdx.x;
  const int M = static_cast<int>(c.M), MB = g.MB;
  const int HC = c.HC, HS = c.HS, K = c.K, r = c.r, n_out = c.n_out, w = g.w;
  const int ntok = MB / 8;

  int* s_flag = reinterpret_cast<int*>(smem + 240);
  float* s_rr = reinterpret_cast<float*>(smem + g.off_rr);     // [MB][HC]
  float* s_iw = reinterpret_cast<float*>(smem + g.off_iw);     // [MB][HC]
  bf16_t* s_x3r = reinterpret_cast<bf16_t*>(smem + g.off_x3r); // [M][HC][nc_max]
  bf16_t* s_x3y = reinterpret_cast<bf16_t*>(smem + g.off_x3y); // [M][nc_max]
  bf16_t* s_x3w = reinterpret_cast<bf16_t*>(smem + g.off_x3w); // [HC][nc_max]
  bf16_t* s_ahi = reinterpret_cast<bf16_t*>(smem + g.off_ahi); // [MB][w]
  bf16_t* s_alo = reinterpret_cast<bf16_t*>(smem + g.off_alo);
  float* s_ss1 = reinterpret_cast<float*>(smem + g.off_ss1);   // [MB][nch_max]
  float* s_pbox = reinterpret_cast<float*>(smem + g.off_pbox); // [G][Q]
  float* s_ss = reinterpret_cast<float*>(smem + g.off_ss);     // [G][M]
  float* s_red = reinterpret_cast<float*>(smem + g.off_red);   // [HC][Q]
  bf16_t* s_h = reinterpret_cast<bf16_t*>(smem + g.off_h);     // [MB][hstride]
  float* s_g = reinterpret_cast<float*>(smem + g.off_g);       // [MB][rows_u]

  // phase-1 slice and phase-3 channel range of this CTA
  const int s = b / g.P;
  const int c0 = (b % g.P) * w;
  const int nch = (min(HS, c0 + w) - c0) / 8;
  const int k0 = s * HS + c0;
  const int cp0 = min(HS, b * g.nc_max);
  const int nc = min(HS, cp0 + g.nc_max) - cp0;

  const uint32_t bar0 = smem_u32(smem);
  auto barW = [&](int i) { return bar0 + 8u * i; };               // slots 0..7
  auto barU = [&](int i) { return bar0 + 64u + 8u * i; };         // slots 8..15
  const uint32_t barWi = bar0 + 128u, barP = bar0 + 136u, barL = bar0 + 144u;

  if (tid == 0) {
    prefetch_tmap(&p.tm_wd);
    prefetch_tmap(&p.tm_wi);
    prefetch_tmap(&p.tm_wu);
    prefetch_tmap(&p.tm_part);
    for (int i = 0; i < 19; ++i) mbar_init(bar0 + 8u * i, 1);
    fence_mbar_init();
  }
  __syncthreads();

  auto issue_w = [&](int bx) {
    const int slot = bx % g.nslot_w;
    mbar_arrive_expect_tx(barW(slot), static_cast<uint32_t>(g.rows_box * w * 2));
    tma_load_3d(smem_u32(smem + g.off_w + slot * g.slot_w), &p.tm_wd, c0, s, bx * g.rows_box,
                barW(slot));
  };
  auto issue_u = [&](int q) {
    const int slot = q % g.nslot_u;
    mbar_arrive_expect_tx(barU(slot), static_cast<uint32_t>(g.rows_u * 128));
    tma_load_3d(smem_u32(smem + g.off_u + slot * g.slot_u), &p.tm_wu, q * 64, cp0, 0, barU(slot));
  };
  int issued_w = 0, issued_u = 0, done_w = 0, done_u = 0;   // uniform across the CTA
  for (; issued_w < g.nslot_w; ++issued_w)
    if (tid == 0) issue_w(issued_w);
  if (tid == 0) {
    mbar_arrive_expect_tx(barWi, static_cast<uint32_t>(HC * w * 2));
    tma_load_3d(smem_u32(smem + g.off_wi), &p.tm_wi, c0, s, 0, barWi);
  }
  if (nc > 0)
    for (; issued_u < g.nslot_u; ++issued_u)
      if (tid == 0) issue_u(issued_u);

  // --- phase 1a: COMBINE on this CTA's slice, R2 stored, MMA operands
  for (int it = tid; it < MB * g.nch_max; it += NT) {
    const int m = it / g.nch_max, ch = it % g.nch_max;
    uint4 hv = make_uint4(0, 0, 0, 0), lv = make_uint4(0, 0, 0, 0);
    float ss = 0.f;
    if (m < M && ch < nch) {
      const int64_t kk = static_cast<int64_t>(m) * K + k0 + ch * 8;
      const float iw = 2.0f * sigmoidf_dev(c.inj[m * c.ld_inj + s] / static_cast<float>(HC));
      float rv[8], yv[8], wv[8], a[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(c.R + kk)), rv);
      unpack8(__ldg(reinterpret_cast<const uint4*>(c.y + static_cast<int64_t>(m) * HS + c0 + ch * 8)), yv);
      unpack8(__ldg(reinterpret_cast<const uint4*>(c.Wnorm + k0 + ch * 8)), wv);
      uint32_t pr[4], ph[4], pl[4];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float r2 = bf16_to_f32(f32_to_bf16(fmaf(yv[i], iw, rv[i])));
        ss = fmaf(r2, r2, ss);
        rv[i] = r2;
        a[i] = c.fold ? r2 : r2 * (1.0f + wv[i]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        pr[i] = pack2(rv[2 * i], rv[2 * i + 1]);
        const float h0 = bf16_to_f32(f32_to_bf16(a[2 * i]));
        const float h1 = bf16_to_f32(f32_to_bf16(a[2 * i + 1]));
        ph[i] = pack2(h0, h1);
        pl[i] = pack2(a[2 * i] - h0, a[2 * i + 1] - h1);
      }
      *reinterpret_cast<uint4*>(c.R2 + kk) = make_uint4(pr[0], pr[1], pr[2], pr[3]);
      hv = make_uint4(ph[0], ph[1], ph[2], ph[3]);
      lv = make_uint4(pl[0], pl[1], pl[2], pl[3]);
    }
    *reinterpret_cast<uint4*>(s_ahi + m * w + ch * 8) = hv;
    *reinterpret_cast<uint4*>(s_alo + m * w + ch * 8) = lv;
    s_ss1[m * g.nch_max + ch] = ss;
  }
  __syncthreads();
  if (tid < M) {
    float ss = 0.f;
    for (int ch = 0; ch < nch; ++ch) ss += s_ss1[tid * g.nch_max + ch];
    p.sumsq[b * M + tid] = ss;
  }

  // --- phase 0: inputs of this CTA's channel range for the final mix (iw,
  // R, y and Wnorm), one merged index space so a thread's loads overlap
  {
    const int n_iw = M * HC, n_r = M * HC * nc, n_y = M * nc, n_w = HC * nc;
#pragma unroll 4
    for (int i = tid; i < n_iw + n_r + n_y + n_w; i += NT) {
      if (i < n_iw) {
        s_iw[i] = 2.0f * sigmoidf_dev(c.inj[(i / HC) * c.ld_inj + (i % HC)] / static_cast<float>(HC));
      } else if (i < n_iw + n_r) {
        const int j = i - n_iw;
        const int m = j / (HC * nc), rem = j % (HC * nc), ss = rem / nc, cc = rem % nc;
        s_x3r[(m * HC + ss) * g.nc_max + cc] =
            __ldg(c.R + static_cast<int64_t>(m) * K + ss * HS + cp0 + cc);
      } else if (i < n_iw + n_r + n_y) {
        const int j = i - n_iw - n_r;
        const int m = j / nc, cc = j % nc;
        s_x3y[m * g.nc_max + cc] = __ldg(c.y + static_cast<int64_t>(m) * HS + cp0 + cc);
      } else {
        const int j = i - n_iw - n_r - n_y;
        const int ss = j / nc, cc = j % nc;
        s_x3w[ss * g.nc_max + cc] = __ldg(c.Wnorm + ss * HS + cp0 + cc);
      }
    }
  }

  // --- phase 1b: partial products on the tensor cores
  const int nk16 = w / 16;
  const bool k8 = (w & 15) != 0;
  const bool lo_pass = !c.fold;
  auto tile_mma = [&](const unsigned char* rows, int row0, int tt, float* acc) {
    // rows: shared-memory rows of w bf16 (stride 2w bytes); 16 rows from row0.
    // The hi and lo terms accumulate separately (two short MMA chains).
    const unsigned char* ra = rows + (row0 + gq) * w * 2;
    const unsigned char* rb = ra + 8 * w * 2;
    const unsigned char* bh = reinterpret_cast<const unsigned char*>(s_ahi + (tt * 8 + gq) * w);
    const unsigned char* bl = reinterpret_cast<const unsigned char*>(s_alo + (tt * 8 + gq) * w);
    float lo[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int ks = 0; ks < nk16; ++ks) {
      const int cb = (ks * 16 + 2 * tq) * 2;
      const uint32_t a0 = lds32(ra + cb), a1 = lds32(rb + cb), a2 = lds32(ra + cb + 16),
                     a3 = lds32(rb + cb + 16);
      mma_16816(acc, a0, a1, a2, a3, lds32(bh + cb), lds32(bh + cb + 16));
      if (lo_pass) mma_16816(lo, a0, a1, a2, a3, lds32(bl + cb), lds32(bl + cb + 16));
    }
    if (k8) {
      const int cb = (nk16 * 16 + 2 * tq) * 2;
      const uint32_t a0 = lds32(ra + cb), a1 = lds32(rb + cb);
      mma_1688(acc, a0, a1, lds32(bh + cb));
      if (lo_pass) mma_1688(lo, a0, a1, lds32(bl + cb));
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] += lo[e];
  };
  auto store_part = [&](int nbase, int nvalid, int row0, int tt, const float* acc) {
    const int m0 = tt * 8 + 2 * tq;
    const int rows[2] = {row0 + gq, row0 + gq + 8};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (rows[h] >= nvalid) continue;
      const int n = nbase + rows[h];
      float* dst = p.part + static_cast<int64_t>(b) * g.part_ld + n;
      if (m0 < M) dst[m0 * n_out] = acc[2 * h];
      if (m0 + 1 < M) dst[(m0 + 1) * n_out] = acc[2 * h + 1];
    }
  };

  bool ok = true;
  for (int bx = 0; bx < g.nbox && ok; ++bx) {
    const int slot = bx % g.nslot_w;
    const bool got = mbar_wait_bounded(barW(slot), (bx / g.nslot_w) & 1, p.err, p.limit_ns);
    if (!__syncthreads_and(got)) { ok = false; break; }
    ++done_w;
    const int n_lo = bx * g.rows_box;
    const int nrows = min(r, n_lo + g.rows_box) - n_lo;
    const int ntile = (nrows + 15) / 16;
    const unsigned char* base = smem + g.off_w + slot * g.slot_w;
    for (int pr = warp; pr < ntile * ntok; pr += NW) {
      const int nt = pr / ntok, tt = pr % ntok;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      tile_mma(base, nt * 16, tt, acc);
      store_part(n_lo, nrows, nt * 16, tt, acc);
    }
    __syncthreads();
    if (issued_w < g.nbox) {
      if (tid == 0) issue_w(issued_w);
      ++issued_w;
    }
  }
  bool wi_done = false;
  if (ok) {
    const bool got = mbar_wait_bounded(barWi, 0, p.err, p.limit_ns);
    wi_done = ok = __syncthreads_and(got);
    if (ok) {
      for (int tt = warp; tt < ntok; tt += NW) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        tile_mma(smem + g.off_wi, 0, tt, acc);
        store_part(r, HC, 0, tt, acc);
      }
    }
  }

  // A test hook: this CTA leaves before the first barrier, as if it had died.
  if (c.debug_fault == 1 && b == 0) ok = false;
  if (ok) ok = grid_barrier(p.bar, g.G, p.err, p.limit_ns, s_flag);

  // --- phase 2: rrms, then lora / inj_next for this CTA's output range
  if (ok) {
    if (tid == 0) {
      fence_proxy_async_global();
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(barP, static_cast<uint32_t>(g.G * g.Q * 4 + g.ss_bytes));
      tma_load_2d(smem_u32(s_pbox), &p.tm_part, b * g.Q, 0, barP);
      bulk_g2s(smem_u32(s_ss), p.sumsq, static_cast<uint32_t>(g.ss_bytes), barP);
    }
    const bool got = mbar_wait_bounded(barP, 0, p.err, p.limit_ns);
    ok = __syncthreads_and(got);
  }
  if (ok) {
    for (int i = warp; i < M * HC; i += NW) {
      const int m = i / HC, ss = i % HC;
      float a = 0.f;
      for (int j = lane; j < g.P; j += 32) a += s_ss[(ss * g.P + j) * M + m];
      a = warp_sum(a);
      const float rr = 1.0f / sqrtf(a / static_cast<float>(HS) + c.eps);
      if (lane == 0) {
        s_rr[i] = rr;
        if (b == 0) c.rrms[i] = rr;
      }
    }
    // per (output o, stream s): the stream's P partials in order (consecutive
    // threads read consecutive outputs: no bank conflicts), scaled by rrms_s
    const int n_own = min(g.Q, M * n_out - b * g.Q);
    for (int i = tid; i < g.Q * HC; i += NT) {
      const int o = i % g.Q, ss = i / g.Q;
      const int og = b * g.Q + o;
      float a = 0.f;
      if (o < n_own) {
        const float* col = s_pbox + ss * g.P * g.Q + o;
        for (int j = 0; j < g.P; ++j) a += col[j * g.Q];
        a *= s_rr[(og / n_out) * HC + ss];
      }
      s_red[ss * g.Q + o] = a;
    }
    __syncthreads();
    const float inv_hc = 1.0f / static_cast<float>(HC);
    for (int o = tid; o < n_own; o += NT) {
      const int og = b * g.Q + o;
      const int m = og / n_out, n = og % n_out;
      float acc = 0.f;
      for (int ss = 0; ss < HC; ++ss) acc += s_red[ss * g.Q + o];
      if (n < r) {
        c.lora[static_cast<int64_t>(m) * r + n] = acc;
        const float u = acc * inv_hc;
        p.hdec[m * r + n] = f32_to_bf16(u * sigmoidf_dev(u));
      } else {
        c.inj_next[static_cast<int64_t>(m) * HC + (n - r)] = acc;
      }
    }
    ok = grid_barrier(p.bar, g.G, p.err, p.limit_ns, s_flag);
  }

  // --- phase 3: h, gates for this CTA's channels, gated mean
  if (ok && nc > 0) {
    if (warp == 0) {
      if (lane == 0) {
        fence_proxy_async_global();
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(barL, static_cast<uint32_t>(M * r * 2));
      }
      __syncwarp();
      for (int m = lane; m < M; m += 32)   // rows land at the padded stride
        bulk_g2s(smem_u32(s_h + m * g.hstride), p.hdec + m * r, static_cast<uint32_t>(r * 2), barL);
    }
    for (int i = tid; i < (MB - M) * g.hstride; i += NT) s_h[M * g.hstride + i] = 0;
    const bool got = mbar_wait_bounded(barL, 0, p.err, p.limit_ns);
    ok = __syncthreads_and(got);
  }
  if (ok && nc > 0) {
    const float inv_hc = 1.0f / static_cast<float>(HC);
    const int nrt = g.rows_u16 / 16;
    const int npair = nrt * ntok;
    float acc[MAXP][4];
#pragma unroll
    for (int j = 0; j < MAXP; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    auto chunk_mma = [&](const unsigned char* ub, int q) {
      const int kc = min(64, r - q * 64);
#pragma unroll
      for (int j = 0; j < MAXP; ++j) {
        const int pr = warp + j * NW;
        if (pr >= npair) break;
        const int rt = pr / ntok, tt = pr % ntok;
        const int i0 = rt * 16 + gq, i1 = i0 + 8;       // rows of the swizzled box (i1 % 8 == i0 % 8)
        const unsigned char* ra = ub + i0 * 128;
        const unsigned char* rb = ub + i1 * 128;
        const int sw = i0 & 7;
        const unsigned char* hb = reinterpret_cast<const unsigned char*>(
            s_h + (tt * 8 + gq) * g.hstride + q * 64);
        int ks = 0;
        for (; ks + 16 <= kc; ks += 16) {
          const int ch0 = ks >> 3;
          const int o0 = ((ch0 ^ sw) << 4) + tq * 4, o1 = (((ch0 + 1) ^ sw) << 4) + tq * 4;
          mma_16816(acc[j], lds32(ra + o0), lds32(rb + o0), lds32(ra + o1), lds32(rb + o1),
                    lds32(hb + (ks + 2 * tq) * 2), lds32(hb + (ks + 8 + 2 * tq) * 2));
        }
        if (ks < kc) {
          const int o0 = (((ks >> 3) ^ sw) << 4) + tq * 4;
          mma_1688(acc[j], lds32(ra + o0), lds32(rb + o0), lds32(hb + (ks + 2 * tq) * 2));
        }
      }
    };
    if (g.nslot_u == g.nchunk_u) {
      // every chunk has its own slot, all issued at kernel start
      bool got = true;
      for (int q = 0; q < g.nchunk_u; ++q)
        got = mbar_wait_bounded(barU(q), 0, p.err, p.limit_ns) && got;
      ok = __syncthreads_and(got);
      if (ok) {
        done_u = issued_u;
        for (int q = 0; q < g.nchunk_u; ++q) chunk_mma(smem + g.off_u + q * g.slot_u, q);
      }
    } else {
      for (int q = 0; q < g.nchunk_u && ok; ++q) {
        const int slot = q % g.nslot_u;
        const bool got = mbar_wait_bounded(barU(slot), (q / g.nslot_u) & 1, p.err, p.limit_ns);
        if (!__syncthreads_and(got)) { ok = false; break; }
        ++done_u;
        chunk_mma(smem + g.off_u + slot * g.slot_u, q);
        __syncthreads();
        if (issued_u < g.nchunk_u) {
          if (tid == 0) issue_u(issued_u);
          ++issued_u;
        }
      }
    }
    if (ok) {
#pragma unroll
      for (int j = 0; j < MAXP; ++j) {
        const int pr = warp + j * NW;
        if (pr >= npair) break;
        const int rt = pr / ntok, tt = pr % ntok;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = rt * 16 + gq + (e >> 1) * 8;
          const int m = tt * 8 + 2 * tq + (e & 1);
          if (i < g.rows_u && m < M) s_g[m * g.rows_u + i] = sigmoidf_dev(acc[j][e]);
        }
      }
      __syncthreads();
      for (int i = tid; i < M * nc; i += NT) {
        const int m = i / nc, cc = i % nc, ch = cp0 + cc;
        float sum = 0.f;
        for (int ss = 0; ss < HC; ++ss) {
          const float rv = bf16_to_f32(s_x3r[(m * HC + ss) * g.nc_max + cc]);
          const float yv = bf16_to_f32(s_x3y[m * g.nc_max + cc]);
          const float r2 = bf16_to_f32(f32_to_bf16(fmaf(yv, s_iw[m * HC + ss], rv)));
          const float xn = r2 * s_rr[m * HC + ss] * (1.0f + bf16_to_f32(s_x3w[ss * g.nc_max + cc]));
          sum = fmaf(s_g[m * g.rows_u + ss * g.nc_max + cc], xn, sum);
        }
        c.x[static_cast<int64_t>(m) * HS + ch] = f32_to_bf16(sum * inv_hc);
      }
    }
  }

  // Let every copy this CTA issued land before its shared memory is released
  // (only outstanding after a failed wait or an early exit).
  for (int i = done_w; i < issued_w; ++i)
    mbar_wait_bounded(barW(i % g.nslot_w), (i / g.nslot_w) & 1, p.err, p.limit_ns);
  if (!wi_done) mbar_wait_bounded(barWi, 0, p.err, p.limit_ns);
  for (int i = done_u; i < issued_u; ++i)
    mbar_wait_bounded(barU(i % g.nslot_u), (i / g.nslot_u) & 1, p.err, p.limit_ns);
}

}  // namespace

size_t decode_ws_part_floats(const Device& dev, int K_max, int n_out_max) {
  (void)K_max;
  return static_cast<size_t>(dev.sms) * (static_cast<size_t>(DECODE_MAX_M) * n_out_max + 4);
}

cudaError_t launch_decode(const Call& c, const Workspace& ws, const Device& dev,
                          cudaStream_t stream) {
  Params prm;
  prm.c = c;
  prm.part = ws.part;
  prm.sumsq = ws.sumsq;
  prm.hdec = ws.hdec;
  prm.bar = nullptr;
  prm.err = ws.err;
  prm.limit_ns = c.debug_fault ? 50ull * 1000 * 1000 : 1000ull * 1000 * 1000;
  if (!make_geom(c, dev, prm.g)) return cudaErrorNotSupported;
  const Geom& g = prm.g;
  if (g.G > MAX_GRID) return cudaErrorNotSupported;
  prm.bar = ws.bar + g.G;
  const uint64_t wstr[2] = {static_cast<uint64_t>(c.HS) * 2, static_cast<uint64_t>(c.K) * 2};
  const uint64_t dwd[3] = {static_cast<uint64_t>(c.HS), static_cast<uint64_t>(c.HC),
                           static_cast<uint64_t>(c.r)};
  const uint32_t bwd[3] = {static_cast<uint32_t>(g.w), 1u, static_cast<uint32_t>(g.rows_box)};
  const uint64_t dwi[3] = {static_cast<uint64_t>(c.HS), static_cast<uint64_t>(c.HC),
                           static_cast<uint64_t>(c.HC)};
  const uint32_t bwi[3] = {static_cast<uint32_t>(g.w), 1u, static_cast<uint32_t>(c.HC)};
  const uint64_t dwu[3] = {static_cast<uint64_t>(c.r), static_cast<uint64_t>(c.HS),
                           static_cast<uint64_t>(c.HC)};
  const uint64_t swu[2] = {static_cast<uint64_t>(c.r) * 2, static_cast<uint64_t>(c.HS) * c.r * 2};
  const uint32_t bwu[3] = {64u, static_cast<uint32_t>(g.nc_max), static_cast<uint32_t>(c.HC)};
  const uint64_t dp[2] = {static_cast<uint64_t>(g.part_ld), static_cast<uint64_t>(g.G)};
  const uint64_t sp[1] = {static_cast<uint64_t>(g.part_ld) * 4};
  const uint32_t bp[2] = {static_cast<uint32_t>(g.Q), static_cast<uint32_t>(g.G)};
  if (!make_tmap_bf16(&prm.tm_wd, c.Wd, 3, dwd, wstr, bwd) ||
      !make_tmap_bf16(&prm.tm_wi, c.Wi, 3, dwi, wstr, bwi) ||
      !make_tmap_bf16(&prm.tm_wu, c.Wu, 3, dwu, swu, bwu, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap(&prm.tm_part, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ws.part, 2, dp, sp, bp))
    return cudaErrorNotSupported;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.G);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = g.total + 1024;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel, prm);
}

}  // namespace hcgr

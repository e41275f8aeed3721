// Decode path of the HC gated residual: one cooperative persistent kernel for
// small token counts (M <= 32), where the time goes into streaming the
// weights once (aiter PR #5913, "Technical Details"; the page's skinny decode
// with split-K partials and a last-stage reduce is the prior art).
//
// Grid: G = HC * P CTAs (at most one per SM).  Three phases separated by
// bounded grid barriers:
//   1. CTA b owns a channel slice [c0, c0 + w) of one stream s (w a multiple
//      of 8; every slice has the same width, the last one of a stream is
//      clipped by the stream end).  It forms R2 = bf16(R + y * iw) for that
//      slice (writes R2), the partial sum of R2^2 per token, and the partial
//      products
//        part[b][m][n] = sum_{c in slice} R2[m,s,c] * f[k] * W[n, k],
//      f = (1 + Wnorm) (1 for a folded weight), for all r + HC rows n of the
//      down and inject weights.  Because rrms_s is constant over stream s,
//      lora = sum_b rrms_{s(b)} part[b] is exact: the per-stream factor
//      commutes out of the K-sum.
//   2. rrms from the partial sums of squares; lora and inj_next as the
//      rrms-weighted sum of the partial products (fixed order, so the result
//      is deterministic).
//   3. CTA b owns a channel range of x: it forms h = SiLU(lora / HC), the
//      gates G[s, c] = sigmoid(h . Wu[s * HS + c]) for its channels and all
//      streams, rebuilds xn from R2, rrms and Wnorm, and writes the gated
//      mean x.
// Weight traffic: the down/inject slice arrives as a few 3-D TMA boxes (the
// tensor map treats the stream as its own dimension, so a box never crosses
// a stream end), the up-weight rows of a stream as one contiguous bulk copy.
// All of them are issued at kernel start when they fit in shared memory, so
// the whole weight stream is in flight before the first barrier; otherwise
// they stream through two-slot rings.
#include <algorithm>

#include "hc_gr_internal.cuh"
#include "tmap.h"

namespace hcgr {
namespace {

constexpr int NT = 384;            // threads per CTA
constexpr int NW = NT / 32;
constexpr int MAX_SLOTS = 8;
constexpr int BOX_CAP = 32 * 1024; // bytes per down/inject weight box
constexpr size_t SMEM_BUDGET = 200 * 1024;
constexpr size_t SMEM_ALLOC = SMEM_BUDGET + 128;

struct Geom {
  int G, P, w, nch_max;            // phase 1: P slices of w channels per stream
  int nbox, rows_box, slot_w;      // down weight boxes (rows per box, slot bytes)
  int nslot_w;
  int slot_u, nslot_u;             // up weight: one slot per stream block
  int nc_max;                      // phase 3 channel range
  int off_act, off_h, off_g, off_ss, off_rr, off_red, off_wi, off_w, off_u, total;
};

__host__ __device__ inline int round_up(int v, int a) { return (v + a - 1) / a * a; }

struct Params {
  CUtensorMap tm_wd;   // Wd as [r][HC][HS] (inner HS)
  CUtensorMap tm_wi;   // Wi as [HC][HC][HS]
  Call c;
  Geom g;
  float* part;
  float* sumsq;
  unsigned* bar;
  int* err;
  uint64_t limit_ns;
};

bool make_geom(const Call& c, const Device& dev, int MB, Geom& g) {
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
  g.nbox = std::max(1, (c.r * w * 2 + BOX_CAP - 1) / BOX_CAP);
  g.rows_box = round_up((c.r + g.nbox - 1) / g.nbox, 8);
  while (g.rows_box > 256) {
    ++g.nbox;
    g.rows_box = round_up((c.r + g.nbox - 1) / g.nbox, 8);
  }
  g.nbox = (c.r + g.rows_box - 1) / g.rows_box;
  g.slot_w = round_up(g.rows_box * w * 2, 128);
  g.nc_max = (c.HS + g.G - 1) / g.G;
  g.slot_u = round_up(g.nc_max * c.r * 2, 128);
  // phase-1 activations share space with the phase-3 gates, the phase-2
  // partial sums of squares with phase-3 h (their lifetimes do not overlap)
  int off = 256;                                       // mbarriers + flag
  g.off_act = g.off_g = off;
  off += round_up(std::max(MB * w, MB * c.HC * g.nc_max) * 4, 128);
  g.off_ss = g.off_h = off;
  off += round_up(std::max(std::max(MB * g.nch_max, MB * g.G), MB * c.r) * 4, 128);
  g.off_rr = off;   off += round_up(MB * c.HC * 4, 128);
  g.off_red = off;  off += round_up(NW * 32 * 4, 128);
  g.off_wi = off;   off += round_up(c.HC * w * 2, 128);
  const int left = static_cast<int>(SMEM_BUDGET) - off;
  if (g.nbox * g.slot_w + c.HC * g.slot_u <= left && g.nbox <= MAX_SLOTS && c.HC <= MAX_SLOTS) {
    g.nslot_w = g.nbox;
    g.nslot_u = c.HC;
  } else {
    // two-slot rings; the down-weight box height takes what the up ring leaves
    g.nslot_u = std::min(c.HC, 2);
    const int rows = ((left - g.nslot_u * g.slot_u) / 2 / (w * 2)) / 8 * 8;
    if (rows < 8) return false;
    g.rows_box = std::min(std::min(rows, 256), round_up(c.r, 8));
    g.nbox = (c.r + g.rows_box - 1) / g.rows_box;
    g.slot_w = round_up(g.rows_box * w * 2, 128);
    g.nslot_w = std::min(g.nbox, 2);
  }
  g.off_w = off;  off += g.nslot_w * g.slot_w;
  g.off_u = off;  off += g.nslot_u * g.slot_u;
  g.total = off;
  return g.total <= static_cast<int>(SMEM_BUDGET);
}

// --------------------------------------------------------------- the kernel
template <int MB>
__global__ void __launch_bounds__(NT, 1) decode_kernel(const __grid_constant__ Params p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  const Call& c = p.c;
  const Geom& g = p.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const int M = static_cast<int>(c.M);
  const int HC = c.HC, HS = c.HS, K = c.K, r = c.r, n_out = c.n_out;

  int* s_flag = reinterpret_cast<int*>(smem + 240);
  float* s_act = reinterpret_cast<float*>(smem + g.off_act);   // [MB][w]
  float* s_h = reinterpret_cast<float*>(smem + g.off_h);       // [MB][r]
  float* s_g = reinterpret_cast<float*>(smem + g.off_g);       // [MB][HC * nc_max]
  float* s_ss = reinterpret_cast<float*>(smem + g.off_ss);
  float* s_rr = reinterpret_cast<float*>(smem + g.off_rr);     // [MB][HC]
  float* s_red = reinterpret_cast<float*>(smem + g.off_red);   // [NW][32]

  // phase-1 slice of this CTA
  const int s = b / g.P;
  const int c0 = (b % g.P) * g.w;
  const int nch = (min(HS, c0 + g.w) - c0) / 8;
  const int k0 = s * HS + c0;
  // phase-3 channel range of this CTA
  const int cp0 = min(HS, b * g.nc_max);
  const int nc = min(HS, cp0 + g.nc_max) - cp0;

  const uint32_t bar0 = smem_u32(smem);
  auto barW = [&](int i) { return bar0 + 8u * i; };               // [0, 8)
  auto barU = [&](int i) { return bar0 + 64u + 8u * i; };         // [8, 16)
  const uint32_t barWi = bar0 + 128u;

  if (tid == 0) {
    for (int i = 0; i < 17; ++i) mbar_init(bar0 + 8u * i, 1);
    fence_mbar_init();
  }
  __syncthreads();

  // --- weight copies (thread 0 of warp 0 issues; tiny instruction count)
  auto issue_w = [&](int bx) {
    const int slot = bx % g.nslot_w;
    mbar_arrive_expect_tx(barW(slot), static_cast<uint32_t>(g.rows_box * g.w * 2));
    tma_load_3d(smem_u32(smem + g.off_w + slot * g.slot_w), &p.tm_wd, c0, s, bx * g.rows_box,
                barW(slot));
  };
  auto issue_u = [&](int sb) {
    const int slot = sb % g.nslot_u;
    mbar_arrive_expect_tx(barU(slot), static_cast<uint32_t>(nc * r * 2));
    bulk_g2s(smem_u32(smem + g.off_u + slot * g.slot_u),
             c.Wu + static_cast<int64_t>(sb * HS + cp0) * r, static_cast<uint32_t>(nc * r * 2),
             barU(slot));
  };
  int issued_w = 0, issued_u = 0, done_w = 0, done_u = 0;   // uniform across the CTA
  if (tid == 0) {
    mbar_arrive_expect_tx(barWi, static_cast<uint32_t>(HC * g.w * 2));
    tma_load_3d(smem_u32(smem + g.off_wi), &p.tm_wi, c0, s, 0, barWi);
  }
  for (; issued_w < g.nslot_w; ++issued_w)
    if (tid == 0) issue_w(issued_w);
  if (nc > 0)
    for (; issued_u < g.nslot_u; ++issued_u)
      if (tid == 0) issue_u(issued_u);

  bool ok = true;
  // --- phase 1a: COMBINE on this CTA's slice, R2 stored, partial sums of R2^2
  for (int it = tid; it < M * nch; it += NT) {
    const int m = it / nch, ch = it % nch;
    const int64_t kk = static_cast<int64_t>(m) * K + k0 + ch * 8;
    const float iw = 2.0f * sigmoidf_dev(c.inj[m * c.ld_inj + s] / static_cast<float>(HC));
    float rv[8], yv[8], wv[8];
    unpack8(__ldg(reinterpret_cast<const uint4*>(c.R + kk)), rv);
    unpack8(__ldg(reinterpret_cast<const uint4*>(c.y + static_cast<int64_t>(m) * HS + c0 + ch * 8)), yv);
    unpack8(__ldg(reinterpret_cast<const uint4*>(c.Wnorm + k0 + ch * 8)), wv);
    float ss = 0.f, r2[8];
    uint32_t packed[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      r2[i] = bf16_to_f32(f32_to_bf16(fmaf(yv[i], iw, rv[i])));
      ss = fmaf(r2[i], r2[i], ss);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) packed[i] = pack2(r2[2 * i], r2[2 * i + 1]);
    *reinterpret_cast<uint4*>(c.R2 + kk) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    float* a = s_act + m * g.w + ch * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = c.fold ? r2[i] : r2[i] * (1.0f + wv[i]);
    s_ss[m * g.nch_max + ch] = ss;
  }
  __syncthreads();
  if (tid < M) {
    float ss = 0.f;
    for (int ch = 0; ch < nch; ++ch) ss += s_ss[tid * g.nch_max + ch];
    p.sumsq[b * M + tid] = ss;
  }

  // --- phase 1b: partial products over the slice for all n_out rows
  auto dot_rows = [&](const unsigned char* rows, int n_lo, int n_hi, int n_base) {
    for (int n = n_lo + tid; n < n_hi; n += NT) {
      float acc[MB];
#pragma unroll
      for (int m = 0; m < MB; ++m) acc[m] = 0.f;
      const unsigned char* wrow = rows + (n - n_lo) * g.w * 2;
      for (int ch = 0; ch < nch; ++ch) {
        float wf[8];
        unpack8(*reinterpret_cast<const uint4*>(wrow + ch * 16), wf);
#pragma unroll
        for (int m = 0; m < MB; ++m) {
          if (m < M) {
            const float4 a0 = *reinterpret_cast<const float4*>(s_act + m * g.w + ch * 8);
            const float4 a1 = *reinterpret_cast<const float4*>(s_act + m * g.w + ch * 8 + 4);
            float t = acc[m];
            t = fmaf(a0.x, wf[0], t); t = fmaf(a0.y, wf[1], t);
            t = fmaf(a0.z, wf[2], t); t = fmaf(a0.w, wf[3], t);
            t = fmaf(a1.x, wf[4], t); t = fmaf(a1.y, wf[5], t);
            t = fmaf(a1.z, wf[6], t); t = fmaf(a1.w, wf[7], t);
            acc[m] = t;
          }
        }
      }
#pragma unroll
      for (int m = 0; m < MB; ++m)
        if (m < M) p.part[(static_cast<int64_t>(b) * M + m) * n_out + n_base + n] = acc[m];
    }
  };
  for (int bx = 0; bx < g.nbox && ok; ++bx) {
    const int slot = bx % g.nslot_w;
    const bool got = mbar_wait_bounded(barW(slot), (bx / g.nslot_w) & 1, p.err, p.limit_ns);
    if (!__syncthreads_and(got)) { ok = false; break; }
    ++done_w;
    const int n_lo = bx * g.rows_box, n_hi = min(r, n_lo + g.rows_box);
    dot_rows(smem + g.off_w + slot * g.slot_w, n_lo, n_hi, 0);
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
    if (ok) dot_rows(smem + g.off_wi, 0, HC, r);
  }

  // A test hook: this CTA leaves before the first barrier, as if it had died.
  if (c.debug_fault == 1 && b == 0) ok = false;
  if (ok) ok = grid_barrier(p.bar, g.G, p.err, p.limit_ns, s_flag);

  // --- phase 2: rrms, then lora / inj_next as rrms-weighted sums of partials
  if (ok) {
    for (int i = tid; i < M * g.G; i += NT) {
      const int m = i / g.G, bb = i % g.G;
      s_ss[i] = __ldcg(p.sumsq + bb * M + m);
    }
    __syncthreads();
    for (int i = tid; i < M * HC; i += NT) {
      const int m = i / HC, ss = i % HC;
      const float* v = s_ss + m * g.G + ss * g.P;
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
      int q = 0;
      for (; q + 4 <= g.P; q += 4) { a0 += v[q]; a1 += v[q + 1]; a2 += v[q + 2]; a3 += v[q + 3]; }
      for (; q < g.P; ++q) a0 += v[q];
      const float rr = 1.0f / sqrtf(((a0 + a1) + (a2 + a3)) / static_cast<float>(HS) + c.eps);
      s_rr[i] = rr;
      if (b == 0) c.rrms[i] = rr;
    }
    __syncthreads();
    const int ntn = (n_out + 31) / 32;
    for (int t = b; t < M * ntn; t += g.G) {
      const int m = t / ntn;
      const int n = (t % ntn) * 32 + lane;
      float acc = 0.f;
      if (n < n_out) {
#pragma unroll 4
        for (int bb = warp; bb < g.G; bb += NW)
          acc = fmaf(s_rr[m * HC + bb / g.P],
                     __ldcg(p.part + (static_cast<int64_t>(bb) * M + m) * n_out + n), acc);
      }
      s_red[warp * 32 + lane] = acc;
      __syncthreads();
      if (warp == 0 && n < n_out) {
        float tot = 0.f;
        for (int w = 0; w < NW; ++w) tot += s_red[w * 32 + lane];
        if (n < r) c.lora[static_cast<int64_t>(m) * r + n] = tot;
        else c.inj_next[static_cast<int64_t>(m) * HC + (n - r)] = tot;
      }
      __syncthreads();
    }
    ok = grid_barrier(p.bar, g.G, p.err, p.limit_ns, s_flag);
  }

  // --- phase 3: h, gates for this CTA's channels, gated mean
  if (ok && nc > 0) {
    for (int i = tid; i < M * r; i += NT) {
      const float u = __ldcg(c.lora + i) / static_cast<float>(HC);
      s_h[i] = u * sigmoidf_dev(u);
    }
    __syncthreads();
    for (int sb = 0; sb < HC; ++sb) {
      const int slot = sb % g.nslot_u;
      const bool got = mbar_wait_bounded(barU(slot), (sb / g.nslot_u) & 1, p.err, p.limit_ns);
      if (!__syncthreads_and(got)) { ok = false; break; }
      ++done_u;
      const bf16_t* wblk = reinterpret_cast<const bf16_t*>(smem + g.off_u + slot * g.slot_u);
      for (int cc = warp; cc < nc; cc += NW) {
        const bf16_t* wu = wblk + static_cast<int64_t>(cc) * r;
        float acc[MB];
#pragma unroll
        for (int m = 0; m < MB; ++m) acc[m] = 0.f;
        for (int n = lane; n < r; n += 32) {
          const float wv = bf16_to_f32(wu[n]);
#pragma unroll
          for (int m = 0; m < MB; ++m)
            if (m < M) acc[m] = fmaf(s_h[m * r + n], wv, acc[m]);
        }
#pragma unroll
        for (int m = 0; m < MB; ++m) {
          if (m < M) {
            const float v = warp_sum(acc[m]);
            if (lane == 0) s_g[m * HC * g.nc_max + sb * g.nc_max + cc] = sigmoidf_dev(v);
          }
        }
      }
      __syncthreads();
      if (issued_u < HC) {
        if (tid == 0) issue_u(issued_u);
        ++issued_u;
      }
    }
    if (ok) {
      for (int i = tid; i < M * nc; i += NT) {
        const int m = i / nc, cc = i % nc, ch = cp0 + cc;
        float acc = 0.f;
        for (int ss = 0; ss < HC; ++ss) {
          const int64_t k = static_cast<int64_t>(ss) * HS + ch;
          const float r2 = bf16_to_f32(__ldcg(c.R2 + static_cast<int64_t>(m) * K + k));
          const float xn = r2 * s_rr[m * HC + ss] * (1.0f + bf16_to_f32(__ldg(c.Wnorm + k)));
          acc = fmaf(s_g[m * HC * g.nc_max + ss * g.nc_max + cc], xn, acc);
        }
        c.x[static_cast<int64_t>(m) * HS + ch] = f32_to_bf16(acc / static_cast<float>(HC));
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

template <int MB>
cudaError_t launch_mb(const Params& prm, cudaStream_t stream) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<MB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_ALLOC));
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(prm.g.G);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = prm.g.total + 128;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<MB>, prm);
}

}  // namespace

size_t decode_ws_part_floats(const Device& dev, int K_max, int n_out_max) {
  (void)K_max;
  return static_cast<size_t>(dev.sms) * DECODE_MAX_M * n_out_max;
}

cudaError_t launch_decode(const Call& c, const Workspace& ws, const Device& dev,
                          cudaStream_t stream) {
  Params prm;
  prm.c = c;
  prm.part = ws.part;
  prm.sumsq = ws.sumsq;
  prm.bar = ws.bar;
  prm.err = ws.err;
  prm.limit_ns = c.debug_fault ? 50ull * 1000 * 1000 : 1000ull * 1000 * 1000;
  const int M = static_cast<int>(c.M);
  const int MB = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : M <= 16 ? 16 : 32;
  if (!make_geom(c, dev, MB, prm.g)) return cudaErrorNotSupported;
  const Geom& g = prm.g;
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(c.HS), static_cast<uint64_t>(c.HC),
                              static_cast<uint64_t>(c.r)};
    const uint64_t strides[2] = {static_cast<uint64_t>(c.HS) * 2, static_cast<uint64_t>(c.K) * 2};
    const uint32_t box[3] = {static_cast<uint32_t>(g.w), 1u, static_cast<uint32_t>(g.rows_box)};
    if (!make_tmap_bf16(&prm.tm_wd, c.Wd, 3, dims, strides, box)) return cudaErrorInvalidValue;
    const uint64_t dims_i[3] = {static_cast<uint64_t>(c.HS), static_cast<uint64_t>(c.HC),
                                static_cast<uint64_t>(c.HC)};
    const uint32_t box_i[3] = {static_cast<uint32_t>(g.w), 1u, static_cast<uint32_t>(c.HC)};
    if (!make_tmap_bf16(&prm.tm_wi, c.Wi, 3, dims_i, strides, box_i)) return cudaErrorInvalidValue;
  }
  switch (MB) {
    case 1: return launch_mb<1>(prm, stream);
    case 2: return launch_mb<2>(prm, stream);
    case 4: return launch_mb<4>(prm, stream);
    case 8: return launch_mb<8>(prm, stream);
    case 16: return launch_mb<16>(prm, stream);
    default: return launch_mb<32>(prm, stream);
  }
}

}  // namespace hcgr

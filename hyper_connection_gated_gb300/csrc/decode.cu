// Decode path of the HC gated residual: one cooperative persistent kernel for
// small token counts (M <= 32), where the time goes into streaming the
// weights once (aiter PR #5913, "Technical Details"; the page's skinny decode
// with split-K partials and a last-stage reduce is the prior art).
//
// Grid: G CTAs, one per SM, G a multiple of HC.  Three phases separated by
// bounded grid barriers:
//   1. CTA b owns a channel slice [c0, c0 + w) of one stream s (w a multiple
//      of 8, so every row slice is a 16-byte aligned run).  It forms
//      R2 = bf16(R + y * iw) for that slice (writes R2), the partial sum of
//      R2^2 per token, and the partial products
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
// Every CTA issues the bulk copies of its weight slices (down/inject rows
// and up rows) at kernel start, so the whole weight stream is in flight
// before the first barrier.
#include <algorithm>

#include "hc_gr_internal.cuh"

namespace hcgr {
namespace {

constexpr int NT = 384;            // threads per CTA
constexpr int NW = NT / 32;
constexpr int NSTAGE = 2;          // ring depth per weight stream
constexpr size_t SMEM_BUDGET = 200 * 1024;

struct Geom {
  int G, per_stream, nch_max, wmax, wstride;   // phase 1 slice geometry
  int nc_max;                                  // phase 3 channel range
  int rows_w, nblk_w, stage_w_bytes;           // down/inject rows per stage
  int rows_u, stage_u_bytes;                   // up rows per stage
  int off_w, off_u, off_act, off_h, off_g, off_ss, off_rr, off_red, off_misc, total;
};

__host__ __device__ inline int round_up(int v, int a) { return (v + a - 1) / a * a; }

// Row stride in shared memory for a w-wide bf16 slice: an odd number of
// 16-byte units, so 8 consecutive lanes reading 16 bytes each from 8
// different rows hit 8 different bank groups.
__host__ __device__ inline int w_stride_bytes(int w) {
  int u = (w * 2 + 15) / 16;
  if ((u & 1) == 0) ++u;
  return u * 16;
}

struct Params {
  Call c;
  Geom g;
  float* part;
  float* sumsq;
  unsigned* bar;
  int* err;
  uint64_t limit_ns;
};

bool make_geom(const Call& c, int G, int MB, Geom& g) {
  g.G = G;
  g.per_stream = G / c.HC;
  const int nchunk = c.HS / 8;
  g.nch_max = (nchunk + g.per_stream - 1) / g.per_stream;
  g.wmax = g.nch_max * 8;
  g.wstride = w_stride_bytes(g.wmax);
  g.nc_max = (c.HS + G - 1) / G;
  const int n_out = c.n_out;
  // fixed regions
  int off = 64;                                        // 4 mbarriers + flag
  g.off_misc = 0;
  g.off_act = off;  off += round_up(MB * g.wmax * 4, 128);
  g.off_h = off;    off += round_up(MB * c.r * 4, 128);
  g.off_g = off;    off += round_up(MB * c.HC * g.nc_max * 4, 128);
  g.off_ss = off;   off += round_up(std::max(MB * g.nch_max, MB * G) * 4, 128);
  g.off_rr = off;   off += round_up(MB * c.HC * 4, 128);
  g.off_red = off;  off += round_up(NW * 32 * 4, 128);
  // weight rings: all rows in one stage when they fit, else NSTAGE stages
  const int left = static_cast<int>(SMEM_BUDGET) - off;
  if (left < 4096) return false;
  const int w_all = n_out * g.wstride;
  const int u_all = c.HC * g.nc_max * c.r * 2;
  if (w_all + u_all <= left) {
    g.rows_w = n_out;
    g.stage_w_bytes = round_up(w_all, 128);
    g.rows_u = c.HC * g.nc_max;
    g.stage_u_bytes = round_up(std::max(u_all, 16), 128);
  } else {
    const int per = left / 2 / NSTAGE;
    g.rows_w = std::min(n_out, per / g.wstride);
    g.rows_u = std::min(c.HC * g.nc_max, per / (c.r * 2));
    if (g.rows_w < 1 || g.rows_u < 1) return false;
    g.stage_w_bytes = round_up(g.rows_w * g.wstride, 128);
    g.stage_u_bytes = round_up(g.rows_u * c.r * 2, 128);
  }
  g.nblk_w = (n_out + g.rows_w - 1) / g.rows_w;
  const int nst_w = g.nblk_w > 1 ? NSTAGE : 1;
  g.off_w = off;  off += nst_w * g.stage_w_bytes;
  const int nblk_u = (c.HC * g.nc_max + g.rows_u - 1) / g.rows_u;
  const int nst_u = nblk_u > 1 ? NSTAGE : 1;
  g.off_u = off;  off += nst_u * g.stage_u_bytes;
  g.total = off;
  return g.total <= static_cast<int>(SMEM_BUDGET) + 1024;
}

// --------------------------------------------------------------- the kernel
template <int MB>
__global__ void __launch_bounds__(NT, 1) decode_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const Call& c = p.c;
  const Geom& g = p.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const int M = static_cast<int>(c.M);
  const int HC = c.HC, HS = c.HS, K = c.K, r = c.r, n_out = c.n_out;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);          // [0,1] W ring, [2,3] Wu ring
  int* s_flag = reinterpret_cast<int*>(smem + 40);
  float* s_act = reinterpret_cast<float*>(smem + g.off_act);   // [MB][wmax]
  float* s_h = reinterpret_cast<float*>(smem + g.off_h);       // [MB][r]
  float* s_g = reinterpret_cast<float*>(smem + g.off_g);       // [MB][HC * nc]
  float* s_ss = reinterpret_cast<float*>(smem + g.off_ss);
  float* s_rr = reinterpret_cast<float*>(smem + g.off_rr);     // [MB][HC]
  float* s_red = reinterpret_cast<float*>(smem + g.off_red);   // [NW][32]
  unsigned char* s_w = smem + g.off_w;
  unsigned char* s_u = smem + g.off_u;

  // phase-1 slice of this CTA
  const int s = b / g.per_stream;
  const int j = b % g.per_stream;
  const int nchunk = HS / 8;
  const int lo = j * nchunk / g.per_stream, hi = (j + 1) * nchunk / g.per_stream;
  const int c0 = lo * 8, nch = hi - lo;
  const int k0 = s * HS + c0;
  // phase-3 channel range of this CTA
  const int cp0 = static_cast<int>(static_cast<int64_t>(b) * HS / g.G);
  const int cp1 = static_cast<int>(static_cast<int64_t>(b + 1) * HS / g.G);
  const int nc = cp1 - cp0;
  const int rows_u_all = HC * nc;

  const int nst_w = g.nblk_w > 1 ? NSTAGE : 1;
  const int nblk_u = rows_u_all > 0 ? (rows_u_all + g.rows_u - 1) / g.rows_u : 0;
  const int nst_u = ((HC * g.nc_max + g.rows_u - 1) / g.rows_u) > 1 ? NSTAGE : 1;

  const uint32_t bar0 = smem_u32(bars);
  auto barW = [&](int st) { return bar0 + 8u * st; };
  auto barU = [&](int st) { return bar0 + 16u + 8u * st; };

  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(bar0 + 8u * i, 1);
    fence_mbar_init();
  }
  __syncthreads();

  // --- weight copies.  Issued by warp 0: lane 0 arms the stage's mbarrier
  // with the stage's byte count, then the lanes issue one bulk copy per row.
  auto issue_w = [&](int blk) {
    const int st = blk % nst_w;
    const int n_lo = blk * g.rows_w, n_hi = min(n_out, n_lo + g.rows_w);
    const uint32_t bytes = static_cast<uint32_t>((n_hi - n_lo) * nch * 16);
    if (lane == 0) mbar_arrive_expect_tx(barW(st), bytes);
    __syncwarp();
    if (nch > 0) {
      for (int n = n_lo + lane; n < n_hi; n += 32) {
        const bf16_t* src = (n < r ? c.Wd + static_cast<int64_t>(n) * K
                                   : c.Wi + static_cast<int64_t>(n - r) * K) + k0;
        bulk_g2s(smem_u32(s_w + st * g.stage_w_bytes + (n - n_lo) * g.wstride), src,
                 static_cast<uint32_t>(nch * 16), barW(st));
      }
    }
  };
  auto issue_u = [&](int blk) {
    const int st = blk % nst_u;
    const int i_lo = blk * g.rows_u, i_hi = min(rows_u_all, i_lo + g.rows_u);
    if (lane == 0) mbar_arrive_expect_tx(barU(st), static_cast<uint32_t>((i_hi - i_lo) * r * 2));
    __syncwarp();
    for (int i = i_lo + lane; i < i_hi; i += 32) {
      const int ss = i / nc, cc = i % nc;
      const bf16_t* src = c.Wu + static_cast<int64_t>(ss * HS + cp0 + cc) * r;
      bulk_g2s(smem_u32(s_u + st * g.stage_u_bytes + (i - i_lo) * r * 2), src,
               static_cast<uint32_t>(r * 2), barU(st));
    }
  };
  if (warp == 0) {
    for (int blk = 0; blk < min(nst_w, g.nblk_w); ++blk) issue_w(blk);
    for (int blk = 0; blk < min(nst_u, nblk_u); ++blk) issue_u(blk);
  }

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
    float* a = s_act + m * g.wmax + ch * 8;
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
  bool ok = true;
  for (int blk = 0; blk < g.nblk_w; ++blk) {
    const int st = blk % nst_w;
    if (!mbar_wait_bounded(barW(st), (blk / nst_w) & 1, p.err, p.limit_ns)) { ok = false; break; }
    const int n_lo = blk * g.rows_w, n_hi = min(n_out, n_lo + g.rows_w);
    for (int n = n_lo + tid; n < n_hi; n += NT) {
      float acc[MB];
#pragma unroll
      for (int m = 0; m < MB; ++m) acc[m] = 0.f;
      const unsigned char* wrow = s_w + st * g.stage_w_bytes + (n - n_lo) * g.wstride;
      for (int ch = 0; ch < nch; ++ch) {
        float wf[8];
        unpack8(*reinterpret_cast<const uint4*>(wrow + ch * 16), wf);
#pragma unroll
        for (int m = 0; m < MB; ++m) {
          if (m < M) {
            const float4 a0 = *reinterpret_cast<const float4*>(s_act + m * g.wmax + ch * 8);
            const float4 a1 = *reinterpret_cast<const float4*>(s_act + m * g.wmax + ch * 8 + 4);
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
        if (m < M) p.part[(static_cast<int64_t>(b) * M + m) * n_out + n] = acc[m];
    }
    __syncthreads();
    if (warp == 0 && blk + nst_w < g.nblk_w) issue_w(blk + nst_w);
  }

  // A test hook: this CTA leaves before the first barrier, as if it had died.
  if (c.debug_fault == 1 && b == 0) ok = false;
  if (!ok) {
    // let this CTA's outstanding up-weight copies land before leaving
    for (int blk = 0; blk < min(nst_u, nblk_u); ++blk)
      mbar_wait_bounded(barU(blk % nst_u), 0, p.err, p.limit_ns);
    return;
  }
  if (!grid_barrier(p.bar, g.G, p.err, p.limit_ns, s_flag)) goto drain;

  // --- phase 2: rrms, then lora / inj_next as rrms-weighted sums of partials
  for (int i = tid; i < M * g.G; i += NT) {
    const int m = i / g.G, bb = i % g.G;
    s_ss[i] = __ldcg(p.sumsq + bb * M + m);
  }
  __syncthreads();
  for (int i = tid; i < M * HC; i += NT) {
    const int m = i / HC, ss = i % HC;
    const float* v = s_ss + m * g.G + ss * g.per_stream;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    int q = 0;
    for (; q + 4 <= g.per_stream; q += 4) { a0 += v[q]; a1 += v[q + 1]; a2 += v[q + 2]; a3 += v[q + 3]; }
    for (; q < g.per_stream; ++q) a0 += v[q];
    const float rr = 1.0f / sqrtf(((a0 + a1) + (a2 + a3)) / static_cast<float>(HS) + c.eps);
    s_rr[i] = rr;
    if (b == 0) c.rrms[i] = rr;
  }
  __syncthreads();
  {
    const int ntn = (n_out + 31) / 32;
    for (int t = b; t < M * ntn; t += g.G) {
      const int m = t / ntn;
      const int n = (t % ntn) * 32 + lane;
      float acc = 0.f;
      if (n < n_out) {
#pragma unroll 4
        for (int bb = warp; bb < g.G; bb += NW)
          acc = fmaf(s_rr[m * HC + bb / g.per_stream],
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
  }
  if (!grid_barrier(p.bar, g.G, p.err, p.limit_ns, s_flag)) goto drain;

  // --- phase 3: h, gates for this CTA's channels, gated mean
  for (int i = tid; i < M * r; i += NT) {
    const float u = __ldcg(c.lora + i) / static_cast<float>(HC);
    s_h[i] = u * sigmoidf_dev(u);
  }
  __syncthreads();
  for (int blk = 0; blk < nblk_u; ++blk) {
    const int st = blk % nst_u;
    if (!mbar_wait_bounded(barU(st), (blk / nst_u) & 1, p.err, p.limit_ns)) return;
    const int i_lo = blk * g.rows_u, i_hi = min(rows_u_all, i_lo + g.rows_u);
    for (int i = i_lo + warp; i < i_hi; i += NW) {
      const bf16_t* wu = reinterpret_cast<const bf16_t*>(s_u + st * g.stage_u_bytes) +
                         static_cast<int64_t>(i - i_lo) * r;
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
          if (lane == 0) s_g[m * HC * g.nc_max + i] = sigmoidf_dev(v);
        }
      }
    }
    __syncthreads();
    if (warp == 0 && blk + nst_u < nblk_u) issue_u(blk + nst_u);
  }
  for (int i = tid; i < M * nc; i += NT) {
    const int m = i / nc, cc = i % nc, ch = cp0 + cc;
    float acc = 0.f;
    for (int ss = 0; ss < HC; ++ss) {
      const int64_t k = static_cast<int64_t>(ss) * HS + ch;
      const float r2 = bf16_to_f32(__ldcg(c.R2 + static_cast<int64_t>(m) * K + k));
      const float xn = r2 * s_rr[m * HC + ss] * (1.0f + bf16_to_f32(__ldg(c.Wnorm + k)));
      acc = fmaf(s_g[m * HC * g.nc_max + ss * nc + cc], xn, acc);
    }
    c.x[static_cast<int64_t>(m) * HS + ch] = f32_to_bf16(acc / static_cast<float>(HC));
  }
  return;

drain:
  // A barrier failed: wait (bounded) for the prefetched up-weight copies.
  for (int blk = 0; blk < min(nst_u, nblk_u); ++blk)
    mbar_wait_bounded(barU(blk % nst_u), 0, p.err, p.limit_ns);
}

template <int MB>
cudaError_t launch_mb(const Params& prm, cudaStream_t stream) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<MB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_BUDGET) + 1024);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(prm.g.G);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = prm.g.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<MB>, prm);
}

}  // namespace

int decode_grid(const Device& dev, int HC, int HS) {
  const int per_stream = std::max(1, std::min(dev.sms / HC, HS / 8));
  return per_stream * HC;
}

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
  const int G = decode_grid(dev, c.HC, c.HS);
  const int M = static_cast<int>(c.M);
  const int MB = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : M <= 16 ? 16 : 32;
  if (!make_geom(c, G, MB, prm.g)) return cudaErrorInvalidConfiguration;
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

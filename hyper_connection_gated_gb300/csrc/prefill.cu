// Prefill path of the HC gated residual (large M): tensor-core kernels on
// tcgen05 with TMA-fed shared memory and tensor-memory accumulators.
//
// The split follows the page's two-stage design (aiter PR #5913, "Technical
// Details": Kernel 1 = COMBINE + N + G1 GEMM + INJ and writes R2 / rrms /
// lora / inj_next; Kernel 2 = SiLU + up-GEMM + gated mean with xn rebuilt from
// R2 * rrms * (1 + Wnorm), so xn and the gate never reach HBM), re-designed
// for sm_103a:
//
// K1, one CTA per (128-token tile, stream s).  Because rrms_s is constant over
//   stream s, lora = sum_s rrms_s * (R2_s . W_s^T): the CTA owns the whole
//   K-range of its stream, so it knows rrms_s at the end of its K-loop and
//   scales its partial product there.  Warp roles:
//     warp 8      TMA producer: R and y tiles (128 x 64, 128-byte swizzle),
//                 the matching 64 columns of Wd (all r rows) and of Wi;
//     warps 0-7   converters: R2 = bf16(R + y * iw) (written to HBM), sum of
//                 R2^2 and the inject dot products per row on the CUDA cores,
//                 and the MMA operand in place: R2 for a folded weight, else
//                 the hi/lo bf16 split of R2 * (1 + Wnorm) (two MMAs, so the
//                 product keeps ~16 mantissa bits);
//     warp 9      one thread issues tcgen05.mma (M=128, N=r split in <= 256
//                 column blocks) into tensor memory.
//   Epilogue (warps 0-7): rrms_s, inj_next partial, lora partial
//   rrms_s * acc -> part[s][m][:].
// R  (reduce): lora = sum_s part[s], inj_next = sum_s inj_part[s], and the
//   up-GEMM operand h = bf16(SiLU(lora / HC)).
// K2, persistent over (128-token tile, 64-channel block) units: A = h tile,
//   B = the HC * 64 rows {s * HS + c} of Wu, D = 128 x (HC * 64) fp32 in
//   tensor memory (double-buffered when it fits).  Epilogue warps read a
//   row's gates for all streams, apply sigmoid, rebuild xn from R2, rrms and
//   Wnorm and write x = (1/HC) * sum_s G * xn.
#include <algorithm>

#include "hc_gr_internal.cuh"
#include "tmap.h"

namespace hcgr {
namespace {

constexpr int BM = 128;   // token tile (MMA M)
constexpr int BK = 64;    // K block: one 128-byte swizzle row of bf16
constexpr uint32_t TILE_BYTES = BM * BK * 2;   // 16 KB

// ===================================================================== K1
constexpr int K1_CONV_WARPS = 8;
constexpr int K1_THREADS = (K1_CONV_WARPS + 2) * 32;
constexpr int K1_TMA_WARP = K1_CONV_WARPS;
constexpr int K1_MMA_WARP = K1_CONV_WARPS + 1;
constexpr int K1_NST = 2;

struct K1Params {
  CUtensorMap tm_R;    // [M][K], box {64, 128}, 128B swizzle
  CUtensorMap tm_y;    // [M][HS], box {64, 128}, 128B swizzle
  CUtensorMap tm_w;    // Wd [r][K], box {64, wbox_rows}, 128B swizzle
  CUtensorMap tm_wi;   // Wi [HC][K], box {64, HC}
  const float* inj;
  int64_t ld_inj;
  const bf16_t* Wnorm;
  bf16_t* R2;
  float* rrms;
  float* part;        // [HC][M][r]
  float* inj_part;    // [HC][M][HC]
  int M, HC, HS, K, r, fold;
  float eps;
  int nkb, wbox_rows, nwbox, mma_n, n_mma;
  uint32_t stage_bytes, tmem_cols;
  int* err;
  uint64_t limit_ns;
};

struct K1Smem {
  uint32_t off_b, off_wi, off_bar, off_rowss, off_rowinj, total;
};

__host__ __device__ inline K1Smem k1_smem(int r, int HC) {
  K1Smem s;
  s.off_b = 2 * TILE_BYTES;
  s.off_wi = s.off_b + r * 128;
  const uint32_t stage = s.off_wi + ((HC * 128 + 1023) / 1024) * 1024;
  s.off_bar = K1_NST * stage;
  s.off_rowss = s.off_bar + 128;
  s.off_rowinj = s.off_rowss + BM * 4;
  s.total = s.off_rowinj + BM * HC * 4;
  return s;
}

__global__ void __launch_bounds__(K1_THREADS, 1) k1_kernel(const __grid_constant__ K1Params p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const K1Smem L = k1_smem(p.r, p.HC);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s = blockIdx.x % p.HC;
  const int m0 = (blockIdx.x / p.HC) * BM;
  const int HC = p.HC, HS = p.HS, r = p.r, nkb = p.nkb;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar = sbase + L.off_bar;
  auto full = [&](int st) { return bar + 8u * st; };
  auto conv = [&](int st) { return bar + 16u + 8u * st; };
  auto freeb = [&](int st) { return bar + 32u + 8u * st; };
  const uint32_t accb = bar + 48u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.off_bar + 64);
  float* rowss = reinterpret_cast<float*>(smem + L.off_rowss);
  float* rowinj = reinterpret_cast<float*>(smem + L.off_rowinj);

  if (tid == 0) {
    for (int i = 0; i < K1_NST; ++i) {
      mbar_init(full(i), 1);
      mbar_init(conv(i), K1_CONV_WARPS);
      mbar_init(freeb(i), 1);
    }
    mbar_init(accb, 1);
    fence_mbar_init();
  }
  if (warp == K1_MMA_WARP) {
    tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == K1_TMA_WARP) {
    if (lane == 0) {
      int last_issued[K1_NST] = {-1, -1};
      bool ok = true;
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int st = kb % K1_NST;
        if (kb >= K1_NST)
          ok = mbar_wait_bounded(freeb(st), ((kb / K1_NST) - 1) & 1, p.err, p.limit_ns);
        if (!ok) break;
        const uint32_t sb = sbase + st * p.stage_bytes;
        mbar_arrive_expect_tx(full(st), 2 * TILE_BYTES + r * 128 + HC * 128);
        tma_load_2d(sb, &p.tm_R, s * HS + kb * BK, m0, full(st));
        tma_load_2d(sb + TILE_BYTES, &p.tm_y, kb * BK, m0, full(st));
        for (int bx = 0; bx < p.nwbox; ++bx)
          tma_load_2d(sb + L.off_b + bx * p.wbox_rows * 128, &p.tm_w, s * HS + kb * BK,
                      bx * p.wbox_rows, full(st));
        tma_load_2d(sb + L.off_wi, &p.tm_wi, s * HS + kb * BK, 0, full(st));
        last_issued[st] = kb;
      }
      // outstanding copies land before the CTA can leave
      for (int st = 0; st < K1_NST; ++st)
        if (last_issued[st] >= 0)
          mbar_wait_bounded(full(st), (last_issued[st] / K1_NST) & 1, p.err, p.limit_ns);
    }
  } else if (warp == K1_MMA_WARP) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(BM, p.mma_n);
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb) {
        const int st = kb % K1_NST;
        ok = mbar_wait_bounded(conv(st), (kb / K1_NST) & 1, p.err, p.limit_ns);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sb = sbase + st * p.stage_bytes;
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks) {
          const uint64_t a_hi = desc_sw128(sb + ks * 32);
          const uint64_t a_lo = desc_sw128(sb + TILE_BYTES + ks * 32);
          for (int nn = 0; nn < p.n_mma; ++nn) {
            const uint64_t bd = desc_sw128(sb + L.off_b + nn * p.mma_n * 128 + ks * 32);
            umma_bf16(tmem + nn * p.mma_n, a_hi, bd, idesc, (kb | ks) != 0);
            if (!p.fold) umma_bf16(tmem + nn * p.mma_n, a_lo, bd, idesc, 1);
          }
        }
        umma_commit(freeb(st));
      }
      umma_commit(accb);
      mbar_wait_bounded(accb, 0, p.err, p.limit_ns);
    }
  } else {
    // ---------------- converters: warps 0-7.  Thread t owns row t / 2 of the
    // tile and channel chunks 4 * (t & 1) .. +3 (8 channels each) of every
    // K block, so its row's partial sums stay in registers.  In the 128-byte
    // swizzled tile chunk c of row i sits at i * 128 + ((c ^ (i & 7)) << 4);
    // any 8 consecutive threads touch 8 distinct chunk positions, so the
    // shared-memory accesses are free of bank conflicts.
    const int row = tid >> 1, cbase = (tid & 1) * 4;
    const int m = m0 + row;
    const bool valid = m < p.M;
    const float iw =
        valid ? 2.0f * sigmoidf_dev(p.inj[m * p.ld_inj + s] / static_cast<float>(HC)) : 0.f;
    float ss = 0.f, ij[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) ij[j] = 0.f;
    bf16_t* r2row = p.R2 + static_cast<int64_t>(valid ? m : 0) * p.K + static_cast<int64_t>(s) * HS;
    bool ok = true;
    for (int kb = 0; kb < nkb; ++kb) {
      const int st = kb % K1_NST;
      ok = mbar_wait_bounded(full(st), (kb / K1_NST) & 1, p.err, p.limit_ns);
      if (!ok) break;
      unsigned char* sb = smem + st * p.stage_bytes;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int ch = cbase + i;
        const int col = kb * BK + ch * 8;           // channel within the stream
        const uint32_t off = row * 128 + ((ch ^ (row & 7)) << 4);
        float rv[8], yv[8], wn[8], a[8];
        unpack8(*reinterpret_cast<const uint4*>(sb + off), rv);
        unpack8(*reinterpret_cast<const uint4*>(sb + TILE_BYTES + off), yv);
        unpack8(__ldg(reinterpret_cast<const uint4*>(p.Wnorm + static_cast<int64_t>(s) * HS + col)), wn);
        uint32_t pr[4], ph[4], pl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pr[e] = pack2(fmaf(yv[2 * e], iw, rv[2 * e]), fmaf(yv[2 * e + 1], iw, rv[2 * e + 1]));
          const float r0 = lo_bf16(pr[e]), r1 = hi_bf16(pr[e]);
          ss = fmaf(r0, r0, ss);
          ss = fmaf(r1, r1, ss);
          a[2 * e] = p.fold ? r0 : r0 * (1.0f + wn[2 * e]);
          a[2 * e + 1] = p.fold ? r1 : r1 * (1.0f + wn[2 * e + 1]);
          ph[e] = pack2(a[2 * e], a[2 * e + 1]);
          pl[e] = pack2(a[2 * e] - lo_bf16(ph[e]), a[2 * e + 1] - hi_bf16(ph[e]));
        }
        if (valid)
          *reinterpret_cast<uint4*>(r2row + col) = make_uint4(pr[0], pr[1], pr[2], pr[3]);
        if (p.fold) {
          *reinterpret_cast<uint4*>(sb + off) = make_uint4(pr[0], pr[1], pr[2], pr[3]);
        } else {
          *reinterpret_cast<uint4*>(sb + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
          *reinterpret_cast<uint4*>(sb + TILE_BYTES + off) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j < HC) {
            float wi[8];
            unpack8(*reinterpret_cast<const uint4*>(sb + L.off_wi + j * 128 + ch * 16), wi);
            float t = ij[j];
#pragma unroll
            for (int e = 0; e < 8; ++e) t = fmaf(a[e], wi[e], t);
            ij[j] = t;
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(conv(st));
    }
    // per-row totals: the two threads of a row are lanes 2i and 2i+1
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
#pragma unroll
    for (int j = 0; j < 8; ++j) ij[j] += __shfl_xor_sync(0xffffffffu, ij[j], 1);
    if ((tid & 1) == 0) {
      rowss[row] = ss;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < HC) rowinj[row * HC + j] = ij[j];
    }
    named_bar_sync(1, K1_CONV_WARPS * 32);
    // ---------------- epilogue: rrms_s, inj partial, lora partial
    if (ok) ok = mbar_wait_bounded(accb, 0, p.err, p.limit_ns);
    tc_fence_after();
    const int q = warp & 3, half = warp >> 2;
    const int erow = 32 * q + lane;
    const int em = m0 + erow;
    const bool v = em < p.M;
    const float rr = 1.0f / sqrtf(rowss[erow] / static_cast<float>(HS) + p.eps);
    if (v && half == 0) {
      p.rrms[static_cast<int64_t>(em) * HC + s] = rr;
      for (int j = 0; j < HC; ++j)
        p.inj_part[(static_cast<int64_t>(s) * p.M + em) * HC + j] = rr * rowinj[erow * HC + j];
    }
    if (ok) {
      const int cols = r / 2;
      float* dst = p.part + (static_cast<int64_t>(s) * p.M + (v ? em : 0)) * r + half * cols;
      for (int c0 = 0; c0 < cols; c0 += 16) {
        uint32_t acc[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + half * cols + c0, acc);
        tmem_ld_wait();
        if (v) {
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(dst + c0 + e) =
                make_float4(__uint_as_float(acc[e]) * rr, __uint_as_float(acc[e + 1]) * rr,
                            __uint_as_float(acc[e + 2]) * rr, __uint_as_float(acc[e + 3]) * rr);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == K1_MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

// ================================================================ reduce
__global__ void k1_reduce_kernel(const float* __restrict__ part, const float* __restrict__ inj_part,
                                 float* __restrict__ lora, float* __restrict__ inj_next,
                                 bf16_t* __restrict__ h, int64_t M, int HC, int r) {
  const int64_t n4 = M * r / 4;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const float inv_hc = 1.0f / static_cast<float>(HC);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 acc = reinterpret_cast<const float4*>(part)[i];
    for (int s = 1; s < HC; ++s) {
      const float4 v = reinterpret_cast<const float4*>(part)[s * n4 + i];
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    reinterpret_cast<float4*>(lora)[i] = acc;
    const float u0 = acc.x * inv_hc, u1 = acc.y * inv_hc, u2 = acc.z * inv_hc, u3 = acc.w * inv_hc;
    uint2 hv;
    hv.x = pack2(u0 * sigmoidf_dev(u0), u1 * sigmoidf_dev(u1));
    hv.y = pack2(u2 * sigmoidf_dev(u2), u3 * sigmoidf_dev(u3));
    reinterpret_cast<uint2*>(h)[i] = hv;
  }
  const int64_t ni = M * HC;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < ni; i += stride) {
    float acc = inj_part[i];
    for (int s = 1; s < HC; ++s) acc += inj_part[s * ni + i];
    inj_next[i] = acc;
  }
}

// ===================================================================== K2
constexpr int K2_THREADS = 384;
constexpr int K2_TMA_WARP = 0;
constexpr int K2_MMA_WARP = 1;
constexpr int K2_ALLOC_WARP = 2;
constexpr int K2_EPI_WARP0 = 4;
constexpr int K2_EPI_WARPS = 8;
constexpr int NC = 64;   // channels per unit

struct K2Params {
  CUtensorMap tm_h;    // h [M][r], box {64, 128}, 128B swizzle
  CUtensorMap tm_wu;   // Wu [K][r], box {64, 64}, 128B swizzle
  const bf16_t* R2;
  const float* rrms;
  const bf16_t* Wnorm;
  bf16_t* x;
  int M, HC, HS, K, r;
  int nkb, ncb, n_units, nst, nacc, ncols_acc;
  uint32_t stage_bytes, tmem_cols, wn_bytes;
  int* err;
  uint64_t limit_ns;
};

template <int HCT>
__global__ void __launch_bounds__(K2_THREADS, 1) k2_kernel(const __grid_constant__ K2Params p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int HC = HCT;
  const int HS = p.HS, nkb = p.nkb, nst = p.nst, nacc = p.nacc;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar = sbase + nst * p.stage_bytes;
  const uint32_t wnbar = bar + 160u;
  const bf16_t* s_wn = reinterpret_cast<const bf16_t*>(smem + nst * p.stage_bytes + 256);
  auto full = [&](int st) { return bar + 8u * st; };
  auto freeb = [&](int st) { return bar + 64u + 8u * st; };
  auto accfull = [&](int a) { return bar + 128u + 8u * a; };
  auto accfree = [&](int a) { return bar + 144u + 8u * a; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + nst * p.stage_bytes + 192);

  if (tid == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(full(i), 1);
      mbar_init(freeb(i), 1);
    }
    for (int a = 0; a < nacc; ++a) {
      mbar_init(accfull(a), 1);
      mbar_init(accfree(a), K2_EPI_WARPS);
    }
    mbar_init(wnbar, 1);
    fence_mbar_init();
  }
  if (warp == K2_ALLOC_WARP) {
    tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_local = p.n_units > static_cast<int>(blockIdx.x)
                          ? (p.n_units - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  if (warp == K2_TMA_WARP) {
    if (lane == 0) {
      // Wnorm, staged once for the epilogue
      mbar_arrive_expect_tx(wnbar, p.wn_bytes);
      bulk_g2s(smem_u32(s_wn), p.Wnorm, p.wn_bytes, wnbar);
      int g = 0;
      bool ok = true;
      int last_g[8];
      for (int i = 0; i < 8; ++i) last_g[i] = -1;
      for (int i = 0; i < n_local && ok; ++i) {
        const int u = blockIdx.x + i * gridDim.x;
        const int t = u / p.ncb, cb = u % p.ncb;
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int st = g % nst;
          if (g >= nst) ok = mbar_wait_bounded(freeb(st), ((g / nst) - 1) & 1, p.err, p.limit_ns);
          if (!ok) break;
          const uint32_t sb = sbase + st * p.stage_bytes;
          mbar_arrive_expect_tx(full(st), TILE_BYTES + HC * NC * 128);
          tma_load_2d(sb, &p.tm_h, kb * BK, t * BM, full(st));
          for (int ss = 0; ss < HC; ++ss)
            tma_load_2d(sb + TILE_BYTES + ss * NC * 128, &p.tm_wu, kb * BK, ss * HS + cb * NC,
                        full(st));
          last_g[st] = g;
        }
      }
      for (int st = 0; st < nst; ++st)
        if (last_g[st] >= 0) mbar_wait_bounded(full(st), (last_g[st] / nst) & 1, p.err, p.limit_ns);
      mbar_wait_bounded(wnbar, 0, p.err, p.limit_ns);
    }
  } else if (warp == K2_MMA_WARP) {
    if (lane == 0) {
      const int N = HC * NC;
      int g = 0;
      bool ok = true;
      int issued = 0;
      for (int i = 0; i < n_local && ok; ++i) {
        const int ab = i % nacc;
        if (i >= nacc) ok = mbar_wait_bounded(accfree(ab), ((i / nacc) - 1) & 1, p.err, p.limit_ns);
        if (!ok) break;
        tc_fence_after();
        const uint32_t dcol = tmem + ab * p.ncols_acc;
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int st = g % nst;
          ok = mbar_wait_bounded(full(st), (g / nst) & 1, p.err, p.limit_ns);
          if (!ok) break;
          tc_fence_after();
          const uint32_t sb = sbase + st * p.stage_bytes;
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {
            const uint64_t ad = desc_sw128(sb + ks * 32);
            for (int n0 = 0; n0 < N; n0 += 256) {
              const int nn = min(256, N - n0);
              const uint64_t bd = desc_sw128(sb + TILE_BYTES + n0 * 128 + ks * 32);
              umma_bf16(dcol + n0, ad, bd, idesc_bf16(BM, nn), (kb | ks) != 0);
            }
          }
          umma_commit(freeb(st));
        }
        if (!ok) break;
        umma_commit(accfull(ab));
        ++issued;
      }
      // all issued MMAs finish before tensor memory is released
      if (issued > 0) {
        const int last = issued - 1;
        mbar_wait_bounded(accfull(last % nacc), (last / nacc) & 1, p.err, p.limit_ns);
      }
    }
  } else if (warp >= K2_EPI_WARP0) {
    // Epilogue: thread = one token row (TMEM lane), 32 channels of the unit
    // (warps 4-7 the first half, 8-11 the second).  Channels go in chunks of
    // CC; the R2 values of chunk q+1 are loaded while chunk q is computed, and
    // those of chunk 0 (and rrms) before waiting for the accumulator.
    constexpr int CC = HC <= 4 ? 16 : 8;
    constexpr int NCH = 32 / CC;
    constexpr int V = CC / 8;
    const int ew = warp - K2_EPI_WARP0;
    const int q4 = warp & 3, half = ew >> 2;
    const float inv_hc = 1.0f / static_cast<float>(HC);
    bool wn_ready = mbar_wait_bounded(wnbar, 0, p.err, p.limit_ns);
    for (int i = 0; i < n_local && wn_ready; ++i) {
      const int u = blockIdx.x + i * gridDim.x;
      const int t = u / p.ncb, cb = u % p.ncb;
      const int ab = i % nacc;
      const int row = 32 * q4 + lane;
      const int64_t m = static_cast<int64_t>(t) * BM + row;
      const bool v = m < p.M;
      const int cbase = cb * NC + half * 32;          // first channel of this thread
      const bf16_t* r2p = p.R2 + (v ? m : 0) * p.K + cbase;
      float rr[HC];
      uint4 bufA[HC][V], bufB[HC][V];
#pragma unroll
      for (int ss = 0; ss < HC; ++ss) rr[ss] = v ? __ldg(p.rrms + m * HC + ss) : 0.f;
      auto load = [&](int q, uint4 (&buf)[HC][V]) {
#pragma unroll
        for (int ss = 0; ss < HC; ++ss)
#pragma unroll
          for (int j = 0; j < V; ++j)
            buf[ss][j] = v ? __ldg(reinterpret_cast<const uint4*>(r2p + ss * HS + q * CC + j * 8))
                           : make_uint4(0, 0, 0, 0);
      };
      load(0, bufA);
      if (!mbar_wait_bounded(accfull(ab), (i / nacc) & 1, p.err, p.limit_ns)) break;
      tc_fence_after();
      const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q4) << 16) + ab * p.ncols_acc;
#pragma unroll
      for (int q = 0; q < NCH; ++q) {
        uint4 (&cur)[HC][V] = (q & 1) ? bufB : bufA;
        uint4 (&nxt)[HC][V] = (q & 1) ? bufA : bufB;
        if (q + 1 < NCH) load(q + 1, nxt);
        float acc[CC];
#pragma unroll
        for (int e = 0; e < CC; ++e) acc[e] = 0.f;
#pragma unroll
        for (int ss = 0; ss < HC; ++ss) {
          uint32_t gv[CC];
          if constexpr (CC == 16) tmem_ld16(tbase + ss * NC + half * 32 + q * CC, gv);
          else tmem_ld8(tbase + ss * NC + half * 32 + q * CC, gv);
          tmem_ld_wait();
          float r2[CC], wn[CC];
#pragma unroll
          for (int j = 0; j < V; ++j) {
            unpack8(cur[ss][j], r2 + 8 * j);
            unpack8(*reinterpret_cast<const uint4*>(s_wn + ss * HS + cbase + q * CC + j * 8), wn + 8 * j);
          }
#pragma unroll
          for (int e = 0; e < CC; ++e) {
            const float G = sigmoid_tanh(__uint_as_float(gv[e]));
            acc[e] = fmaf(G, r2[e] * rr[ss] * (1.0f + wn[e]), acc[e]);
          }
        }
        if (v) {
          uint32_t o[CC / 2];
#pragma unroll
          for (int e = 0; e < CC / 2; ++e) o[e] = pack2(acc[2 * e] * inv_hc, acc[2 * e + 1] * inv_hc);
          uint4* xp = reinterpret_cast<uint4*>(p.x + m * HS + cbase + q * CC);
#pragma unroll
          for (int j = 0; j < V; ++j) xp[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(accfree(ab));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == K2_ALLOC_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

uint32_t pow2_cols(int n) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(n)) c <<= 1;
  return c;
}

template <int HCT>
cudaError_t launch_k2(const K2Params& p, int grid, size_t smem, const Device& dev,
                      cudaStream_t stream) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k2_kernel<HCT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, dev.smem_optin);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  k2_kernel<HCT><<<grid, K2_THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

bool prefill_supported(const Call& c) {
  return c.HS % 64 == 0 && c.r % 64 == 0 && c.r <= 512 && c.HC >= 1 && c.HC <= 8;
}

}  // namespace

size_t prefill_ws_bytes(int64_t max_M, int HC, int HS, int r) {
  (void)HS;
  const size_t part = static_cast<size_t>(HC) * max_M * r * 4;
  const size_t injp = static_cast<size_t>(HC) * max_M * HC * 4;
  const size_t h = static_cast<size_t>(max_M) * r * 2;
  return part + 256 + injp + 256 + h + 256;
}

cudaError_t launch_prefill(const Call& c, const Workspace& ws, const Device& dev,
                           cudaStream_t stream) {
  if (!prefill_supported(c)) return cudaErrorNotSupported;
  if (prefill_ws_bytes(c.M, c.HC, c.HS, c.r) > ws.prefill_bytes) return cudaErrorNotSupported;
  const int M = static_cast<int>(c.M);
  const int n_mt = (M + BM - 1) / BM;
  // workspace carve-up (sized by prefill_ws_bytes for max_M)
  float* part = ws.k1_part;
  float* inj_part = reinterpret_cast<float*>(
      reinterpret_cast<unsigned char*>(part) + ((static_cast<size_t>(c.HC) * M * c.r * 4 + 255) / 256) * 256);
  bf16_t* h = reinterpret_cast<bf16_t*>(
      reinterpret_cast<unsigned char*>(inj_part) + ((static_cast<size_t>(c.HC) * M * c.HC * 4 + 255) / 256) * 256);

  // ---------------- K1
  static bool k1_attr = false;
  {
    K1Params p;
    const uint64_t dR[2] = {static_cast<uint64_t>(c.K), static_cast<uint64_t>(M)};
    const uint64_t sR[1] = {static_cast<uint64_t>(c.K) * 2};
    const uint32_t bT[2] = {BK, BM};
    if (!make_tmap_bf16(&p.tm_R, c.R, 2, dR, sR, bT, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    const uint64_t dy[2] = {static_cast<uint64_t>(c.HS), static_cast<uint64_t>(M)};
    const uint64_t sy[1] = {static_cast<uint64_t>(c.HS) * 2};
    if (!make_tmap_bf16(&p.tm_y, c.y, 2, dy, sy, bT, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    p.nwbox = c.r > 256 ? 2 : 1;
    p.wbox_rows = c.r / p.nwbox;
    const uint64_t dw[2] = {static_cast<uint64_t>(c.K), static_cast<uint64_t>(c.r)};
    const uint32_t bw[2] = {BK, static_cast<uint32_t>(p.wbox_rows)};
    if (!make_tmap_bf16(&p.tm_w, c.Wd, 2, dw, sR, bw, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    const uint64_t di[2] = {static_cast<uint64_t>(c.K), static_cast<uint64_t>(c.HC)};
    const uint32_t bi[2] = {BK, static_cast<uint32_t>(c.HC)};
    if (!make_tmap_bf16(&p.tm_wi, c.Wi, 2, di, sR, bi)) return cudaErrorInvalidValue;
    p.inj = c.inj;
    p.ld_inj = c.ld_inj;
    p.Wnorm = c.Wnorm;
    p.R2 = c.R2;
    p.rrms = c.rrms;
    p.part = part;
    p.inj_part = inj_part;
    p.M = M;
    p.HC = c.HC;
    p.HS = c.HS;
    p.K = c.K;
    p.r = c.r;
    p.fold = c.fold;
    p.eps = c.eps;
    p.nkb = c.HS / BK;
    p.n_mma = c.r > 256 ? 2 : 1;
    p.mma_n = c.r / p.n_mma;
    const K1Smem L = k1_smem(c.r, c.HC);
    p.stage_bytes = L.off_bar / K1_NST;
    p.tmem_cols = pow2_cols(c.r);
    p.err = ws.err;
    p.limit_ns = 1000ull * 1000 * 1000;
    const size_t smem = L.total + 1024;
    if (smem > static_cast<size_t>(dev.smem_optin)) return cudaErrorNotSupported;
    if (!k1_attr) {
      cudaError_t e = cudaFuncSetAttribute(k1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           dev.smem_optin);
      if (e != cudaSuccess) return e;
      k1_attr = true;
    }
    k1_kernel<<<n_mt * c.HC, K1_THREADS, smem, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // ---------------- reduce
  {
    const int64_t n4 = c.M * c.r / 4;
    const int blocks = static_cast<int>(std::min<int64_t>((n4 + 255) / 256, dev.sms * 8));
    k1_reduce_kernel<<<std::max(blocks, 1), 256, 0, stream>>>(part, inj_part, c.lora, c.inj_next, h,
                                                             c.M, c.HC, c.r);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // ---------------- K2
  {
    K2Params p;
    const uint64_t dh[2] = {static_cast<uint64_t>(c.r), static_cast<uint64_t>(M)};
    const uint64_t sh[1] = {static_cast<uint64_t>(c.r) * 2};
    const uint32_t bh[2] = {BK, BM};
    if (!make_tmap_bf16(&p.tm_h, h, 2, dh, sh, bh, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    const uint64_t du[2] = {static_cast<uint64_t>(c.r), static_cast<uint64_t>(c.K)};
    const uint32_t bu[2] = {BK, NC};
    if (!make_tmap_bf16(&p.tm_wu, c.Wu, 2, du, sh, bu, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    p.R2 = c.R2;
    p.rrms = c.rrms;
    p.Wnorm = c.Wnorm;
    p.x = c.x;
    p.M = M;
    p.HC = c.HC;
    p.HS = c.HS;
    p.K = c.K;
    p.r = c.r;
    p.nkb = c.r / BK;
    p.ncb = c.HS / NC;
    p.n_units = n_mt * p.ncb;
    p.stage_bytes = TILE_BYTES + c.HC * NC * 128;
    p.wn_bytes = static_cast<uint32_t>(c.K) * 2;
    const int budget = dev.smem_optin - 1024 - 256 - static_cast<int>(p.wn_bytes);
    p.nst = std::min(4, budget / static_cast<int>(p.stage_bytes));
    if (p.nst < 2) return cudaErrorNotSupported;
    p.ncols_acc = c.HC * NC;
    p.nacc = 2 * p.ncols_acc <= 512 ? 2 : 1;
    p.tmem_cols = pow2_cols(p.nacc * p.ncols_acc);
    p.err = ws.err;
    p.limit_ns = 1000ull * 1000 * 1000;
    const size_t smem = static_cast<size_t>(p.nst) * p.stage_bytes + 256 + p.wn_bytes + 1024;
    const int grid = std::min(p.n_units, dev.sms);
    cudaError_t e = cudaSuccess;
    switch (c.HC) {
      case 1: e = launch_k2<1>(p, grid, smem, dev, stream); break;
      case 2: e = launch_k2<2>(p, grid, smem, dev, stream); break;
      case 3: e = launch_k2<3>(p, grid, smem, dev, stream); break;
      case 4: e = launch_k2<4>(p, grid, smem, dev, stream); break;
      case 5: e = launch_k2<5>(p, grid, smem, dev, stream); break;
      case 6: e = launch_k2<6>(p, grid, smem, dev, stream); break;
      case 7: e = launch_k2<7>(p, grid, smem, dev, stream); break;
      default: e = launch_k2<8>(p, grid, smem, dev, stream); break;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace hcgr

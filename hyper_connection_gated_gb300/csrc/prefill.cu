// Prefill path of the HC gated residual (large M): tensor-core kernels on
// tcgen05 with TMA-fed shared memory and tensor-memory accumulators.
//
// The split follows the page's two-stage design (aiter PR #5913, "Technical
// Details": Kernel 1 = COMBINE + N + G1 GEMM + INJ and writes R2 / rrms /
// lora / inj_next; Kernel 2 = SiLU + up-GEMM + gated mean with xn rebuilt from
// R2 * rrms * (1 + Wnorm), so xn and the gate never reach HBM), re-designed
// for sm_103a:
//
// K1, one CTA per (128-token tile, stream s, K chunk of that stream).  Because
//   rrms_s is constant over stream s, lora = sum_s rrms_s * (R2_s . W_s^T):
//   the products are accumulated per stream without rrms and scaled later.
//   Warp roles:
//     warp 8      TMA: R and y tiles (128 x 64, 128-byte swizzle) and the K
//                 block's Wnorm values into the R/y ring;
//     warp 10     TMA: the matching 64 columns of the Wd rows and of the
//                 inject rows, in one or two column blocks, into the weight
//                 ring;
//     warps 0-7   converters: R2 = bf16(R + y * iw) (written to HBM), the sum
//                 of R2^2 per row, and the MMA operand in place: R2 for a
//                 folded weight, else the hi/lo bf16 split of R2 * (1 + Wnorm)
//                 (two MMAs, so the product keeps ~16 mantissa bits);
//     warps 9, 11 tcgen05.mma, one column block each (M=128, N = r + 16: the
//                 Wd rows and the inject rows, in <= 256-column blocks), one
//                 elected lane issuing; warp 9 also owns the TMEM allocation.
//   When r + 16 exceeds the 512 tensor-memory columns the inject dot
//   products run on the converters' CUDA cores instead.  The epilogue writes
//   the partial sums of squares and the un-scaled partial products.  Without
//   y (the mix alone) the converters take R as R2 and store nothing for it;
//   the Wnorm slice of stream s starts at s * ld_wnorm (0 for one [HS] norm
//   weight shared by the streams).
// R  (reduce): rrms_s from the partial sums of squares, lora / inj_next =
//   sum_s rrms_s * (sum of the stream's partial products), and the up-GEMM
//   operand hh = bf16(SiLU(lora / HC) / 2).  With few token tiles K1 splits
//   each stream's K range into chunks so that the CTAs cover the SMs.  The
//   partials are laid out [tile][stream, chunk][column][128 rows]: column-major
//   inside a token tile, so K1's epilogue (a thread per row) stores whole
//   128-byte lines and the reduce reads them as float4 runs.
// K2, persistent over (128-token tile, NCU-channel block) units with
//   N = HC * NCU = 256 for HC = 4 and 8: A = hh tile, B = the HC * NCU rows
//   {s * HS + c} of Wu, D = 128 x N fp32 (G / 2) in double-buffered tensor
//   memory.  The unit's R2 tile and 1 + Wnorm stream through a ring of
//   per-stream slots; epilogue warps read a row's gates stream by stream,
//   apply sigmoid, rebuild xn from R2, rrms and 1 + Wnorm and store
//   x = (1/HC) * sum_s G * xn.  For the mix alone, R itself is the R2 tile.
#include <cstring>
#include <algorithm>
#include <type_traits>
#include <utility>

#include "hc_gr_internal.cuh"
#include "tmap.h"

namespace hcgr {
namespace {

constexpr int BM = 128;   // token tile (MMA M)
constexpr int BK = 64;    // K block: one 128-byte swizzle row of bf16
constexpr uint32_t TILE_BYTES = BM * BK * 2;   // 16 KB

// ===================================================================== K1
// Shared memory holds two rings: R/y slots (the R and y tiles of one K block,
// 32 KB, converted in place into the MMA's A operand) and weight slots (one
// column block of the B tile: Wd rows, plus the inject rows in the last
// block).  The R/y ring runs deeper because its tiles come from HBM; the
// weights are L2-resident.
constexpr int K1_CONV_WARPS = 8;
constexpr int K1_RY_WARP = 8;     // TMA: R, y tiles and the K block's Wnorm values
constexpr int K1_MMA_WARP = 9;    // MMAs of column block 0 (and the TMEM allocation)
constexpr int K1_W_WARP = 10;     // TMA: weight column blocks
constexpr int K1_MMA1_WARP = 11;  // MMAs of column block 1
constexpr int K1_THREADS = 12 * 32;
constexpr int K1_MAX_RY = 6;
constexpr int K1_MAX_W = 8;
constexpr uint32_t RY_BYTES = 2 * TILE_BYTES;
constexpr uint32_t K1_BAR_BYTES = 512;
constexpr int WI_ROWS = 16;   // inject rows in the MMA's B tile (HC real, rest zero-filled)

struct K1Params {
  CUtensorMap tm_R;    // [M][K], box {64, 128}, 128B swizzle
  CUtensorMap tm_y;    // [M][HS], box {64, 128}, 128B swizzle (unused when !has_y)
  CUtensorMap tm_w0;   // Wd rows [0, wrows0): box {64, wrows0}, 128B swizzle
  CUtensorMap tm_w1;   // Wd rows [wrows0, r): box {64, r - wrows0}, 128B swizzle
  CUtensorMap tm_wi;   // Wi [HC][K], box {64, 16} (128B swizzle) or {64, HC} (plain)
  const float* inj;
  int64_t ld_inj;
  bf16_t* R2;         // NULL: R2 not stored (mix only)
  const bf16_t* Wnorm;
  int64_t ld_wnorm;   // HS, or 0 when one [HS] Wnorm is shared by every stream
  float* part;        // [tile][HC * S][np][128 rows]: lora columns, then the HC inject columns
  float* sumsq;       // [tile][HC * S][128 rows] partial sums of R2^2
  int M, HS, K, r, np, fold;
  int has_y;          // 0: mix only -- R is already the combined residual, y and inj unused
  int S;              // K chunks per stream
  int nkb;
  int n1, n2;         // MMA column blocks (B rows): [0, n1) and [n1, n1 + n2); n2 may be 0
  int wrows0;         // Wd rows in column block 0 (the rest, and the inject rows, in block 1)
  int nry, nw;        // ring depths
  uint32_t w_slot, tmem_cols;
  uint32_t off_w, off_wn, off_wic, off_bar, off_rowss, off_rowinj;
  int* err;
  uint64_t limit_ns;
};

template <int HCT, bool INJ_MMA>
__global__ void __launch_bounds__(K1_THREADS, 1) k1_kernel(const __grid_constant__ K1Params p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int HC = HCT;
  const int NRY = p.nry, NW = p.nw;
  const int nh = p.n2 > 0 ? 2 : 1;   // weight column blocks per K block
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = blockIdx.x % p.S;
  const int s = (blockIdx.x / p.S) % HC;
  const int m0 = (blockIdx.x / (p.S * HC)) * BM;
  const int pid = s * p.S + chunk;                 // partial index
  const int HS = p.HS, r = p.r;
  const int kb0 = chunk * p.nkb / p.S, kb1 = (chunk + 1) * p.nkb / p.S;
  const int nkb = kb1 - kb0;                       // K blocks of this CTA
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar = sbase + p.off_bar;
  auto ryfull = [&](int st) { return bar + 8u * st; };
  auto conv = [&](int st) { return bar + 48u + 8u * st; };
  auto ryfree = [&](int st) { return bar + 96u + 8u * st; };
  auto wfull = [&](int ws) { return bar + 144u + 8u * ws; };
  auto wfree = [&](int ws) { return bar + 208u + 8u * ws; };
  const uint32_t accb = bar + 272u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.off_bar + 280);
  float* rowss = reinterpret_cast<float*>(smem + p.off_rowss);
  float* rowinj = reinterpret_cast<float*>(smem + p.off_rowinj);

  if (tid == 0) {
    prefetch_tmap(&p.tm_R);
    if (p.has_y) prefetch_tmap(&p.tm_y);
    prefetch_tmap(&p.tm_w0);
    prefetch_tmap(&p.tm_w1);
    prefetch_tmap(&p.tm_wi);
    for (int i = 0; i < NRY; ++i) {
      mbar_init(ryfull(i), 1);
      mbar_init(conv(i), K1_CONV_WARPS);
      mbar_init(ryfree(i), nh);
    }
    for (int i = 0; i < NW; ++i) {
      mbar_init(wfull(i), 1);
      mbar_init(wfree(i), 1);
    }
    mbar_init(accb, nh);
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
  // Launched as a programmatic dependent (hc_gr_args.pdl) this prologue may
  // overlap the previous kernel in the stream; its inputs and outputs are
  // touched only after that kernel has finished.  A no-op otherwise.
  grid_dep_wait();

  if (warp == K1_RY_WARP) {
    if (lane == 0) {
      bool ok = true;
      int kb = 0;
      const uint32_t wic_tx = INJ_MMA ? 0u : HC * 128u;
      for (; kb < nkb && ok; ++kb) {
        const int st = kb % NRY;
        if (kb >= NRY) ok = mbar_wait_bounded(ryfree(st), ((kb / NRY) - 1) & 1, p.err, p.limit_ns);
        if (!ok) break;
        const uint32_t sb = sbase + st * RY_BYTES;
        const int kx = (kb0 + kb) * BK;           // column within the stream
        mbar_arrive_expect_tx(ryfull(st), (p.has_y ? RY_BYTES : TILE_BYTES) + 128 + wic_tx);
        tma_load_2d(sb, &p.tm_R, s * HS + kx, m0, ryfull(st));
        if (p.has_y) tma_load_2d(sb + TILE_BYTES, &p.tm_y, kx, m0, ryfull(st));
        bulk_g2s(sbase + p.off_wn + st * 128, p.Wnorm + s * p.ld_wnorm + kx, 128,
                 ryfull(st));
        if constexpr (!INJ_MMA)
          tma_load_2d(sbase + p.off_wic + st * HC * 128, &p.tm_wi, s * HS + kx, 0, ryfull(st));
      }
      // outstanding copies land before the CTA can leave
      for (int j = max(0, kb - NRY); j < kb; ++j)
        mbar_wait_bounded(ryfull(j % NRY), (j / NRY) & 1, p.err, p.limit_ns);
    }
  } else if (warp == K1_W_WARP) {
    if (lane == 0) {
      bool ok = true;
      int g = 0;
      const uint32_t bytes0 = p.n2 > 0 ? p.wrows0 * 128u
                                       : r * 128u + (INJ_MMA ? WI_ROWS * 128u : 0u);
      const uint32_t bytes1 = (r - p.wrows0) * 128u + (INJ_MMA ? WI_ROWS * 128u : 0u);
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int kx = s * HS + (kb0 + kb) * BK;
        for (int hh = 0; hh < nh; ++hh, ++g) {
          const int ws = g % NW;
          if (g >= NW) ok = mbar_wait_bounded(wfree(ws), ((g / NW) - 1) & 1, p.err, p.limit_ns);
          if (!ok) break;
          const uint32_t wb = sbase + p.off_w + ws * p.w_slot;
          if (hh == 0) {
            mbar_arrive_expect_tx(wfull(ws), bytes0);
            tma_load_2d(wb, &p.tm_w0, kx, 0, wfull(ws));
            if (p.n2 == 0) {
              if (r > p.wrows0) tma_load_2d(wb + p.wrows0 * 128, &p.tm_w1, kx, p.wrows0, wfull(ws));
              if constexpr (INJ_MMA) tma_load_2d(wb + r * 128, &p.tm_wi, kx, 0, wfull(ws));
            }
          } else {
            mbar_arrive_expect_tx(wfull(ws), bytes1);
            tma_load_2d(wb, &p.tm_w1, kx, p.wrows0, wfull(ws));
            if constexpr (INJ_MMA)
              tma_load_2d(wb + (r - p.wrows0) * 128, &p.tm_wi, kx, 0, wfull(ws));
          }
        }
      }
      for (int j = max(0, g - NW); j < g; ++j)
        mbar_wait_bounded(wfull(j % NW), (j / NW) & 1, p.err, p.limit_ns);
    }
  } else if (warp == K1_MMA_WARP || warp == K1_MMA1_WARP) {
    // One warp per weight column block (two issuing threads keep the tensor
    // pipe fed; the blocks write disjoint accumulator columns).  The whole
    // warp walks the loop (every lane observes the barriers) and one elected
    // lane issues; the vote keeps the warp together if a wait expires.
    const int hh = warp == K1_MMA_WARP ? 0 : 1;
    if (hh < nh) {
      const uint32_t id = idesc_bf16(BM, hh ? p.n2 : p.n1);
      const uint32_t d = tmem + (hh ? p.n1 : 0);
      bool ok = true;
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int st = kb % NRY;
        const int g = kb * nh + hh, ws = g % NW;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(conv(st), (kb / NRY) & 1, p.err, p.limit_ns));
        ok = ok && __all_sync(0xffffffffu, mbar_wait_bounded(wfull(ws), (g / NW) & 1, p.err, p.limit_ns));
        if (!ok) break;
        tc_fence_after();
        const uint32_t ab = sbase + st * RY_BYTES;
        const uint64_t a_hi = desc_sw128(ab), a_lo = desc_sw128(ab + TILE_BYTES);
        const uint64_t bd = desc_sw128(sbase + p.off_w + ws * p.w_slot);
        if (elect_one()) {
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {
            umma_bf16(d, a_hi + 2u * ks, bd + 2u * ks, id, (kb | ks) != 0);
            if (!p.fold) umma_bf16(d, a_lo + 2u * ks, bd + 2u * ks, id, 1);
          }
          umma_commit(wfree(ws));
          umma_commit(ryfree(st));
        }
        __syncwarp();
      }
      // the accumulator is complete (or abandoned) once every issued MMA is
      if (elect_one()) umma_commit(accb);
      __syncwarp();
      mbar_wait_bounded(accb, 0, p.err, p.limit_ns);
    }
  } else if (warp < K1_CONV_WARPS) {
    // ---------------- converters: warps 0-7.  Thread (warp w, lane l) owns
    // channel chunk l & 7 (8 channels) of every K block and the four rows
    // 4w + (l >> 3) + 32 pp, pp < 4.  In the 128-byte swizzled tile chunk c of
    // row i sits at i * 128 + ((c ^ (i & 7)) << 4): the 8 lanes of a row read
    // 8 distinct chunk positions, so there are no bank conflicts; the Wnorm
    // factor (1 + w) of the chunk is formed once and reused for four rows.
    const int ch = lane & 7;
    const int rbase = warp * 4 + (lane >> 3);
    float iw[4], ss[4];
    bool valid[4];
    float ij[4][HC];
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const int m = m0 + rbase + 32 * pp;
      valid[pp] = m < p.M;
      iw[pp] = valid[pp] && p.has_y ? combine_weight(p.inj[m * p.ld_inj + s], 1.0f / static_cast<float>(HC))
                                    : 0.f;
      ss[pp] = 0.f;
#pragma unroll
      for (int j = 0; j < HC; ++j) ij[pp][j] = 0.f;
    }
    // The K-block loop in four copies -- with COMBINE (y injected) or without
    // (mix only: R is R2), for a folded weight (the operand is R2 itself) or
    // an unfolded one (the hi/lo split of R2 * (1 + Wnorm)) -- so that
    // call-uniform choices stay out of the per-element code.  Element pairs
    // go through the paired fp32 instructions (FFMA2 / FMUL2); each lane is
    // an ordinary round-to-nearest fma or multiply, so R2 is the same as
    // with scalar fmaf.
    float2 ss2[4];
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) ss2[pp] = make_float2(0.f, 0.f);
    auto convert = [&](auto has_y_c, auto fold_c) -> bool {
    constexpr bool HY = decltype(has_y_c)::value;
    constexpr bool FOLD = decltype(fold_c)::value;
    for (int kb = 0; kb < nkb; ++kb) {
      const int st = kb % NRY;
      if (!mbar_wait_bounded(ryfull(st), (kb / NRY) & 1, p.err, p.limit_ns)) return false;
      unsigned char* sb = smem + st * RY_BYTES;
      const int col = (kb0 + kb) * BK + ch * 8;   // channel within the stream
      float2 f2[4];
      if constexpr (!FOLD) {
        const uint4 wn = *reinterpret_cast<const uint4*>(smem + p.off_wn + st * 128 + ch * 16);
        const uint32_t ww[4] = {wn.x, wn.y, wn.z, wn.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          f2[e] = __fadd2_rn(make_float2(lo_bf16(ww[e]), hi_bf16(ww[e])), make_float2(1.f, 1.f));
      }
      [[maybe_unused]] float wi[INJ_MMA ? 1 : HC][8];
      if constexpr (!INJ_MMA) {
#pragma unroll
        for (int j = 0; j < HC; ++j)
          unpack8(*reinterpret_cast<const uint4*>(smem + p.off_wic + (st * HC + j) * 128 + ch * 16), wi[j]);
      }
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const int row = rbase + 32 * pp;
        const uint32_t off = row * 128 + ((ch ^ (row & 7)) << 4);
        const uint4 rraw = *reinterpret_cast<const uint4*>(sb + off);
        const uint32_t rw[4] = {rraw.x, rraw.y, rraw.z, rraw.w};
        uint32_t pr[4], ph[4], pl[4];
        [[maybe_unused]] float a[8];
        if constexpr (HY) {
          const uint4 yraw = *reinterpret_cast<const uint4*>(sb + TILE_BYTES + off);
          const uint32_t yw[4] = {yraw.x, yraw.y, yraw.z, yraw.w};
          const float2 iw2 = make_float2(iw[pp], iw[pp]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 v = __ffma2_rn(make_float2(lo_bf16(yw[e]), hi_bf16(yw[e])), iw2,
                                        make_float2(lo_bf16(rw[e]), hi_bf16(rw[e])));
            pr[e] = pack2(v.x, v.y);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) pr[e] = rw[e];
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 r2 = make_float2(lo_bf16(pr[e]), hi_bf16(pr[e]));
          ss2[pp] = __ffma2_rn(r2, r2, ss2[pp]);
          if constexpr (FOLD) {
            a[2 * e] = r2.x;
            a[2 * e + 1] = r2.y;
          } else {
            const float2 av = __fmul2_rn(r2, f2[e]);
            ph[e] = pack2(av.x, av.y);
            // a - bf16(a) is exact in fp32, so the fma with -1 is exact too
            const float2 lo = __ffma2_rn(make_float2(lo_bf16(ph[e]), hi_bf16(ph[e])),
                                         make_float2(-1.f, -1.f), av);
            pl[e] = pack2(lo.x, lo.y);
            a[2 * e] = av.x;
            a[2 * e + 1] = av.y;
          }
        }
        if (HY && valid[pp])
          *reinterpret_cast<uint4*>(p.R2 + static_cast<int64_t>(m0 + row) * p.K +
                                    static_cast<int64_t>(s) * HS + col) =
              make_uint4(pr[0], pr[1], pr[2], pr[3]);
        if constexpr (FOLD) {
          *reinterpret_cast<uint4*>(sb + off) = make_uint4(pr[0], pr[1], pr[2], pr[3]);
        } else {
          *reinterpret_cast<uint4*>(sb + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
          *reinterpret_cast<uint4*>(sb + TILE_BYTES + off) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
        }
        if constexpr (!INJ_MMA) {
#pragma unroll
          for (int j = 0; j < HC; ++j) {
            float t = ij[pp][j];
#pragma unroll
            for (int e = 0; e < 8; ++e) t = fmaf(a[e], wi[j][e], t);
            ij[pp][j] = t;
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(conv(st));
    }
    return true;
    };
    using T_ = std::true_type;
    using F_ = std::false_type;
    bool ok = p.has_y ? (p.fold ? convert(T_{}, T_{}) : convert(T_{}, F_{}))
                      : (p.fold ? convert(F_{}, T_{}) : convert(F_{}, F_{}));
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) ss[pp] = ss2[pp].x + ss2[pp].y;
    // per-row totals: the 8 lanes of a row hold its 8 channel chunks
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        ss[pp] += __shfl_xor_sync(0xffffffffu, ss[pp], o);
        if constexpr (!INJ_MMA) {
#pragma unroll
          for (int j = 0; j < HC; ++j) ij[pp][j] += __shfl_xor_sync(0xffffffffu, ij[pp][j], o);
        }
      }
      if (ch == 0) {
        const int row = rbase + 32 * pp;
        rowss[row] = ss[pp];
        if constexpr (!INJ_MMA) {
#pragma unroll
          for (int j = 0; j < HC; ++j) rowinj[row * HC + j] = ij[pp][j];
        }
      }
    }
    named_bar_sync(1, K1_CONV_WARPS * 32);
    // ---------------- epilogue: partial sums of squares and the un-scaled
    // partial products (lora columns, then the inject columns); the reduce
    // kernel applies rrms once all K chunks of the stream are in.
    if (ok) ok = mbar_wait_bounded(accb, 0, p.err, p.limit_ns);
    tc_fence_after();
    const int q = warp & 3, half = warp >> 2;
    const int erow = 32 * q + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);
    // column-major within the tile: consecutive threads (rows) write
    // consecutive words, one 128-byte line per warp and column
    const int64_t tp = static_cast<int64_t>(m0 / BM) * (HC * p.S) + pid;
    float* dst = p.part + tp * p.np * BM + erow;
    if (ok && half == 0) {
      float injv[HC];
      if constexpr (INJ_MMA) {
        uint32_t acc[16];
        tmem_ld16_wait(tl + r, acc);
#pragma unroll
        for (int j = 0; j < HC; ++j) injv[j] = __uint_as_float(acc[j]);
      } else {
#pragma unroll
        for (int j = 0; j < HC; ++j) injv[j] = rowinj[erow * HC + j];
      }
      p.sumsq[tp * BM + erow] = rowss[erow];
#pragma unroll
      for (int j = 0; j < HC; ++j) dst[(r + j) * BM] = injv[j];
    }
    if (ok) {
      const int cols = r / 2;
      for (int c0 = 0; c0 < cols; c0 += 16) {
        uint32_t acc[16];
        tmem_ld16_wait(tl + half * cols + c0, acc);
#pragma unroll
        for (int e = 0; e < 16; ++e) dst[(half * cols + c0 + e) * BM] = __uint_as_float(acc[e]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // every store of this CTA is issued: the reduce may launch (it waits for
  // this grid's completion before it reads anything)
  grid_dep_launch();
  if (warp == K1_MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

// ================================================================ reduce
// Per token row: rrms_s from the stream's partial sums of squares, then
// lora / inj_next = sum_s rrms_s * (sum over the stream's K chunks of the
// partial products), and the up-GEMM operand hh = bf16(SiLU(lora / HC) / 2):
// the halving is exact and makes K2's accumulator hold G / 2, the argument of
// tanh in sigmoid(G) = (1 + tanh(G / 2)) / 2.  The grid also writes
// w1 = 1 + Wnorm in fp32 for K2's epilogue.  A block takes a 128-row tile
// x RED_COLS columns: it reads the column-major partials in float4s, 512
// contiguous bytes per warp, column and stream, and transposes through shared
// memory to write the row-major outputs in 32-byte row runs.  Eight columns
// a block keep a thread at one column (at HC <= 4 under 64 registers with one
// K chunk per batch: four blocks an SM), so more loads are in flight per SM
// than with 16.
constexpr int RED_THREADS = 256;
constexpr int RED_COLS = 8;           // columns per block (a block covers a whole 128-row tile)

template <int HC, int CB>
__global__ void __launch_bounds__(RED_THREADS, CB > 1 || HC > 4 ? 2 : 4)
    k1_reduce_kernel(const float* __restrict__ part, const float* __restrict__ sumsq,
                     float* __restrict__ rrms, float* __restrict__ lora,
                     float* __restrict__ inj_next, bf16_t* __restrict__ hh,
                     const bf16_t* __restrict__ Wnorm, int ld_wnorm, float* __restrict__ w1,
                     int M, int S, int r, int np, int HS, float inv_hs, float eps) {
  __shared__ float s_acc[RED_COLS][BM + 1];
  const int tid = threadIdx.x;
  // As K1's programmatic dependent this grid may start before K1 has
  // finished: K1's partials are read only after the wait, and through L2.
  grid_dep_wait();
  const int bid = blockIdx.y * gridDim.x + blockIdx.x;
  const int K = HC * HS;
  for (int k = bid * RED_THREADS + tid; k < K; k += gridDim.x * gridDim.y * RED_THREADS)
    w1[k] = 1.0f + bf16_to_f32(Wnorm[(k / HS) * ld_wnorm + k % HS]);
  const int tile = blockIdx.y, n0 = blockIdx.x * RED_COLS;
  // thread = (4 consecutive rows, RED_COLS / 8 columns): rows 4 (tid % 32) ..,
  // columns n0 + tid / 32 + 8 j; a warp reads 512 contiguous bytes per column
  // and stream
  const int r4 = (tid & 31) * 4, cw = tid >> 5;
  constexpr int NCOL = RED_COLS / 8;
  const int ns = HC * S;
  const int64_t tb = static_cast<int64_t>(tile) * ns;
  float4 rs[HC];
  float4 pv[NCOL][HC];
  if (S == 1) {
    // one K chunk per stream (the usual case): every load issues before any
    // is used
    float4 q[HC];
#pragma unroll
    for (int ss = 0; ss < HC; ++ss)
      q[ss] = __ldcg(reinterpret_cast<const float4*>(sumsq + (tb + ss) * BM + r4));
#pragma unroll
    for (int j = 0; j < NCOL; ++j) {
      const int n = min(n0 + cw + 8 * j, np - 1);
#pragma unroll
      for (int ss = 0; ss < HC; ++ss)
        pv[j][ss] = __ldcg(reinterpret_cast<const float4*>(part + ((tb + ss) * np + n) * BM + r4));
    }
#pragma unroll
    for (int ss = 0; ss < HC; ++ss)
      rs[ss] = make_float4(rsqrt_nr(fmaf(q[ss].x, inv_hs, eps)), rsqrt_nr(fmaf(q[ss].y, inv_hs, eps)),
                           rsqrt_nr(fmaf(q[ss].z, inv_hs, eps)), rsqrt_nr(fmaf(q[ss].w, inv_hs, eps)));
  } else {
    // K chunks: the chunks' loads issue CB at a time (their sums are still
    // added in chunk order).  Warp w < HC also sums stream w's partial sums
    // of squares for its lanes' rows and shares the stream's rrms through
    // shared memory, so a thread's batch holds its column's products and at
    // most one stream's squares instead of every stream's: fewer dependent
    // batches for the same registers.  CB > 1 halves the resident blocks, so
    // the host picks it only when the grid fits one wave either way.
    __shared__ float4 s_rs[HC][32];
    float4 qw = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < NCOL; ++j)
#pragma unroll
      for (int ss = 0; ss < HC; ++ss) pv[j][ss] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int c0 = 0; c0 < S; c0 += CB) {
      float4 qc[CB], vc[CB][NCOL][HC];
#pragma unroll
      for (int u = 0; u < CB; ++u) {
        const int c = min(c0 + u, S - 1);
        qc[u] = cw < HC ? __ldcg(reinterpret_cast<const float4*>(sumsq + (tb + cw * S + c) * BM + r4))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < NCOL; ++j) {
          const int n = min(n0 + cw + 8 * j, np - 1);
#pragma unroll
          for (int ss = 0; ss < HC; ++ss)
            vc[u][j][ss] = __ldcg(reinterpret_cast<const float4*>(part + ((tb + ss * S + c) * np + n) * BM + r4));
        }
      }
#pragma unroll
      for (int u = 0; u < CB; ++u) {
        if (c0 + u < S) {
          qw.x += qc[u].x; qw.y += qc[u].y; qw.z += qc[u].z; qw.w += qc[u].w;
#pragma unroll
          for (int j = 0; j < NCOL; ++j)
#pragma unroll
            for (int ss = 0; ss < HC; ++ss) {
              pv[j][ss].x += vc[u][j][ss].x; pv[j][ss].y += vc[u][j][ss].y;
              pv[j][ss].z += vc[u][j][ss].z; pv[j][ss].w += vc[u][j][ss].w;
            }
        }
      }
    }
    if (cw < HC)
      s_rs[cw][tid & 31] = make_float4(rsqrt_nr(fmaf(qw.x, inv_hs, eps)), rsqrt_nr(fmaf(qw.y, inv_hs, eps)),
                                       rsqrt_nr(fmaf(qw.z, inv_hs, eps)), rsqrt_nr(fmaf(qw.w, inv_hs, eps)));
    __syncthreads();
#pragma unroll
    for (int ss = 0; ss < HC; ++ss) rs[ss] = s_rs[ss][tid & 31];
  }
  if (blockIdx.x == 0 && cw == 0) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int m = tile * BM + r4 + e;
      if (m < M) {
#pragma unroll
        for (int ss = 0; ss < HC; ++ss)
          rrms[static_cast<int64_t>(m) * HC + ss] = e == 0 ? rs[ss].x : e == 1 ? rs[ss].y : e == 2 ? rs[ss].z : rs[ss].w;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < NCOL; ++j) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int ss = 0; ss < HC; ++ss) {
      acc.x = fmaf(rs[ss].x, pv[j][ss].x, acc.x); acc.y = fmaf(rs[ss].y, pv[j][ss].y, acc.y);
      acc.z = fmaf(rs[ss].z, pv[j][ss].z, acc.z); acc.w = fmaf(rs[ss].w, pv[j][ss].w, acc.w);
    }
    float* dstc = &s_acc[cw + 8 * j][r4];
    dstc[0] = acc.x; dstc[1] = acc.y; dstc[2] = acc.z; dstc[3] = acc.w;
  }
  __syncthreads();
  // rows out: RED_COLS consecutive columns of a row per RED_COLS lanes
  const float inv_hc = 1.0f / static_cast<float>(HC);
  const int cn = tid & (RED_COLS - 1), n = n0 + cn;
#pragma unroll
  for (int j = 0; j < BM * RED_COLS / RED_THREADS; ++j) {
    const int rw = tid / RED_COLS + (RED_THREADS / RED_COLS) * j;
    const int m = tile * BM + rw;
    if (m >= M || n >= np) continue;
    const float v = s_acc[cn][rw];
    if (n < r) {
      lora[static_cast<int64_t>(m) * r + n] = v;
      const float u = v * inv_hc;
      hh[static_cast<int64_t>(m) * r + n] = f32_to_bf16(0.5f * (u * sigmoid_fast(u)));
    } else if (n - r < HC) {
      inj_next[static_cast<int64_t>(m) * HC + (n - r)] = v;
    }
  }
  // every store of this block is issued: K2 may launch (it waits for this
  // grid's completion before it reads anything)
  grid_dep_launch();
}

// ===================================================================== K2
// Unit = (128-token tile t, NCU-channel block cb); the MMA N dimension holds
// the HC streams of those channels (N = HC * NCU rows of Wu, at most 256, so
// that one tcgen05.mma does 128 tensor cycles of work per issue).  Roles:
//   warp 0  TMA: per K block, the hh tile (128 x 64) and the HC x NCU rows of
//           Wu (one 3-D box over Wu viewed as [HC][HS][r]) into a stage ring;
//   warp 1  tcgen05.mma into a double-buffered accumulator; the whole warp
//           walks the loop and one elected lane issues;
//   warp 2  tensor-memory allocation;
//   warp 3  TMA: the unit's R2 tile one stream at a time (128 x NCU box) and
//           that stream's slice of 1 + Wnorm (fp32), into a ring of stream
//           slots;
//   warps 4-11  epilogue: thread = (token row, half of the NCU channels); it
//           reads the row's gates stream by stream from tensor memory,
//           rebuilds xn from R2, rrms and Wnorm and stores its x channels.
constexpr int K2_THREADS = 384;
constexpr int K2_TMA_WARP = 0;
constexpr int K2_MMA_WARP = 1;
constexpr int K2_ALLOC_WARP = 2;
constexpr int K2_R2_WARP = 3;
constexpr int K2_EPI_WARP0 = 4;
constexpr int K2_EPI_WARPS = 8;
constexpr int K2_MAX_ST = 8;     // stage ring slots
constexpr int K2_MAX_R2 = 16;    // R2 stream slots
constexpr uint32_t K2_BAR_BYTES = 512;

// Channels per unit: 64 up to HC = 4, 32 above (MMA N = HC * NCU <= 256).
// At HC = 4 the host halves the block (N = 128) when even the halved units
// fit one round over the SMs (one 128-token tile).
__host__ __device__ constexpr int k2_ncu(int hc) { return hc <= 4 ? 64 : 32; }
__host__ __device__ constexpr uint32_t k2_tmem_cols(int hc, int ncu) {
  return 2 * hc * ncu <= 128 ? 128u : (2 * hc * ncu <= 256 ? 256u : 512u);
}

struct K2Params {
  CUtensorMap tm_h;    // hh [M][r], box {64, 128}, 128B swizzle
  CUtensorMap tm_wu;   // Wu as [HC][HS][r], box {64, NCU, HC}, 128B swizzle
  CUtensorMap tm_r2;   // R2 [M][K], box {NCU, 128}, (NCU * 2)-byte swizzle
  CUtensorMap tm_w1;   // 1 + Wnorm (fp32) as [HC][HS], box {NCU, 1}
  const float* rrms;
  bf16_t* x;
  int M, HS, r;
  int nkb, ncb, n_units, nst, nr2;
  uint32_t stage_bytes;
  uint32_t off_r2, off_w1, off_bar;
  int* err;
  uint64_t limit_ns;
};

// Byte offset of 16-byte chunk `chunk` of row `row` in a box whose rows are
// ROWB bytes and that TMA wrote with the ROWB-byte swizzle (the chunk index
// is XORed with address bits 7.. of the row start).
template <int ROWB>
__device__ __forceinline__ uint32_t swz_off(int row, int chunk) {
  if constexpr (ROWB == 128) return row * 128 + ((chunk ^ (row & 7)) << 4);
  else if constexpr (ROWB == 64) return row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4);
  else return row * 32 + ((chunk ^ ((row >> 2) & 1)) << 4);
}

template <int HCT, int NCUT>
__global__ void __launch_bounds__(K2_THREADS, 1) k2_kernel(const __grid_constant__ K2Params p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int HC = HCT;
  constexpr int NCU = NCUT;
  constexpr int N = HC * NCU;
  constexpr uint32_t BOXB = BM * NCU * 2;        // one stream's R2 box
  constexpr uint32_t TMEM_COLS = k2_tmem_cols(HCT, NCUT);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int HS = p.HS, nkb = p.nkb, nst = p.nst, nr2 = p.nr2;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar = sbase + p.off_bar;
  auto full = [&](int st) { return bar + 8u * st; };
  auto freeb = [&](int st) { return bar + 64u + 8u * st; };
  auto accfull = [&](int a) { return bar + 128u + 8u * a; };
  auto accfree = [&](int a) { return bar + 144u + 8u * a; };
  auto r2full = [&](int q) { return bar + 160u + 8u * q; };
  auto r2free = [&](int q) { return bar + 288u + 8u * q; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.off_bar + 416);

  const int u0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * p.n_units / gridDim.x);
  const int u1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * p.n_units / gridDim.x);
  const int n_local = u1 - u0;

  if (tid == 0) {
    prefetch_tmap(&p.tm_h);
    prefetch_tmap(&p.tm_wu);
    prefetch_tmap(&p.tm_r2);
    prefetch_tmap(&p.tm_w1);
    for (int i = 0; i < nst; ++i) {
      mbar_init(full(i), 1);
      mbar_init(freeb(i), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accfull(a), 1);
      mbar_init(accfree(a), K2_EPI_WARPS);
    }
    for (int q = 0; q < nr2; ++q) {
      mbar_init(r2full(q), 1);
      mbar_init(r2free(q), K2_EPI_WARPS);
    }
    fence_mbar_init();
  }
  if (warp == K2_ALLOC_WARP) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // hh, rrms, 1 + Wnorm (the reduce) and R2 (K1): as the reduce's
  // programmatic dependent this prologue may overlap the reduce's tail, so
  // they are read only after the wait -- by TMA, after the proxy fence, or
  // through L2 (rrms).
  grid_dep_wait();
  fence_proxy_async_global();

  if (warp == K2_TMA_WARP) {
    if (lane == 0) {
      bool ok = true;
      int g = 0;
      for (int i = 0; i < n_local && ok; ++i) {
        const int u = u0 + i, t = u / p.ncb, cb = u % p.ncb;
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int st = g % nst;
          if (g >= nst) ok = mbar_wait_bounded(freeb(st), ((g / nst) - 1) & 1, p.err, p.limit_ns);
          if (!ok) break;
          const uint32_t sb = sbase + st * p.stage_bytes;
          mbar_arrive_expect_tx(full(st), p.stage_bytes);
          tma_load_2d(sb, &p.tm_h, kb * BK, t * BM, full(st));
          tma_load_3d(sb + TILE_BYTES, &p.tm_wu, kb * BK, cb * NCU, 0, full(st));
        }
      }
      // the copies still in flight land before the CTA can leave
      for (int j = max(0, g - nst); j < g; ++j)
        mbar_wait_bounded(full(j % nst), (j / nst) & 1, p.err, p.limit_ns);
    }
  } else if (warp == K2_R2_WARP) {
    if (lane == 0) {
      bool ok = true;
      int n = 0;
      for (int i = 0; i < n_local && ok; ++i) {
        const int u = u0 + i, t = u / p.ncb, cb = u % p.ncb;
        for (int ss = 0; ss < HC; ++ss, ++n) {
          const int q = n % nr2;
          if (n >= nr2) ok = mbar_wait_bounded(r2free(q), ((n / nr2) - 1) & 1, p.err, p.limit_ns);
          if (!ok) break;
          mbar_arrive_expect_tx(r2full(q), BOXB + NCU * 4);
          tma_load_2d(sbase + p.off_r2 + q * BOXB, &p.tm_r2, ss * HS + cb * NCU, t * BM, r2full(q));
          tma_load_2d(sbase + p.off_w1 + q * 256u, &p.tm_w1, cb * NCU, ss, r2full(q));
        }
      }
      for (int j = max(0, n - nr2); j < n; ++j)
        mbar_wait_bounded(r2full(j % nr2), (j / nr2) & 1, p.err, p.limit_ns);
    }
  } else if (warp == K2_MMA_WARP) {
    // Every lane waits on the barriers (so the electing lane has observed
    // them); the vote keeps the warp on one path if a wait expires.
    constexpr uint32_t idesc = idesc_bf16(BM, N);
    bool ok = true;
    int g = 0, issued = 0;
    for (int i = 0; i < n_local && ok; ++i) {
      const int ab = i & 1;
      if (i >= 2)
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(accfree(ab), ((i >> 1) - 1) & 1, p.err, p.limit_ns));
      if (!ok) break;
      tc_fence_after();
      const uint32_t dcol = tmem + ab * N;
      for (int kb = 0; kb < nkb; ++kb, ++g) {
        const int st = g % nst;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(full(st), (g / nst) & 1, p.err, p.limit_ns));
        if (!ok) break;
        tc_fence_after();
        const uint32_t sb = sbase + st * p.stage_bytes;
        const uint64_t ad = desc_sw128(sb), bd = desc_sw128(sb + TILE_BYTES);
        if (elect_one()) {
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks)
            umma_bf16(dcol, ad + 2u * ks, bd + 2u * ks, idesc, (kb | ks) != 0);
          umma_commit(freeb(st));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (elect_one()) umma_commit(accfull(ab));
      __syncwarp();
      ++issued;
    }
    if (issued > 0)
      mbar_wait_bounded(accfull((issued - 1) & 1), ((issued - 1) >> 1) & 1, p.err, p.limit_ns);
  } else if (warp >= K2_EPI_WARP0) {
    constexpr int CPT = NCU / 2;          // channels per thread
    constexpr int V = CPT / 8;            // 16-byte chunks per thread and stream
    const int ew = warp - K2_EPI_WARP0;
    const int q4 = warp & 3, half = ew >> 2;
    const int row = 32 * q4 + lane;
    const float inv_hc = 1.0f / static_cast<float>(HC);
    int n = 0;
    for (int i = 0; i < n_local; ++i, n += HC) {
      const int u = u0 + i, t = u / p.ncb, cb = u % p.ncb;
      const int ab = i & 1;
      const int64_t m = static_cast<int64_t>(t) * BM + row;
      const bool v = m < p.M;
      float rr[HC];
#pragma unroll
      for (int ss = 0; ss < HC; ++ss) rr[ss] = v ? __ldcg(p.rrms + m * HC + ss) : 0.f;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(accfull(ab), (i >> 1) & 1, p.err, p.limit_ns)))
        break;
      tc_fence_after();
      const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q4) << 16) + ab * N + half * CPT;
      float2 acc[CPT / 2];
#pragma unroll
      for (int e = 0; e < CPT / 2; ++e) acc[e] = make_float2(0.f, 0.f);
      uint32_t gv[CPT];
      bool ok = true;
#pragma unroll
      for (int ss = 0; ss < HC; ++ss) {
        const int q = (n + ss) % nr2;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(r2full(q), ((n + ss) / nr2) & 1, p.err, p.limit_ns));
        if (!ok) break;
        if constexpr (CPT == 32) tmem_ld32_wait(tbase + ss * NCU, gv);
        else tmem_ld16_wait(tbase + ss * NCU, gv);
        const unsigned char* rb = smem + p.off_r2 + q * BOXB;
        const float* wb = reinterpret_cast<const float*>(smem + p.off_w1 + q * 256u) + half * CPT;
        const float2 rr2 = make_float2(rr[ss], rr[ss]);
#pragma unroll
        for (int j = 0; j < V; ++j) {
          const uint4 rv = *reinterpret_cast<const uint4*>(rb + swz_off<NCU * 2>(row, half * V + j));
          const float4 wa = *reinterpret_cast<const float4*>(wb + 8 * j);
          const float4 wc = *reinterpret_cast<const float4*>(wb + 8 * j + 4);
          const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
          const float2 w[4] = {make_float2(wa.x, wa.y), make_float2(wa.z, wa.w),
                               make_float2(wc.x, wc.y), make_float2(wc.z, wc.w)};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            // xn = R2 * rrms * (1 + Wnorm); sigmoid(G) = 1/2 + tanh(G / 2) / 2
            const float2 xn = __fmul2_rn(__fmul2_rn(make_float2(lo_bf16(rw[e]), hi_bf16(rw[e])), rr2), w[e]);
            const float2 th = make_float2(tanh_approx(__uint_as_float(gv[8 * j + 2 * e])),
                                          tanh_approx(__uint_as_float(gv[8 * j + 2 * e + 1])));
            const float2 sg = __ffma2_rn(th, make_float2(0.5f, 0.5f), make_float2(0.5f, 0.5f));
            acc[4 * j + e] = __ffma2_rn(sg, xn, acc[4 * j + e]);
          }
        }
        // The slot is read with ordinary loads (the generic proxy) and the
        // next TMA write into it goes through the async proxy: this
        // write-after-read across proxies needs the proxy fence before the
        // slot is released, or the TMA refill can overtake the reads (seen
        // as occasional wrong x for one warp of one unit).
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(r2free(q));
      }
      if (!ok) break;
      // every tensor-memory load of this accumulator has completed
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(accfree(ab));
      if (v) {
        uint4* dst = reinterpret_cast<uint4*>(p.x + m * HS + cb * NCU + half * CPT);
#pragma unroll
        for (int j = 0; j < V; ++j) {
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) o[e] = pack2(acc[4 * j + e].x * inv_hc, acc[4 * j + e].y * inv_hc);
          dst[j] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == K2_ALLOC_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

uint32_t pow2_cols(int n) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(n)) c <<= 1;
  return c;
}

// A launch of `kernel` on `stream`, as a programmatic dependent of the
// previous kernel in the stream when pdl is set (its prologue may then overlap
// that kernel; it waits for it with griddepcontrol.wait before touching
// memory the previous kernel may have written).
template <typename... KArgs, typename... Args>
cudaError_t launch_maybe_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <int HCT, bool INJ_MMA>
cudaError_t launch_k1(const K1Params& p, int grid, size_t smem, const Device& dev,
                      cudaStream_t stream, bool pdl) {
  static std::atomic<unsigned long long> attr{0};
  cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(k1_kernel<HCT, INJ_MMA>),
                                  dev.smem_optin, dev.id, attr);
  if (e != cudaSuccess) return e;
  return launch_maybe_pdl(k1_kernel<HCT, INJ_MMA>, dim3(grid), dim3(K1_THREADS), smem, stream, pdl, p);
}

template <int HCT, int NCUT = k2_ncu(HCT)>
cudaError_t launch_k2(const K2Params& p, int grid, size_t smem, const Device& dev,
                      cudaStream_t stream, bool pdl) {
  static std::atomic<unsigned long long> attr{0};
  cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(k2_kernel<HCT, NCUT>),
                                  dev.smem_optin, dev.id, attr);
  if (e != cudaSuccess) return e;
  return launch_maybe_pdl(k2_kernel<HCT, NCUT>, dim3(grid), dim3(K2_THREADS), smem, stream, pdl, p);
}

bool prefill_supported(const Call& c) {
  return c.HS % 64 == 0 && c.r % 64 == 0 && c.r <= 512 && c.HC >= 1 && c.HC <= 8;
}
static_assert(k2_ncu(4) * 4 == 256 && k2_ncu(8) * 8 == 256 && k2_ncu(1) * 8 <= 512,
              "K2 MMA N = 256 for HC = 4 and 8; 2N tensor-memory columns fit");

// K2's channel block at HC = 4: 32 instead of 64 when the halved units still
// fit one round over the SMs, so that the same work spreads over twice the
// CTAs.  Measured on the GB300 at HS = 2560: 1.1 us less at M = 128 (40 or
// 80 units); where halving adds rounds it costs more than it saves (+0.5 us
// at M = 512, +5 at 2048, +12 at 4096: a unit's cost is far from
// proportional to its channels).
int k2_block(int HC, int n_mt, int HS, int sms) {
  const int ncu = k2_ncu(HC);
  if (HC != 4 || HS % 32 != 0) return ncu;
  return static_cast<int64_t>(n_mt) * (HS / 32) <= sms ? 32 : ncu;
}


// K chunks per stream: enough (tile, stream, chunk) CTAs to cover the SMs
// when there are few token tiles, at least two K blocks per chunk.
int k1_chunks(int n_mt, int HC, int nkb, int sms) {
  if (HC * n_mt >= sms) return 1;
  // as many chunks as still fit one wave (a second, nearly empty wave costs
  // a whole CTA time)
  const int want = sms / (HC * n_mt);
  return std::max(1, std::min(want, nkb / 2));
}

int k1_np(int r, int HC) { return (r + HC + 3) / 4 * 4; }

}  // namespace

size_t prefill_ws_bytes(int64_t max_M, int HC, int HS, int r) {
  // the largest partial buffer over M <= max_M: split-K only for small M,
  // where HC * S * M stays below a few hundred tiles of rows
  // rows padded to whole 128-token tiles
  const size_t Mp = static_cast<size_t>((max_M + BM - 1) / BM) * BM;
  size_t part = static_cast<size_t>(HC) * Mp * k1_np(r, HC);
  part = std::max(part, static_cast<size_t>(2 * MAX_GRID) * BM * k1_np(r, HC));
  const size_t sumsq = std::max(static_cast<size_t>(HC) * Mp, static_cast<size_t>(2 * MAX_GRID) * BM);
  const size_t h = static_cast<size_t>(max_M) * r * 2;
  const size_t w1 = static_cast<size_t>(HC) * HS;
  return part * 4 + 256 + sumsq * 4 + 256 + h + 256 + w1 * 4 + 256;
}

cudaError_t launch_prefill(const Call& c, const Workspace& ws, const Device& dev,
                           cudaStream_t stream) {
  if (!prefill_supported(c)) return cudaErrorNotSupported;
  // hc_gr_args.pdl: K1 as a programmatic dependent of the previous kernel in
  // the stream.  The reduce (of K1) and K2 (of the reduce) are always
  // programmatic dependents: their predecessors are this call's own kernels,
  // and each waits for its predecessor's end before it touches memory, so
  // their prologues and launches overlap the predecessor's tail in either mode.
  const bool pdl = c.pdl != 0;
  if (prefill_ws_bytes(c.M, c.HC, c.HS, c.r) > ws.prefill_bytes) return cudaErrorNotSupported;
  const int M = static_cast<int>(c.M);
  const int n_mt = (M + BM - 1) / BM;
  const int nkb = c.HS / BK;
  const int S = k1_chunks(n_mt, c.HC, nkb, dev.sms);
  const int np = k1_np(c.r, c.HC);
  const size_t Mp = static_cast<size_t>(n_mt) * BM;
  const size_t part_floats = static_cast<size_t>(c.HC) * S * Mp * np;
  if (part_floats > std::max(static_cast<size_t>(c.HC) * Mp * np,
                             static_cast<size_t>(2 * MAX_GRID) * BM * np))
    return cudaErrorNotSupported;
  // workspace carve-up (sized by prefill_ws_bytes for max_M)
  float* part = ws.k1_part;
  float* sumsq = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(part) +
                                          (part_floats * 4 + 255) / 256 * 256);
  const size_t sumsq_floats = static_cast<size_t>(c.HC) * S * Mp;
  bf16_t* h = reinterpret_cast<bf16_t*>(reinterpret_cast<unsigned char*>(sumsq) +
                                        (sumsq_floats * 4 + 255) / 256 * 256);
  float* w1 = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(h) +
                                       (static_cast<size_t>(M) * c.r * 2 + 255) / 256 * 256);

  // ---------------- K1
  {
    K1Params p;
    const bool inj_mma = c.r + WI_ROWS <= 512;
    const uint64_t dR[2] = {static_cast<uint64_t>(c.K), static_cast<uint64_t>(M)};
    const uint64_t sR[1] = {static_cast<uint64_t>(c.K) * 2};
    const uint32_t bT[2] = {BK, BM};
    if (!make_tmap_bf16(&p.tm_R, c.R, 2, dR, sR, bT, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    const uint64_t dy[2] = {static_cast<uint64_t>(c.HS), static_cast<uint64_t>(M)};
    const uint64_t sy[1] = {static_cast<uint64_t>(c.HS) * 2};
    if (c.y) {
      if (!make_tmap_bf16(&p.tm_y, c.y, 2, dy, sy, bT, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    } else {
      std::memset(&p.tm_y, 0, sizeof(p.tm_y));
    }
    p.has_y = c.y != nullptr;
    // MMA column blocks over the B tile (r rows of Wd, then 16 inject rows
    // when the inject products run on the tensor cores)
    const int ntot = c.r + (inj_mma ? WI_ROWS : 0);
    if (ntot <= 256) {
      p.n1 = ntot;
      p.n2 = 0;
      p.wrows0 = c.r;
    } else {
      p.n1 = ((ntot / 2) + 15) / 16 * 16;
      p.n2 = ntot - p.n1;
      p.wrows0 = p.n1;
    }
    const uint64_t dw[2] = {static_cast<uint64_t>(c.K), static_cast<uint64_t>(c.r)};
    const uint32_t bw0[2] = {BK, static_cast<uint32_t>(p.wrows0)};
    const uint32_t bw1[2] = {BK, static_cast<uint32_t>(p.n2 > 0 ? c.r - p.wrows0 : 16)};
    if (!make_tmap_bf16(&p.tm_w0, c.Wd, 2, dw, sR, bw0, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_bf16(&p.tm_w1, c.Wd, 2, dw, sR, bw1, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    const uint64_t di[2] = {static_cast<uint64_t>(c.K), static_cast<uint64_t>(c.HC)};
    const uint32_t bi[2] = {BK, static_cast<uint32_t>(inj_mma ? WI_ROWS : c.HC)};
    if (!make_tmap_bf16(&p.tm_wi, c.Wi, 2, di, sR, bi,
                        inj_mma ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    p.inj = c.inj;
    p.ld_inj = c.ld_inj;
    p.R2 = c.R2;
    p.Wnorm = c.Wnorm;
    p.ld_wnorm = c.ld_wnorm;
    p.part = part;
    p.sumsq = sumsq;
    p.M = M;
    p.HS = c.HS;
    p.K = c.K;
    p.r = c.r;
    p.np = np;
    p.fold = c.fold;
    p.S = S;
    p.nkb = nkb;
    // shared memory: [R/y ring | weight ring | Wnorm slices | Wi rows (CUDA-core
    // inject) | barriers | row sums of squares | row inject sums]; the deepest
    // rings that fit
    p.w_slot = static_cast<uint32_t>((std::max(p.n1, p.n2) * 128 + 1023) / 1024 * 1024);
    // The weight ring's slots take the column blocks in turn (box g in slot
    // g % nw, block g % nh), so nw is a multiple of nh: every slot then only
    // ever serves one MMA warp, which waits on its phases in order.  (With an
    // odd nw and two MMA warps a warp could wait on a slot's next phase
    // while the previous one was still incomplete; the parity wait then
    // reports the older phase as complete and the MMAs read a box that has
    // not landed.)
    const int depths[5][2] = {{4, 4}, {4, 3}, {3, 3}, {3, 2}, {2, 2}};
    const int nh = p.n2 > 0 ? 2 : 1;
    size_t smem = 0;
    for (const auto& dpt : depths) {
      if (dpt[1] % nh != 0) continue;
      p.nry = dpt[0];
      p.nw = dpt[1];
      p.off_w = static_cast<uint32_t>(p.nry) * RY_BYTES;
      p.off_wn = p.off_w + static_cast<uint32_t>(p.nw) * p.w_slot;
      p.off_wic = p.off_wn + static_cast<uint32_t>(p.nry) * 128u;
      p.off_bar = p.off_wic + (inj_mma ? 0u : static_cast<uint32_t>(p.nry * c.HC) * 128u);
      p.off_rowss = p.off_bar + K1_BAR_BYTES;
      p.off_rowinj = p.off_rowss + BM * 4;
      smem = p.off_rowinj + (inj_mma ? 0u : static_cast<uint32_t>(BM * c.HC) * 4u) + 1024;
      if (smem <= static_cast<size_t>(dev.smem_optin)) break;
    }
    if (smem > static_cast<size_t>(dev.smem_optin) || p.nry > K1_MAX_RY || p.nw > K1_MAX_W)
      return cudaErrorNotSupported;
    p.tmem_cols = pow2_cols(ntot);
    p.err = ws.err;
    p.limit_ns = 1000ull * 1000 * 1000;
    cudaError_t e = cudaSuccess;
    const int grid = n_mt * c.HC * S;
#define HCGR_K1(HCV)                                                                        \
  case HCV:                                                                                 \
    e = inj_mma ? launch_k1<HCV, true>(p, grid, smem, dev, stream, pdl)                     \
                : launch_k1<HCV, false>(p, grid, smem, dev, stream, pdl);                    \
    break;
    switch (c.HC) {
      HCGR_K1(1) HCGR_K1(2) HCGR_K1(3) HCGR_K1(4) HCGR_K1(5) HCGR_K1(6) HCGR_K1(7)
      default: e = inj_mma ? launch_k1<8, true>(p, grid, smem, dev, stream, pdl)
                           : launch_k1<8, false>(p, grid, smem, dev, stream, pdl);
    }
#undef HCGR_K1
    if (e != cudaSuccess) return e;
  }
  // ---------------- reduce
  {
    const dim3 grid((np + RED_COLS - 1) / RED_COLS, n_mt);
    const bool batched = S > 1 && static_cast<int64_t>(grid.x) * grid.y <= 2 * dev.sms;
    cudaError_t e = cudaSuccess;
#define HCGR_RED(HCV)                                                                        \
  case HCV:                                                                                  \
    e = launch_maybe_pdl(batched ? k1_reduce_kernel<HCV, (HCV <= 4 ? 3 : 2)>               \
                                : k1_reduce_kernel<HCV, 1>,                                  \
                         grid, dim3(RED_THREADS), 0, stream, true, (const float*)part,        \
                         (const float*)sumsq, c.rrms, c.lora, c.inj_next, h, c.Wnorm,         \
                         static_cast<int>(c.ld_wnorm), w1, M, S, c.r, np, c.HS, 1.0f / c.HS,  \
                         c.eps);                                                              \
    break;
    switch (c.HC) {
      HCGR_RED(1) HCGR_RED(2) HCGR_RED(3) HCGR_RED(4) HCGR_RED(5) HCGR_RED(6) HCGR_RED(7)
      default: HCGR_RED(8)
    }
#undef HCGR_RED
    if (e != cudaSuccess) return e;
  }
  // ---------------- K2
  {
    K2Params p;
    const int ncu = k2_block(c.HC, n_mt, c.HS, dev.sms);
    const int N = c.HC * ncu;
    const uint64_t dh[2] = {static_cast<uint64_t>(c.r), static_cast<uint64_t>(M)};
    const uint64_t sh[1] = {static_cast<uint64_t>(c.r) * 2};
    const uint32_t bh[2] = {BK, BM};
    const uint64_t du[3] = {static_cast<uint64_t>(c.r), static_cast<uint64_t>(c.HS),
                            static_cast<uint64_t>(c.HC)};
    const uint64_t su[2] = {static_cast<uint64_t>(c.r) * 2, static_cast<uint64_t>(c.HS) * c.r * 2};
    const uint32_t bu[3] = {BK, static_cast<uint32_t>(ncu), static_cast<uint32_t>(c.HC)};
    const uint64_t dr[2] = {static_cast<uint64_t>(c.K), static_cast<uint64_t>(M)};
    const uint64_t sr[1] = {static_cast<uint64_t>(c.K) * 2};
    const uint32_t br[2] = {static_cast<uint32_t>(ncu), BM};
    const uint64_t dn[2] = {static_cast<uint64_t>(c.HS), static_cast<uint64_t>(c.HC)};
    const uint64_t sn[1] = {static_cast<uint64_t>(c.HS) * 4};
    const uint32_t bn[2] = {static_cast<uint32_t>(ncu), 1};
    const CUtensorMapSwizzle sw = ncu == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (!make_tmap_bf16(&p.tm_h, h, 2, dh, sh, bh, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_bf16(&p.tm_wu, c.Wu, 3, du, su, bu, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_bf16(&p.tm_r2, c.R2 ? c.R2 : c.R, 2, dr, sr, br, sw) ||   // mix only: R2 = R
        !make_tmap(&p.tm_w1, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, w1, 2, dn, sn, bn))
      return cudaErrorInvalidValue;
    p.rrms = c.rrms;
    p.x = c.x;
    p.M = M;
    p.HS = c.HS;
    p.r = c.r;
    p.nkb = c.r / BK;
    p.ncb = c.HS / ncu;
    p.n_units = n_mt * p.ncb;
    // shared memory: [stage ring | R2 stream slots | 1 + Wnorm slices | barriers]
    p.stage_bytes = TILE_BYTES + static_cast<uint32_t>(N) * 128u;
    const int box = BM * ncu * 2;
    const int avail = dev.smem_optin - 1024 - static_cast<int>(K2_BAR_BYTES);
    p.nst = 3;
    p.nr2 = std::min(K2_MAX_R2, (avail - p.nst * static_cast<int>(p.stage_bytes)) / (box + 256));
    if (p.nr2 < 2) {
      p.nst = 2;
      p.nr2 = std::min(K2_MAX_R2, (avail - p.nst * static_cast<int>(p.stage_bytes)) / (box + 256));
    }
    if (p.nr2 < 2 || p.nst > K2_MAX_ST) return cudaErrorNotSupported;
    p.off_r2 = static_cast<uint32_t>(p.nst) * p.stage_bytes;
    p.off_w1 = p.off_r2 + static_cast<uint32_t>(p.nr2 * box);
    p.off_bar = p.off_w1 + static_cast<uint32_t>(p.nr2) * 256u;
    p.err = ws.err;
    p.limit_ns = 1000ull * 1000 * 1000;
    const size_t smem = p.off_bar + K2_BAR_BYTES + 1024;
    if (smem > static_cast<size_t>(dev.smem_optin)) return cudaErrorNotSupported;
    const int grid = std::min(p.n_units, dev.sms);
    cudaError_t e = cudaSuccess;
    switch (c.HC) {
      case 1: e = launch_k2<1>(p, grid, smem, dev, stream, true); break;
      case 2: e = launch_k2<2>(p, grid, smem, dev, stream, true); break;
      case 3: e = launch_k2<3>(p, grid, smem, dev, stream, true); break;
      case 4: e = ncu == 32 ? launch_k2<4, 32>(p, grid, smem, dev, stream, true)
                            : launch_k2<4>(p, grid, smem, dev, stream, true); break;
      case 5: e = launch_k2<5>(p, grid, smem, dev, stream, true); break;
      case 6: e = launch_k2<6>(p, grid, smem, dev, stream, true); break;
      case 7: e = launch_k2<7>(p, grid, smem, dev, stream, true); break;
      default: e = launch_k2<8>(p, grid, smem, dev, stream, true); break;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace hcgr

// Decode path of the HC gated residual: one persistent kernel for small token
// counts (M <= 64), where the time goes into streaming the weights once
// (aiter PR #5913, "Technical Details"; the page's skinny decode with split-K
// partials and a last-stage reduce is the prior art).
//
// The grid has two roles, so that the whole weight set streams from HBM on
// every SM at once: Gd "down" CTAs hold the down/inject weight (Wd and Wi, or
// the merged Wdi), Gu "up" CTAs hold the up weight Wu.
//
// Down CTA b owns the channel slice [c0, c0 + 64 nkc) of stream s = b / P
// (P slices per stream; the stream end clips the last one):
//   1. COMBINE on the slice: R2 = bf16(R + y * iw) (stored), the partial sum
//      of R2^2 per token, and the MMA operand a = R2 * (1 + Wnorm) split into
//      two bf16 terms (hi + lo, ~16 mantissa bits), or a = R2 for a folded
//      weight, written to shared memory in the 128-byte swizzled K-major
//      layout of a tcgen05 operand.
//   2. On the tensor cores (tcgen05.mma, fp32 accumulators in TMEM), for
//      every 128-row tile of the down/inject weight (TMA, 128-byte swizzle):
//      D[n][m] = sum_{c in slice} W[n, s HS + c] a[m, c].  The hi and lo
//      terms are stacked as the two halves of the MMA's N dimension (one MMA
//      per weight tile and k-step), and one thread per row tile issues.
//      rrms_s is constant over stream s, so lora = sum_s rrms_s sum_{b in s}
//      D_b is exact: the per-stream factor commutes out of the K-sum.
//   3. Its piece of every reduce-scatter block (below) goes to a global
//      exchange buffer straight from TMEM; then the down CTA is done.
// Up CTA u owns the channel range [cp0, cp0 + nc) of every stream:
//   4. Reduce-scatter: the M (r + HC) outputs are cut into blocks of Qn
//      outputs of one token; up CTA j mod Gu reduces block j over the Gd
//      pieces in a fixed order (deterministic) and forms rrms, lora,
//      inj_next and h = bf16(SiLU(lora / HC)).
//   5. All-gather: the reducers publish h and rrms to a second exchange
//      buffer; every up CTA reads all of it into the swizzled operand layout,
//      forms the gates G[s, c] = sigmoid(Wu[s HS + c] . h) of its channel
//      range on the tensor cores (its Wu rows landed meanwhile), rebuilds xn
//      from R2 (recomputed from R, y and inj bit-identically to step 1), rrms
//      and Wnorm, and stores x = (1 / HC) sum_s G * xn.
// The exchanges need no grid barrier.  Every 32-bit word of an exchange
// buffer is either the empty marker 0xffffffff or a value, and readers poll
// (bounded in time) until the words they need hold values.  A value never
// equals the marker: floats are stored with NaN canonicalised, and h as a
// pair of bf16 from the rounding conversion, whose NaN is 0x7fff.  The
// reduce-scatter words are emptied again by their one reader at the end of
// its work; the all-gather buffer, which every up CTA reads, alternates
// between two copies by call parity (a ticket counter), and each call empties
// the copy the next call uses.  Whole warps poll together, sleeping briefly
// between rounds on the shared all-gather words: a warp whose lanes part for
// microseconds and then meet at a warp-synchronous instruction loses
// microseconds more, and many threads reading shared words back to back
// crowd the L2 slices those words live in.
//
// Without y (the mix alone) steps 1 and 5 take R as R2 and nothing is stored
// for it; the Wnorm slice of stream s starts at s * ld_wnorm (0 when one [HS]
// norm weight is shared by the streams).
//
// Weights move as TMA boxes issued first thing in the kernel; when they do not
// all fit in shared memory they stream through rings whose slots the MMA
// threads hand back with tcgen05.commit.  Every CTA allows the next kernel in
// the stream to launch early (once its call-ticket arrival is performed):
// that kernel's CTAs take the SMs the down CTAs leave and start their own
// weight copies while this call's up CTAs finish.  With a programmatic dependent launch the weight copies
// start before the previous kernel in the stream has finished; activations
// and exchange buffers are touched, and outputs written, only after it has.
// The kernel is short enough that instruction fetch matters: loops stay
// rolled.
//
// Built with HCGR_TRACE defined, the kernel records %globaltimer stamps of its
// phases per CTA in shared memory and writes them to a device array at its
// end (hc_gr_trace_read, include/hc_gr_trace.h).
#include <algorithm>

#include "hc_gr_internal.cuh"
#include "tmap.h"

namespace hcgr {
namespace {

constexpr int NT = 512;              // threads per CTA
constexpr int NW = NT / 32;
constexpr int MAX_SLOTS = 16;        // ring slots per weight stream
constexpr int XU = 8;                // exchange loads a thread keeps in flight
constexpr int DOWN_ISSUERS = 8;      // threads that may issue the down MMAs (one per row tile)
constexpr uint64_t PF_CHUNK = 16384;   // bytes per L2 prefetch of the weights
constexpr int PF_FIRST_THREAD = 128;   // the weight prefetches are issued by threads from here
constexpr int PF_INPUT_THREAD = 256;   // the COMBINE-input prefetches by threads from here
constexpr int UP_ISSUERS = 15;       // warps that may issue the gate MMAs (one per copy and row tile)
// Smallest reduce-scatter block (outputs of one token).  Measured on GB300 at
// HC=4, HS=2560, r=320: blocks of 36 rather than the 8, 12 or 20 that the
// one-block-per-up-CTA rule alone gives at M = 1, 2, 4 save 0.4-0.8 us per
// chained call and 0.3-0.7 us per plain launch; 44 is slower than 36 at
// every M (the down MMAs finish later), and at HC=8, HS=4096, r=512 the
// floor moves M = 1, 2 by -0.3 and +0.5 us of ~31.
constexpr int QN_MIN = 36;
constexpr int TILE = 16384;          // 128 rows x 64 bf16, 128-byte swizzle
constexpr int HDR = 1024;            // mbarriers, TMEM address, flags
constexpr int SMEM_BUDGET = 220 * 1024;
constexpr int SMEM_ALLOC = SMEM_BUDGET + 1024;
// Dynamic shared memory of a launch is at least this much, so that two CTAs
// (of this grid or of consecutive calls) never share an SM: every CTA holds
// tensor memory, and an exchange must never wait on a CTA that is not running.
constexpr int SMEM_MIN = 120 * 1024;

struct Geom {
  int Nt, Nd, Nu;                 // tokens rounded to 8; down MMA N (hi + lo); up MMA N
  int Gd, Gu, G;                  // down CTAs, up CTAs, grid
  int nkc, P;                     // down: 64-column chunks per slice, slices per stream
  int merged, rows_w, tail, wi_shared, wi_tile, wi_row, ntd, nsl_w;   // down weight
  int nc_max, rows_u, ntu, nchunk_u, slot_u, nsl_u, ncu;               // up weight
  int Qn, Jm, nred, row, nquad, R, ppr, L2w;                           // exchanges
  int tmem_d, tmem_u;             // tensor-memory columns of the two roles
  int d_ss1, d_ssum, d_act, d_w, d_total;                              // down shared memory
  int u_rr, u_iw, u_x3r, u_x3y, u_x3w, u_rl, u_red, u_g, u_hb, u_u, u_total;   // up
  int total;
};

__host__ __device__ inline int round_up(int v, int a) { return (v + a - 1) / a * a; }

struct Params {
  CUtensorMap tm_w;     // down weight (Wd, or merged Wdi) as [rows][HC][HS], box {64, 1, 128}
  CUtensorMap tm_wt;    // Wd's last rows when Wi shares their tile, box {64, 1, tail}
  CUtensorMap tm_wi;    // Wi as [HC][HC][HS], box {64, 1, HC}
  CUtensorMap tm_wu;    // Wu as [HC][HS][r], box {64, nc_max, HC}
  Call c;
  Geom g;
  uint32_t* xred;       // reduce-scatter words [nred][Gd][row]
  uint32_t* xgat;       // all-gather words, two copies of gat_words
  int gat_words;
  unsigned long long* ticket;
  int* err;
  uint64_t limit_ns;
};

int tmem_pow2(int cols) {
  return cols <= 32 ? 32 : cols <= 64 ? 64 : cols <= 128 ? 128 : cols <= 256 ? 256 : 512;
}

bool layout_down(Geom& g) {
  int off = HDR;
  g.d_ss1 = off;  off += round_up(g.Nt * g.nkc * 8 * 4, 128);
  g.d_ssum = off; off += round_up(g.Nt * 4, 128);
  off = round_up(off, 1024);
  g.d_act = off;  off += g.nkc * g.Nd * 128;          // [nkc][Nd rows][128 B], hi rows then lo rows
  g.d_w = off;    off += g.nsl_w * TILE;
  g.d_total = off;
  return off <= SMEM_BUDGET;
}

bool layout_up(const Call& c, Geom& g) {
  const int M = static_cast<int>(c.M), Nt = g.Nt;
  int off = HDR;
  g.u_rr = off;  off += round_up(Nt * c.HC * 4, 128);
  g.u_iw = off;  off += round_up(Nt * c.HC * 4, 128);
  g.u_x3r = off; off += round_up(M * c.HC * g.nc_max * 2, 128);
  g.u_x3y = off; off += round_up(M * g.nc_max * 2, 128);
  g.u_x3w = off; off += round_up(c.HC * g.nc_max * 2, 128);
  g.u_rl = off;  off += round_up(c.HC * 4, 128);
  g.u_red = off; off += round_up(c.HC * g.row * 4, 128);
  g.u_g = off;   off += round_up(M * g.rows_u * 4, 128);
  off = round_up(off, 1024);
  g.u_hb = off;  off += g.nchunk_u * g.Nu * 128;       // [nchunk_u][Nu rows][128 B]
  off = round_up(off, 1024);
  g.u_u = off;   off += g.nsl_u * g.slot_u;
  // the up-weight A tiles read ntu * TILE bytes from a slot's start: the
  // last slot's overhang stays inside the allocation
  off += std::max(0, g.ntu * TILE - g.slot_u);
  g.u_total = off;
  return off <= SMEM_BUDGET;
}

bool make_geom(const Call& c, const Device& dev, Geom& g) {
  const int M = static_cast<int>(c.M);
  if (M < 1 || M > DECODE_MAX_M || c.HS % 64 != 0 || c.r % 8 != 0 || c.HC > 8) return false;
  g.Nt = round_up(M, 8);
  g.Nd = 2 * g.Nt;
  g.Nu = round_up(M, 16);
  g.merged = c.Wi == c.Wd + static_cast<int64_t>(c.r) * c.K;   // rows r.. follow in one tensor
  g.rows_w = g.merged ? c.n_out : c.r;
  g.tail = g.rows_w % 128;
  const int nwd = (g.rows_w + 127) / 128;
  g.wi_shared = !g.merged && g.tail != 0 && g.tail + c.HC <= 128;
  g.wi_tile = g.merged ? -1 : (g.wi_shared ? nwd - 1 : nwd);
  g.wi_row = g.wi_shared ? g.tail : 0;
  g.ntd = g.merged || g.wi_shared ? nwd : nwd + 1;
  g.nchunk_u = (c.r + 63) / 64;
  if (g.ntd > DOWN_ISSUERS || g.nchunk_u > UP_ISSUERS) return false;
  const int hsc = c.HS / 64;                            // 64-column chunks per stream
  const int sms = std::min(dev.sms, MAX_GRID);
  // Every feasible slice size is planned; the plan kept is the one whose
  // larger per-CTA weight share (down: rows x slice, up: channel rows x r) is
  // smallest, since every CTA streams its share at about the same rate (the
  // up share weighted by 2 from 24 tokens, see below).
  Geom best;
  long long best_bytes = -1;
  for (g.nkc = 1; g.nkc <= hsc; ++g.nkc) {
    g.P = (hsc + g.nkc - 1) / g.nkc;
    g.Gd = c.HC * g.P;
    if (g.Gd >= sms) continue;
    // up CTAs: the remaining SMs, each a channel range (an even count) of
    // every stream; no up CTA without channels
    g.nc_max = round_up((c.HS + (sms - g.Gd) - 1) / (sms - g.Gd), 2);
    g.Gu = (c.HS + g.nc_max - 1) / g.nc_max;
    g.G = g.Gd + g.Gu;
    g.rows_u = c.HC * g.nc_max;
    if (g.nc_max > 256 || g.rows_u > 512) continue;
    g.ntu = (g.rows_u + 127) / 128;
    g.slot_u = round_up(g.rows_u * 128, 1024);
    // reduce-scatter blocks: the smallest Qn from QN_MIN (or the whole row,
    // if shorter) that gives every block an up CTA of its own
    for (g.Qn = std::min(QN_MIN, round_up(c.n_out, 4));; g.Qn += 4) {
      g.Jm = (c.n_out + g.Qn - 1) / g.Qn;
      if (M * g.Jm <= g.Gu || g.Jm == 1) break;
    }
    g.nred = M * g.Jm;
    g.row = g.Qn + 4;                       // Qn partials, the sum of squares, 3 pad words
    g.nquad = g.row / 4;
    if (g.nquad > NT) return false;
    // reducer: R sub-ranges (a power of two, consecutive lanes) of ppr
    // pieces per stream and quad; at most 4, so that a lane keeps several
    // loads in flight and the shuffle tree is at most two levels deep
    g.R = 1;
    while (2 * g.R <= 4 && 2 * g.R * c.HC * g.nquad <= NT) g.R *= 2;
    g.ppr = (g.P + g.R - 1) / g.R;
    g.L2w = round_up(c.r / 2 + c.HC, 4);     // h pairs, then rrms, then pad words
    // down: every box resident when they fit, else the deepest ring that
    // fits, with a multiple of ntd slots, so that each slot only ever holds
    // boxes of one row tile: its issuer then waits on the slot's phases in
    // order (a waiter more than one phase ahead would see the older phase)
    const int nbox = g.ntd * g.nkc;
    bool fits = false;
    for (int w = std::min(nbox, MAX_SLOTS); w >= 1 && !fits; --w) {
      if (w < nbox && w % g.ntd != 0) continue;
      g.nsl_w = w;
      fits = layout_down(g);
    }
    if (!fits) continue;
    // up: every chunk resident when it fits, else the deepest ring that fits.
    // The gate products accumulate in ncu tensor-memory copies (copy k takes
    // chunks k, k + ncu, ..; with a ring, ncu = slots, so a slot always feeds
    // the same copy), and one warp issues each (copy, row tile) chain, so up
    // to UP_ISSUERS warps issue side by side.  With every chunk resident, as
    // many copies as fit the tensor memory and the issuers.
    bool fits_u = false;
    for (int u = std::min(g.nchunk_u, MAX_SLOTS); u >= 1 && !fits_u; --u) {
      if (u < g.nchunk_u && u * g.ntu > UP_ISSUERS) continue;
      g.nsl_u = u;
      if (u >= g.nchunk_u) {
        g.ncu = std::max(1, std::min(g.nchunk_u, UP_ISSUERS / g.ntu));
        while (g.ncu > 1 && g.ncu * g.ntu * g.Nu > 512) --g.ncu;
      } else {
        g.ncu = u;
      }
      fits_u = g.ncu * g.ntu * g.Nu <= 512 && g.ncu * g.ntu <= UP_ISSUERS && layout_up(c, g);
    }
    if (!fits_u) continue;
    // down: one accumulator per row tile (one issuing warp each)
    const int cd = g.ntd * g.Nd, cu = g.ncu * g.ntu * g.Nu;
    if (cd > 512 || cu > 512) continue;
    g.tmem_d = tmem_pow2(cd);
    g.tmem_u = tmem_pow2(cu);
    g.total = std::max(std::max(g.d_total, g.u_total), SMEM_MIN - 1024);
    // a kernel that allocates TMEM runs one CTA per SM
    if (g.G > dev.sms) continue;
    // From about 24 tokens the up role's per-token work (the gather, the gate
    // readback and the gated mean, all proportional to its channel range)
    // outweighs the down role's extra MMAs, so the up share counts double:
    // measured at the default shape, 56 down / 96 up CTAs take 1.2 us less
    // than 80 / 72 at M = 32 and up to 1.1 us more at M <= 8.
    const long long down_b = static_cast<long long>(g.rows_w + (g.merged ? 0 : c.HC)) * g.nkc * 128;
    const long long up_b = static_cast<long long>(g.rows_u) * c.r * 2;
    const long long share = std::max(down_b, (M >= 24 ? 2 : 1) * up_b);
    if (best_bytes < 0 || share < best_bytes) {
      best = g;
      best_bytes = share;
    }
  }
  if (best_bytes < 0) return false;
  g = best;
  return true;
}

// Out-of-line slow paths of the bounded waits: one copy of each wait loop
// however many call sites.
__device__ __noinline__ bool wait_bar(uint32_t bar, uint32_t parity, int* err, uint64_t limit_ns) {
  return mbar_wait_bounded(bar, parity, err, limit_ns);
}
// A wait that ignores the status word (copies and MMAs always finish; this
// only lets them land before the CTA leaves), bounded by the time limit.
__device__ __noinline__ void drain_bar(uint32_t bar, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity) && clock64() - t0 < limit) {
  }
}


#ifdef HCGR_TRACE
constexpr int TRACE_SLOTS = 36;
__device__ unsigned long long g_trace[MAX_GRID * TRACE_SLOTS];
__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t) : : "memory");   // no memory access moves across it
  return t;
}
// Phase stamp i of this CTA (the calling thread records it in shared memory;
// the kernel's end writes the CTA's stamps out); HCGR_STAMP_MAX keeps the
// latest time any thread reaches the point.
#define HCGR_STAMP(i) (s_stamp[(i)] = globaltimer_ns())
#define HCGR_STAMP_MAX(i) atomicMax(&s_stamp[(i)], globaltimer_ns())
#else
#define HCGR_STAMP(i) ((void)0)
#define HCGR_STAMP_MAX(i) ((void)0)
#endif

// --------------------------------------------------------------- the kernel
__global__ void __launch_bounds__(NT, 1) decode_kernel(const __grid_constant__ Params p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Call& c = p.c;
  const Geom& g = p.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#ifdef HCGR_TRACE
  __shared__ unsigned long long s_stamp[TRACE_SLOTS];
  if (tid < TRACE_SLOTS) s_stamp[tid] = 0;
#endif
  // Every CTA first asks L2 for its 1/G share of the weights, in contiguous
  // pieces of up to 16 KB: HBM streams them in long runs (the box copies of
  // the operand layout read 128-byte pieces of many rows, a pattern HBM
  // serves at about two thirds of the rate) from the kernel's first
  // instructions on, and the box copies issued later mostly hit L2.  The
  // weights never depend on the previous kernel, so this precedes
  // griddepcontrol.wait.  Warps 4.. issue them: the prologue's other jobs
  // (barrier initialisation in warps 0-2, the call ticket in the last warp)
  // then run side by side, since a thread's second bulk copy instruction
  // waits for its first to be taken.  Only when every CTA holds its whole
  // share in shared memory: with rings (weights larger than the SMs' shared
  // memory) the early stream of all the weights competes with the boxes the
  // rings need first, and measured slower.
  const bool resident = g.nsl_w >= g.ntd * g.nkc && g.nsl_u >= g.nchunk_u;
  if (resident && threadIdx.x >= PF_FIRST_THREAD) {
    const uint64_t G = gridDim.x, me = blockIdx.x;
    const uint64_t rK = static_cast<uint64_t>(c.r) * c.K, hK = static_cast<uint64_t>(c.HC) * c.K;
    const bool merged_w = c.Wi == c.Wd + rK;
    // [lo, hi) of this CTA's share of a buffer of n bytes (16-byte bounds)
    auto share = [&](uint64_t n, uint64_t& lo, uint64_t& hi) {
      const uint64_t piece = (n / G + 16) & ~15ull;   // > n / G, a multiple of 16
      lo = min(n, piece * me);
      hi = min(n, lo + piece);
    };
    uint64_t lo0, hi0, lo1, hi1, lo2, hi2;
    share(2 * (merged_w ? rK + hK : rK), lo0, hi0);
    share(merged_w ? 0 : 2 * hK, lo1, hi1);
    share(2 * rK, lo2, hi2);
    const int n0 = static_cast<int>((hi0 - lo0 + PF_CHUNK - 1) / PF_CHUNK);
    const int n1 = static_cast<int>((hi1 - lo1 + PF_CHUNK - 1) / PF_CHUNK);
    const int n2 = static_cast<int>((hi2 - lo2 + PF_CHUNK - 1) / PF_CHUNK);
#pragma unroll 1
    for (int i = threadIdx.x - PF_FIRST_THREAD; i < n0 + n1 + n2; i += NT - PF_FIRST_THREAD) {
      const char* src;
      uint64_t a, end;
      if (i < n0) {
        src = reinterpret_cast<const char*>(c.Wd); a = lo0 + i * PF_CHUNK; end = hi0;
      } else if (i < n0 + n1) {
        src = reinterpret_cast<const char*>(c.Wi); a = lo1 + (i - n0) * PF_CHUNK; end = hi1;
      } else {
        src = reinterpret_cast<const char*>(c.Wu); a = lo2 + (i - n0 - n1) * PF_CHUNK; end = hi2;
      }
      bulk_prefetch_l2(src + a, static_cast<uint32_t>(end - a < PF_CHUNK ? end - a : PF_CHUNK));
    }
  }
  const int b = blockIdx.x;
  const int M = static_cast<int>(c.M), Nt = g.Nt, Nd = g.Nd, Nu = g.Nu;
  const int HC = c.HC, HS = c.HS, K = c.K, r = c.r, n_out = c.n_out;
  const long long limit = wait_limit_cycles(p.limit_ns);
  const bool down = b < g.Gd;
  const bool has_y = c.y != nullptr;   // false: mix only, R2 = R
  const float inv_hc = 1.0f / static_cast<float>(HC);
  if (tid == 0) HCGR_STAMP(0);

  const uint32_t bar0 = smem_u32(smem);
  // MAX_SLOTS barriers each: full/free of the down ring, full/free of the up ring
  auto full_w = [&](int i) { return bar0 + 8u * i; };
  auto free_w = [&](int i) { return bar0 + 8u * (MAX_SLOTS + i); };
  auto full_u = [&](int i) { return bar0 + 8u * (2 * MAX_SLOTS + i); };
  auto free_u = [&](int i) { return bar0 + 8u * (3 * MAX_SLOTS + i); };
  const uint32_t barD = bar0 + 8u * 4 * MAX_SLOTS, barG = barD + 8u;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + 8 * 4 * MAX_SLOTS + 16);
  uint32_t* s_epoch = s_tmem + 1;
  int* s_mma_ok = reinterpret_cast<int*>(s_tmem + 2);

  // this CTA's work: the down slice, or the up channel range
  const int s = down ? b / g.P : 0;
  const int c0 = down ? (b % g.P) * 64 * g.nkc : 0;
  const int nkv = down ? min(g.nkc, (HS - c0) / 64) : 0;       // chunks of the slice
  const int k0 = s * HS + c0;
  const int nbox = g.ntd * nkv;                                // down weight boxes
  // The COMBINE inputs of a down CTA's slice (R and y rows of every token,
  // the Wnorm slice) into L2 as well: L2 is the point of coherence, so a
  // prefetch before griddepcontrol.wait never hands out data older than a
  // write the previous kernel makes (it only warms the lines).
  if (down && nkv > 0 && tid >= PF_INPUT_THREAD && tid - PF_INPUT_THREAD <= 2 * M) {
    const int j = tid - PF_INPUT_THREAD;
    const uint32_t sb = static_cast<uint32_t>(min(64 * g.nkc, HS - c0)) * 2;
    if (j < M)
      bulk_prefetch_l2(c.R + static_cast<int64_t>(j) * K + k0, sb);
    else if (j < 2 * M && has_y)
      bulk_prefetch_l2(c.y + static_cast<int64_t>(j - M) * HS + c0, sb);
    else if (j == 2 * M)
      bulk_prefetch_l2(c.Wnorm + s * c.ld_wnorm + c0, sb);
  }
  const int u_idx = down ? 0 : b - g.Gd;
  const int cp0 = down ? 0 : min(HS, u_idx * g.nc_max);
  const int nc = down ? 0 : min(HS, cp0 + g.nc_max) - cp0;
  const int nub = nc > 0 ? g.nchunk_u : 0;                     // up weight boxes
  const uint32_t wbase = smem_u32(smem + g.d_w);               // down weight slots
  const uint32_t ubase = smem_u32(smem + g.u_u);               // up weight slots

  auto issue_w = [&](int i) {   // box i: chunk i / ntd, row tile i % ntd
    const int ch = i / g.ntd, t = i - ch * g.ntd, slot = i % g.nsl_w;
    const uint32_t dst = wbase + slot * TILE;
    const int x = c0 + ch * 64;
    const bool wd = t * 128 < g.rows_w;
    const bool wt = wd && g.wi_shared && t == g.wi_tile;
    const bool wi = t == g.wi_tile;
    const uint32_t bytes = (wd ? (wt ? g.tail : 128) * 128 : 0) + (wi ? HC * 128 : 0);
    mbar_arrive_expect_tx(full_w(slot), bytes);
    if (wd) tma_load_3d(dst, wt ? &p.tm_wt : &p.tm_w, x, s, t * 128, full_w(slot));
    if (wi) tma_load_3d(dst + g.wi_row * 128, &p.tm_wi, x, s, 0, full_w(slot));
  };
  auto issue_u = [&](int q) {
    const int slot = q % g.nsl_u;
    mbar_arrive_expect_tx(full_u(slot), static_cast<uint32_t>(g.rows_u * 128));
    tma_load_3d(ubase + slot * g.slot_u, &p.tm_wu, q * 64, cp0, 0, full_u(slot));
  };

  // Prologue: thread 0 initialises the barriers, then lane 0 of warp w
  // issues the role's weight box w, so the issue latencies overlap; warp 15
  // takes the call ticket and warp 3 allocates TMEM meanwhile.  None of this
  // depends on the previous kernel.
  const int pre_w = min(g.nsl_w, nbox), pre_u = min(g.nsl_u, nub);
  int issued_w = down ? pre_w : 0, issued_u = down ? 0 : pre_u;   // kept by warp 0
  // The call ticket: arrivals in the low half, the call's epoch in the high
  // half.  Lane 1 of the last warp takes it now and uses the result only at
  // the CTA's first barrier after the prologue (take_ticket), so the atomic's
  // round trip hides behind the prologue.
  unsigned long long ticket_old = 0;
  if (warp == NW - 1 && lane == 1) ticket_old = atomicAdd(p.ticket, 1ull);
  // The last arrival moves the epoch on and clears the count.  Both atomics
  // are performed before this thread reaches the CTA barrier that precedes
  // the trigger of the next launch, so no arrival of the next call can come
  // between this call's arrivals and its roll-over.
  auto take_ticket = [&]() {
    if (warp == NW - 1 && lane == 1) {
      if ((ticket_old & 0xffffffffull) == static_cast<unsigned long long>(g.G - 1)) {
        atomicAdd(p.ticket, (1ull << 32) - static_cast<unsigned long long>(g.G));
        __threadfence();
      }
      *s_epoch = static_cast<uint32_t>(ticket_old >> 32);
    }
  };
  // Barrier initialisation, one barrier per thread of warps 0-2 (one thread
  // initialising all of them in turn took ~1 µs): full/free of the down
  // ring and full of the up ring count one arrival; an up slot is free once
  // the MMAs of each row tile (one issuer each) have read it; barD and barG
  // take one commit per candidate issuer warp.
  if (tid == 0) HCGR_STAMP(32);
  if (tid < 4 * MAX_SLOTS + 2) {
    const uint32_t count = tid < 3 * MAX_SLOTS ? 1u
                           : tid < 4 * MAX_SLOTS ? static_cast<uint32_t>(g.ntu)
                           : tid == 4 * MAX_SLOTS ? static_cast<uint32_t>(DOWN_ISSUERS)
                                                  : static_cast<uint32_t>(UP_ISSUERS);
    mbar_init(bar0 + 8u * tid, count);
    fence_mbar_init();
  }
  if (tid == 0) {
    *s_mma_ok = 1;
    HCGR_STAMP(33);
  }
  HCGR_STAMP_MAX(34);
  __syncthreads();
  if (tid == 0) HCGR_STAMP(13);
  if (lane == 0) {
    const int npre = down ? pre_w : pre_u;
    if (warp < npre) prefetch_tmap(down ? &p.tm_w : &p.tm_wu);
#pragma unroll 1
    for (int k = warp; k < npre; k += NW) {
      if (down) issue_w(k);
      else issue_u(k);
      if (tid == 0 && k == 0) HCGR_STAMP(14);
    }
  }
  const int tmem_cols = down ? g.tmem_d : g.tmem_u;
  if (warp == 3) {
    __syncwarp();
    tmem_alloc(smem_u32(s_tmem), tmem_cols);
    tmem_relinquish();
  }
  if (tid == 0) HCGR_STAMP(1);
  // inputs, outputs and exchange buffers may belong to the previous kernel
  grid_dep_wait();
  if (tid == 0) HCGR_STAMP(2);

  bool ok = true;
  bool down_issued = false, up_issued = false;   // MMAs to drain at the end
  if (down) {
    // ====================================================== down role
    float* s_ss1 = reinterpret_cast<float*>(smem + g.d_ss1);   // [Nt][8 nkc]
    float* s_ssum = reinterpret_cast<float*>(smem + g.d_ssum); // [Nt] sum of R2^2 on the slice
    const uint32_t act = smem_u32(smem + g.d_act);             // [nkc][Nd rows][128 B]

    // --- step 1: COMBINE on this CTA's slice, R2 stored, MMA operands in the
    // swizzled layout (16-byte unit u of row m of a chunk at (u ^ (m & 7)) *
    // 16; hi in rows m, lo in rows Nt + m)
    const int nu = g.nkc * 8;                                  // 16-byte units per row
    const int nitem = Nt * nu;
    // a thread takes two items per pass and issues all their loads before it
    // uses any, so that a CTA with more items than threads waits through one
    // round of input loads, not two
#pragma unroll 1
    for (int it0 = tid; it0 < nitem; it0 += 2 * NT) {
      uint4 rq[2], yq[2], wq[2];
      float injv[2] = {0.f, 0.f};
      bool val[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int it = it0 + e * NT;
        const int m = it / nu, un = it - m * nu;
        val[e] = it < nitem && m < M && (un >> 3) < nkv;
        rq[e] = yq[e] = wq[e] = make_uint4(0, 0, 0, 0);
        if (val[e]) {
          rq[e] = __ldg(reinterpret_cast<const uint4*>(c.R + static_cast<int64_t>(m) * K + k0 + un * 8));
          if (has_y) {
            injv[e] = c.inj[m * c.ld_inj + s];
            yq[e] = __ldg(reinterpret_cast<const uint4*>(c.y + static_cast<int64_t>(m) * HS + c0 + un * 8));
          }
          wq[e] = __ldg(reinterpret_cast<const uint4*>(c.Wnorm + s * c.ld_wnorm + c0 + un * 8));
        }
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int it = it0 + e * NT;
        if (it >= nitem) break;
        const int m = it / nu, un = it - m * nu;
        const int ch = un >> 3, uu = un & 7;
        uint4 hv = make_uint4(0, 0, 0, 0), lv = make_uint4(0, 0, 0, 0);
        float ss = 0.f;
        if (val[e]) {
          const int64_t kk = static_cast<int64_t>(m) * K + k0 + un * 8;
          float rv[8], yv[8] = {}, wv[8], a[8];
          float iw = 0.f;
          unpack8(rq[e], rv);
          if (has_y) {
            iw = combine_weight(injv[e], inv_hc);
            unpack8(yq[e], yv);
          }
          unpack8(wq[e], wv);
          uint32_t pr[4], ph[4], pl[4];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float r2 = has_y ? bf16_to_f32(f32_to_bf16(fmaf(yv[i], iw, rv[i]))) : rv[i];
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
          if (c.R2) *reinterpret_cast<uint4*>(c.R2 + kk) = make_uint4(pr[0], pr[1], pr[2], pr[3]);
          hv = make_uint4(ph[0], ph[1], ph[2], ph[3]);
          lv = make_uint4(pl[0], pl[1], pl[2], pl[3]);
        }
        const int sw = ch * Nd * 128 + m * 128 + ((uu ^ (m & 7)) << 4);
        *reinterpret_cast<uint4*>(smem + g.d_act + sw) = hv;
        *reinterpret_cast<uint4*>(smem + g.d_act + sw + Nt * 128) = lv;
        s_ss1[m * nu + un] = ss;
      }
    }
    fence_proxy_async_smem();   // the operand rows are read by the tensor cores
    take_ticket();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) HCGR_STAMP(3);
    // This CTA's call-ticket arrival is performed (the barrier above follows
    // it): the next kernel in the stream may launch.  Its CTAs wait for SMs
    // this grid frees, then for this grid's end before they touch
    // activations or exchange buffers.
    grid_dep_launch();
    const uint32_t tmem = *s_tmem;

    // --- step 2: the down/inject products on the tensor cores: warp 2t + 1
    // walks the MMAs of row tile t (all chunks, one accumulator per tile) and
    // one elected lane issues, so up to DOWN_ISSUERS warps issue side by
    // side.  With a ring, warp 0 refills each slot once the MMAs that read it
    // have completed; every issuer warp commits barD.  Whole warps wait
    // together: a warp whose lanes part for microseconds and then meet at a
    // warp-synchronous instruction loses microseconds more.
    const bool dead = c.debug_fault == 1 && b == 0;   // test hook: this CTA writes nothing
    if ((warp & 1) == 1 && (warp >> 1) < DOWN_ISSUERS) {
      const int me = warp >> 1;
      const uint32_t idesc = idesc_bf16(128, Nd);
      bool okm = true;
#pragma unroll 1
      for (int i = me; i < nbox && okm && me < g.ntd; i += g.ntd) {
        const int ch = i / g.ntd, slot = i % g.nsl_w;
        const uint32_t ph = (i / g.nsl_w) & 1;
        okm = __all_sync(0xffffffffu,
                         mbar_test_wait(full_w(slot), ph) || wait_bar(full_w(slot), ph, p.err, p.limit_ns));
        if (!okm) break;
        if (me == 0 && lane == 0 && i == me) HCGR_STAMP(24);
        tc_fence_after();
        const uint32_t a = wbase + slot * TILE, bq = act + ch * Nd * 128;
        const uint32_t d = tmem + me * Nd;
        if (elect_one()) {
#pragma unroll 1
          for (int ks = 0; ks < 4; ++ks)
            umma_bf16(d, desc_sw128(a + ks * 32), desc_sw128(bq + ks * 32), idesc, (ch || ks) ? 1u : 0u);
          umma_commit(free_w(slot));
          if (me == 0 && i == me) HCGR_STAMP(25);
        }
        __syncwarp();
      }
      if (me == 0 && lane == 0) HCGR_STAMP(4);
      if (!okm && lane == 0) *s_mma_ok = 0;
      if (elect_one()) umma_commit(barD);
      __syncwarp();
    } else if (warp == 0) {
      // ring refills: a slot is free once the MMAs that read it have completed
#pragma unroll 1
      for (int i = pre_w; i < nbox; ++i) {
        const int slot = i % g.nsl_w;
        if (!__all_sync(0xffffffffu, wait_bar(free_w(slot), ((i / g.nsl_w) - 1) & 1, p.err, p.limit_ns)))
          break;
        if (lane == 0) issue_w(i);
        __syncwarp();
        ++issued_w;
      }
    }
    down_issued = true;
    // the sum of squares, and the non-product words of this CTA's piece of
    // every reduce-scatter block ([Qn partials][sum of squares][3 pad
    // words], partials past n_out zero)
    if (tid < Nt) {
      float ss = 0.f;
#pragma unroll 1
      for (int j = 0; j < nkv * 8; ++j) ss += s_ss1[tid * nu + j];
      s_ssum[tid] = ss;
    }
    __syncthreads();
    if (!dead) {
#pragma unroll 1
      for (int j = tid; j < g.nred; j += NT) {
        const int m = j / g.Jm, jn = j - m * g.Jm;
        uint32_t* dst = p.xred + (static_cast<size_t>(j) * g.Gd + b) * g.row;
        st_relaxed_v4(dst + g.Qn, make_uint4(xword(s_ssum[m]), 0u, 0u, 0u));
#pragma unroll 1
        for (int q = n_out - jn * g.Qn; q < g.Qn; ++q) st_relaxed_u32(dst + q, 0u);
      }
    }
    // the products, straight from TMEM (hi + lo halves): warp w reads lanes
    // 32 (w % 4) ..; the four warp groups take alternate (tile, 8-token) items
    ok = __all_sync(0xffffffffu, wait_bar(barD, 0, p.err, p.limit_ns));
    if (tid == 0) HCGR_STAMP(30);
    tc_fence_after();
    ok = __syncthreads_and(ok && *s_mma_ok != 0);
    if (tid == 0) HCGR_STAMP(5);
    if (ok && !dead) {
      const int q4 = warp & 3, grp = warp >> 2;
      const int tr = 32 * q4 + lane;                           // row within a tile
      const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q4) << 16);
      const int nmc = Nt / 8;                                  // 8-token chunks
#pragma unroll 1
      for (int item = grp; item < g.ntd * nmc; item += NW / 4) {
        const int t = item / nmc, m0 = (item - t * nmc) * 8;
        const int rt = t * 128 + tr;
        const bool inj_row = t == g.wi_tile && tr >= g.wi_row;
        const int n = inj_row ? r + (tr - g.wi_row) : rt;
        const bool valid = inj_row ? n < n_out : rt < g.rows_w;
        const int jn = n / g.Qn, qn = n - jn * g.Qn;
        uint32_t h0[8], l0[8];
        tmem_ld8x2_wait(tl + t * Nd + m0, tl + t * Nd + Nt + m0, h0, l0);
        if (item == grp) HCGR_STAMP_MAX(23);
        if (valid) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float v = __uint_as_float(h0[e]) + __uint_as_float(l0[e]);
            if (m0 + e < M)
              st_relaxed_u32(p.xred + (static_cast<size_t>((m0 + e) * g.Jm + jn) * g.Gd + b) * g.row + qn,
                             xword(v));
          }
        }
        HCGR_STAMP_MAX(16);
      }
    }
    if (tid == 0) HCGR_STAMP(6);
  } else {
    // ======================================================== up role
    float* s_rr = reinterpret_cast<float*>(smem + g.u_rr);     // [Nt][HC] rrms (all-gather)
    float* s_iw = reinterpret_cast<float*>(smem + g.u_iw);     // [Nt][HC]
    bf16_t* s_x3r = reinterpret_cast<bf16_t*>(smem + g.u_x3r); // [M][HC][nc_max]
    bf16_t* s_x3y = reinterpret_cast<bf16_t*>(smem + g.u_x3y); // [M][nc_max]
    bf16_t* s_x3w = reinterpret_cast<bf16_t*>(smem + g.u_x3w); // [HC][nc_max]
    float* s_rl = reinterpret_cast<float*>(smem + g.u_rl);     // [HC] the reducer's rrms
    float* s_red = reinterpret_cast<float*>(smem + g.u_red);   // [HC][row]
    float* s_g = reinterpret_cast<float*>(smem + g.u_g);       // [M][rows_u]
    const uint32_t hbase = smem_u32(smem + g.u_hb);            // [nchunk_u][Nu rows][128 B]

    // Inputs of this CTA's channel range for the final mix -- R, y, Wnorm in
    // channel pairs, and inj (iw is formed from it later) -- copied
    // asynchronously now, so that their latency hides behind the reduce.
    {
      const int np = nc / 2;
      const int n_iw = has_y ? M * HC : 0, n_r = M * HC * np, n_y = has_y ? M * np : 0, n_w = HC * np;
#pragma unroll 1
      for (int i = tid; i < n_iw + n_r + n_y + n_w; i += NT) {
        if (i < n_iw) {
          cp_async4(s_iw + i, c.inj + (i / HC) * c.ld_inj + (i % HC));
        } else if (i < n_iw + n_r) {
          const int j = i - n_iw, rw = j / np, cc = 2 * (j - rw * np);   // rw = m * HC + stream
          const int m = rw / HC, ss = rw - m * HC;
          cp_async4(s_x3r + rw * g.nc_max + cc, c.R + static_cast<int64_t>(m) * K + ss * HS + cp0 + cc);
        } else if (i < n_iw + n_r + n_y) {
          const int j = i - n_iw - n_r, m = j / np, cc = 2 * (j - m * np);
          cp_async4(s_x3y + m * g.nc_max + cc, c.y + static_cast<int64_t>(m) * HS + cp0 + cc);
        } else {
          const int j = i - n_iw - n_r - n_y, ss = j / np, cc = 2 * (j - ss * np);
          cp_async4(s_x3w + ss * g.nc_max + cc, c.Wnorm + ss * c.ld_wnorm + cp0 + cc);
        }
      }
    }
    // the call ticket's arrival (warp 15) is performed past this barrier:
    // the next kernel in the stream may launch (see the down role)
    take_ticket();
    __syncthreads();
    grid_dep_launch();
    const uint32_t par = *s_epoch & 1u;
    uint32_t* gat = p.xgat + static_cast<size_t>(par) * p.gat_words;

    // --- step 4: the reducer of blocks u, u + Gu, ...  Work item (stream,
    // quad, sub-range) sums quad uq of the stream's pieces in its sub-range,
    // XU loads in flight; the R sub-ranges of one (stream, quad) sit in
    // consecutive lanes and fold with a fixed shuffle tree (deterministic).
#pragma unroll 1
    for (int j = u_idx; j < g.nred && ok; j += g.Gu) {
      const int m = j / g.Jm, jn = j - m * g.Jm;
      const uint32_t* blk = p.xred + static_cast<size_t>(j) * g.Gd * g.row;
      bool got = true;
      const int nitem = HC * g.nquad * g.R;
#pragma unroll 1
      for (int wi0 = 0; wi0 < nitem; wi0 += NT) {            // uniform: whole warps shuffle
        const int wi = wi0 + tid;
        const int su = wi / g.R, jr = wi - su * g.R;         // su = stream * nquad + quad
        const int ss = su / g.nquad, uq = su - ss * g.nquad;
        const int p0 = jr * g.ppr, p1 = wi < nitem ? min(g.P, p0 + g.ppr) : p0;
        float run[4] = {0.f, 0.f, 0.f, 0.f};
        // the warp's lanes take ppr pieces each (a uniform trip count) and
        // poll their missing words together until every lane's are there
#pragma unroll 1
        for (int t0 = 0; t0 < g.ppr && got; t0 += XU) {
          const uint32_t* src = blk + (ss * g.P + p0 + t0) * g.row + uq * 4;
          const int nv = p1 - p0 - t0;                       // this lane's pieces here (may be <= 0)
          uint4 v[XU];
#pragma unroll
          for (int k = 0; k < XU; ++k)
            v[k] = k < nv ? ld_relaxed_v4(src + k * g.row) : make_uint4(0u, 0u, 0u, 0u);
          long long t_wait = 0;
#pragma unroll 1
          for (int it = 0;; ++it) {
            bool mine = true;
#pragma unroll
            for (int k = 0; k < XU; ++k) mine = mine && all_set(v[k]);
            if (__all_sync(0xffffffffu, mine)) break;
            if (it == 0) t_wait = clock64();
            if ((it & 15) == 15) {
              const bool late = clock64() - t_wait > limit;
              if (__any_sync(0xffffffffu, late || *((volatile int*)p.err) != DEV_OK)) {
                if (late && lane == 0) atomicCAS(p.err, DEV_OK, DEV_TIMEOUT);
                got = false;
                break;
              }
            }
            __nanosleep(96);   // fewer reads of lines the down CTAs are writing
#pragma unroll
            for (int k = 0; k < XU; ++k)
              if (!all_set(v[k])) v[k] = ld_relaxed_v4(src + k * g.row);   // only k < nv are unset
          }
          if (!got) break;
          if (j == u_idx && nv > 0) HCGR_STAMP_MAX(17);
#pragma unroll
          for (int k = 0; k < XU; ++k) {
            if (k >= nv) break;
            run[0] += __uint_as_float(v[k].x);
            run[1] += __uint_as_float(v[k].y);
            run[2] += __uint_as_float(v[k].z);
            run[3] += __uint_as_float(v[k].w);
          }
        }
        if (j == u_idx) HCGR_STAMP_MAX(18);
#pragma unroll 1
        for (int o = g.R / 2; o > 0; o >>= 1)
#pragma unroll
          for (int e = 0; e < 4; ++e) run[e] += __shfl_xor_sync(0xffffffffu, run[e], o);
        if (j == u_idx) HCGR_STAMP_MAX(19);
        if (wi < nitem && jr == 0)
          *reinterpret_cast<float4*>(s_red + ss * g.row + uq * 4) = make_float4(run[0], run[1], run[2], run[3]);
        if (j == u_idx) HCGR_STAMP_MAX(20);
      }
      ok = __syncthreads_and(got);
      if (!ok) break;
      if (tid == 0 && j == u_idx) HCGR_STAMP(7);
      if (tid < HC) {
        const float rr = rsqrt_nr(fmaf(s_red[tid * g.row + g.Qn], __fdividef(1.0f, static_cast<float>(HS)), c.eps));
        s_rl[tid] = rr;
        if (jn == 0) c.rrms[m * HC + tid] = rr;
      }
      __syncthreads();
#pragma unroll 1
      for (int qp = tid; qp < g.Qn / 2; qp += NT) {
        float v[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int q = 2 * qp + e;
          float a = 0.f;
#pragma unroll 1
          for (int ss = 0; ss < HC; ++ss) a += s_rl[ss] * s_red[ss * g.row + q];
          v[e] = a;
          const int n = jn * g.Qn + q;
          if (n < r)
            c.lora[static_cast<int64_t>(m) * r + n] = a;
          else if (n < n_out)
            c.inj_next[static_cast<int64_t>(m) * HC + (n - r)] = a;
        }
        const int n0 = jn * g.Qn + 2 * qp;
        if (n0 < r) {   // r is even: n0 + 1 < r too
          const float u0 = v[0] * inv_hc, u1 = v[1] * inv_hc;
          st_relaxed_u32(gat + m * g.L2w + n0 / 2, pack2(u0 * sigmoid_fast(u0), u1 * sigmoid_fast(u1)));
        }
      }
      if (jn == 0) {
#pragma unroll 1
        for (int i = r / 2 + tid; i < g.L2w; i += NT) {
          const int ss = i - r / 2;
          st_relaxed_u32(gat + m * g.L2w + i, ss < HC ? xword(s_rl[ss]) : 0u);
        }
      }
      __syncthreads();   // s_red is reused by the next block
    }
    const bool red_done = ok;   // every block of this CTA read (and reduced)
    if (tid == 0) HCGR_STAMP(8);
    // the final mix's inputs (copied since the prologue) have landed; iw from
    // inj (each thread converts the words it copied)
    cp_async_wait_all();
#pragma unroll 1
    for (int i = tid; i < M * HC; i += NT) s_iw[i] = has_y ? combine_weight(s_iw[i], inv_hc) : 0.f;
    if (tid == 0) HCGR_STAMP(29);

    // --- step 5: all-gather of h (into the swizzled operand layout) and
    // rrms: each warp polls its quads together until all of them hold values
    if (ok && nc > 0) {
      bool got = true;
      const int hw = r / 2;
      const int nq = M * g.L2w / 4;
#pragma unroll 1
      for (int i0 = warp * 32; i0 < nq && got; i0 += XU * NT) {   // warp-uniform trip count
        uint4 v[XU];
#pragma unroll
        for (int k = 0; k < XU; ++k) {
          const int i = i0 + lane + k * NT;
          v[k] = i < nq ? ld_relaxed_v4(gat + i * 4) : make_uint4(0u, 0u, 0u, 0u);
        }
        long long t_wait = 0;
#pragma unroll 1
        for (int it = 0;; ++it) {
          bool mine = true;
#pragma unroll
          for (int k = 0; k < XU; ++k) mine = mine && all_set(v[k]);
          if (__all_sync(0xffffffffu, mine)) break;
          if (it == 0) t_wait = clock64();
          if ((it & 7) == 7) {
            const bool late = clock64() - t_wait > limit;
            if (__any_sync(0xffffffffu, late || *((volatile int*)p.err) != DEV_OK)) {
              if (late && lane == 0) atomicCAS(p.err, DEV_OK, DEV_TIMEOUT);
              got = false;
              break;
            }
          }
          __nanosleep(64);
#pragma unroll
          for (int k = 0; k < XU; ++k)
            if (!all_set(v[k])) v[k] = ld_relaxed_v4(gat + (i0 + lane + k * NT) * 4);   // only i < nq are unset
        }
        if (!got) break;
#pragma unroll
        for (int k = 0; k < XU; ++k) {
          const int i = i0 + lane + k * NT;
          if (i >= nq) break;
          // r / 2 and L2w are multiples of 4: a quad is 8 h values or rrms/pad
          const int m = (i * 4) / g.L2w, w0 = i * 4 - m * g.L2w;
          if (w0 < hw) {
            const int n0 = 2 * w0;                                  // 8 values from n0
            const int q = n0 >> 6, un = (n0 & 63) >> 3;
            *reinterpret_cast<uint4*>(smem + g.u_hb + q * Nu * 128 + m * 128 +
                                      ((un ^ (m & 7)) << 4)) = v[k];
          } else {
            const uint32_t vv[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (w0 + e < hw + HC) s_rr[m * HC + w0 + e - hw] = __uint_as_float(vv[e]);
          }
        }
      }
      HCGR_STAMP_MAX(26);
      // token rows past M, and h columns past r in the last chunk, are zero
#pragma unroll 1
      for (int i = tid; i < g.nchunk_u * Nu * 8; i += NT) {
        const int q = i / (Nu * 8), rem = i - q * Nu * 8, m = rem >> 3, un = rem & 7;
        if (m >= M || q * 64 + un * 8 >= r)
          *reinterpret_cast<uint4*>(smem + g.u_hb + q * Nu * 128 + m * 128 + ((un ^ (m & 7)) << 4)) =
              make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
      ok = __syncthreads_and(got);
    }
    if (tid == 0) HCGR_STAMP(9);
    // the gates on the tensor cores: D[row][m] = Wu[row] . h[m], rows (stream,
    // channel) of this CTA's range.  Warp 1 + k * ntu + t (k < ncu) walks
    // chunks k, k + ncu, .. of row tile t (with a ring, always the same slot)
    // into accumulator copy k and one elected lane issues.  Every candidate
    // warp (1 .. UP_ISSUERS) commits barG.
    const uint32_t tmem = *s_tmem;
    up_issued = ok && nc > 0;
    if (up_issued) {
      if (warp >= 1 && warp <= UP_ISSUERS) {
        const int me = warp - 1, kc = me / g.ntu, tu = me - kc * g.ntu;
        tc_fence_after();
        const uint32_t idesc = idesc_bf16(128, Nu);
        const uint32_t d = tmem + (kc * g.ntu + tu) * Nu;
        bool okm = true;
#pragma unroll 1
        for (int q = kc; q < nub && okm && me < g.ncu * g.ntu; q += g.ncu) {
          const int slot = q % g.nsl_u;
          const uint32_t ph = (q / g.nsl_u) & 1;
          okm = __all_sync(0xffffffffu,
                           mbar_test_wait(full_u(slot), ph) || wait_bar(full_u(slot), ph, p.err, p.limit_ns));
          if (!okm) break;
          if (me == 0 && lane == 0 && q == kc) HCGR_STAMP(27);
          tc_fence_after();
          const uint32_t a = ubase + slot * g.slot_u + tu * TILE, bq = hbase + q * Nu * 128;
          if (elect_one()) {
#pragma unroll 1
            for (int ks = 0; ks < 4; ++ks)
              umma_bf16(d, desc_sw128(a + ks * 32), desc_sw128(bq + ks * 32), idesc,
                        (q >= g.ncu || ks) ? 1u : 0u);
            umma_commit(free_u(slot));
            if (me == 0 && q == kc) HCGR_STAMP(28);
          }
          __syncwarp();
        }
        if (me == 0 && lane == 0) HCGR_STAMP(15);
        if (!okm && lane == 0) *s_mma_ok = 0;
        if (elect_one()) umma_commit(barG);
        __syncwarp();
      } else if (warp == 0) {
#pragma unroll 1
        for (int q = pre_u; q < nub; ++q) {
          const int slot = q % g.nsl_u;
          if (!__all_sync(0xffffffffu, wait_bar(free_u(slot), ((q / g.nsl_u) - 1) & 1, p.err, p.limit_ns)))
            break;
          if (lane == 0) issue_u(q);
          __syncwarp();
          ++issued_u;
        }
      }
      bool got = __all_sync(0xffffffffu, wait_bar(barG, 0, p.err, p.limit_ns));
      if (tid == 0) HCGR_STAMP(31);
      tc_fence_after();
      ok = __syncthreads_and(got && *s_mma_ok != 0);
      if (tid == 0) HCGR_STAMP(10);
      if (ok) {
        const int q4 = warp & 3, grp = warp >> 2;
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q4) << 16);
        const int nmc = Nu / 8;
        const int ncopy = min(g.ncu, nub);   // issuers' accumulator copies that hold a chunk
#pragma unroll 1
        for (int item = grp; item < g.ntu * nmc; item += NW / 4) {
          const int tu = item / nmc, m0 = (item - tu * nmc) * 8;
          const int i = tu * 128 + 32 * q4 + lane;               // row (stream, channel)
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = 0.f;
#pragma unroll 1
          for (int k = 0; k < ncopy; k += 2) {
            uint32_t v0[8], v1[8];
            if (k + 1 < ncopy) {
              tmem_ld8x2_wait(tl + (k * g.ntu + tu) * Nu + m0, tl + ((k + 1) * g.ntu + tu) * Nu + m0, v0, v1);
#pragma unroll
              for (int e = 0; e < 8; ++e) v[e] += __uint_as_float(v0[e]) + __uint_as_float(v1[e]);
            } else {
              tmem_ld8_wait(tl + (k * g.ntu + tu) * Nu + m0, v0);
#pragma unroll
              for (int e = 0; e < 8; ++e) v[e] += __uint_as_float(v0[e]);
            }
          }
          if (i < g.rows_u) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (m0 + e < M) s_g[(m0 + e) * g.rows_u + i] = sigmoid_fast(v[e]);
          }
        }
        HCGR_STAMP_MAX(21);
        __syncthreads();
        // a thread takes a channel pair of one token (nc, nc_max and cp0 are
        // even): paired shared-memory loads and one 4-byte store of x
        const int npr = nc / 2;
#pragma unroll 1
        for (int i = tid; i < M * npr; i += NT) {
          const int m = i / npr, cc = 2 * (i - m * npr), ch = cp0 + cc;
          const uint32_t yp = has_y ? *reinterpret_cast<const uint32_t*>(s_x3y + m * g.nc_max + cc) : 0u;
          float sum0 = 0.f, sum1 = 0.f;
#pragma unroll 4
          for (int ss = 0; ss < HC; ++ss) {
            const uint32_t rp = *reinterpret_cast<const uint32_t*>(s_x3r + (m * HC + ss) * g.nc_max + cc);
            const uint32_t wp = *reinterpret_cast<const uint32_t*>(s_x3w + ss * g.nc_max + cc);
            const float2 gp = *reinterpret_cast<const float2*>(s_g + m * g.rows_u + ss * g.nc_max + cc);
            const float iw = s_iw[m * HC + ss], rr = s_rr[m * HC + ss];
            float r0 = lo_bf16(rp), r1 = hi_bf16(rp);
            if (has_y) {
              r0 = bf16_to_f32(f32_to_bf16(fmaf(lo_bf16(yp), iw, r0)));
              r1 = bf16_to_f32(f32_to_bf16(fmaf(hi_bf16(yp), iw, r1)));
            }
            sum0 = fmaf(gp.x, r0 * rr * (1.0f + lo_bf16(wp)), sum0);
            sum1 = fmaf(gp.y, r1 * rr * (1.0f + hi_bf16(wp)), sum1);
          }
          *reinterpret_cast<uint32_t*>(c.x + static_cast<int64_t>(m) * HS + ch) =
              pack2(sum0 * inv_hc, sum1 * inv_hc);
        }
        HCGR_STAMP_MAX(22);
      }
    }
    if (tid == 0) HCGR_STAMP(11);
    // Off the critical path: empty the reduce-scatter blocks this CTA read
    // (when a wait failed instead, hc_gr_check resets them) and this CTA's
    // share of the all-gather copy the next call uses.
    if (red_done) {
#pragma unroll 1
      for (int j = u_idx; j < g.nred; j += g.Gu) {
        uint4* blk = reinterpret_cast<uint4*>(p.xred + static_cast<size_t>(j) * g.Gd * g.row);
#pragma unroll 1
        for (int i = tid; i < g.Gd * g.row / 4; i += NT) blk[i] = make_uint4(XEMPTY, XEMPTY, XEMPTY, XEMPTY);
      }
    }
    {
      uint4* nxt = reinterpret_cast<uint4*>(p.xgat + static_cast<size_t>(par ^ 1u) * p.gat_words);
      const int nq = p.gat_words / 4;
      const int per = (nq + g.Gu - 1) / g.Gu;
#pragma unroll 1
      for (int i = u_idx * per + tid; i < min(nq, (u_idx + 1) * per); i += NT)
        nxt[i] = make_uint4(XEMPTY, XEMPTY, XEMPTY, XEMPTY);
    }
  }

  // Teardown: every copy this CTA issued lands and every MMA it issued
  // completes (outstanding only after a failed wait: otherwise every box was
  // consumed and every commit waited for), then TMEM is released.
  if (__syncthreads_or(!ok) && warp == 0) {
#pragma unroll 1
    for (int i = max(0, issued_w - g.nsl_w); i < issued_w; ++i)
      drain_bar(full_w(i % g.nsl_w), (i / g.nsl_w) & 1, limit);
#pragma unroll 1
    for (int q = max(0, issued_u - g.nsl_u); q < issued_u; ++q)
      drain_bar(full_u(q % g.nsl_u), (q / g.nsl_u) & 1, limit);
    if (down_issued) drain_bar(barD, 0, limit);
    if (up_issued) drain_bar(barG, 0, limit);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 3) {
    tc_fence_after();
    tmem_dealloc(*s_tmem, tmem_cols);
  }
#ifdef HCGR_TRACE
  if (tid == 0) HCGR_STAMP(12);
  __syncthreads();
  if (tid < TRACE_SLOTS) g_trace[blockIdx.x * TRACE_SLOTS + tid] = s_stamp[tid];
#endif
}

Call shape_call(int64_t M, int HC, int HS, int r) {
  Call c{};
  c.M = M;
  c.HC = HC;
  c.HS = HS;
  c.r = r;
  c.K = HC * HS;
  c.n_out = r + HC;
  return c;
}

}  // namespace

size_t decode_xred_words(const Device& dev, int64_t M, int HC, int HS, int r) {
  Geom g;
  if (!make_geom(shape_call(M, HC, HS, r), dev, g)) return 0;
  return static_cast<size_t>(g.nred) * g.Gd * g.row;
}

size_t decode_xgat_words(int n_out_max) {
  // r / 2 + HC <= r + HC: every shape a handle accepts fits
  return static_cast<size_t>(DECODE_MAX_M) * round_up(n_out_max, 4);
}

cudaError_t launch_decode(const Call& c, const Workspace& ws, const Device& dev,
                          cudaStream_t stream) {
  Params prm;
  prm.c = c;
  prm.xred = ws.xred;
  prm.xgat = ws.xgat;
  prm.gat_words = static_cast<int>(ws.xgat_words);
  prm.ticket = ws.ticket;
  prm.err = ws.err;
  prm.limit_ns = c.debug_fault ? 50ull * 1000 * 1000 : 1000ull * 1000 * 1000;
  if (!make_geom(c, dev, prm.g)) return cudaErrorNotSupported;
  const Geom& g = prm.g;
  if (static_cast<size_t>(g.nred) * g.Gd * g.row > ws.xred_words ||
      static_cast<size_t>(c.M) * g.L2w > ws.xgat_words || ws.xgat_words % 4 != 0)
    return cudaErrorNotSupported;
  const uint64_t wstr[2] = {static_cast<uint64_t>(c.HS) * 2, static_cast<uint64_t>(c.K) * 2};
  const uint64_t dw[3] = {static_cast<uint64_t>(c.HS), static_cast<uint64_t>(c.HC),
                          static_cast<uint64_t>(g.rows_w)};
  const uint32_t bw[3] = {64u, 1u, 128u};
  const uint32_t bwt[3] = {64u, 1u, static_cast<uint32_t>(g.tail > 0 ? g.tail : 8)};
  const uint64_t dwi[3] = {static_cast<uint64_t>(c.HS), static_cast<uint64_t>(c.HC),
                           static_cast<uint64_t>(c.HC)};
  const uint32_t bwi[3] = {64u, 1u, static_cast<uint32_t>(c.HC)};
  const uint64_t dwu[3] = {static_cast<uint64_t>(c.r), static_cast<uint64_t>(c.HS),
                           static_cast<uint64_t>(c.HC)};
  const uint64_t swu[2] = {static_cast<uint64_t>(c.r) * 2, static_cast<uint64_t>(c.HS) * c.r * 2};
  const uint32_t bwu[3] = {64u, static_cast<uint32_t>(g.nc_max), static_cast<uint32_t>(c.HC)};
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  if (!make_tmap_bf16(&prm.tm_w, c.Wd, 3, dw, wstr, bw, SW) ||
      !make_tmap_bf16(&prm.tm_wt, c.Wd, 3, dw, wstr, bwt, SW) ||
      !make_tmap_bf16(&prm.tm_wi, c.Wi, 3, dwi, wstr, bwi, SW) ||
      !make_tmap_bf16(&prm.tm_wu, c.Wu, 3, dwu, swu, bwu, SW))
    return cudaErrorNotSupported;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(decode_kernel), SMEM_ALLOC, dev.id,
                                  attr_done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.G);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = g.total + 1024;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (c.pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  } else {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel, prm);
}

}  // namespace hcgr

#ifdef HCGR_TRACE
// Copies the phase stamps of the last traced decode launch (n <= MAX_GRID *
// TRACE_SLOTS values, [CTA][TRACE_SLOTS] in ns of %globaltimer) to host memory, then clears the
// array, so that a slot no CTA of the next launch passes reads 0.
extern "C" int hc_gr_trace_read(unsigned long long* host, int n) {
  const size_t cap = sizeof(hcgr::g_trace) / sizeof(unsigned long long);
  if (n < 0 || static_cast<size_t>(n) > cap) return static_cast<int>(cudaErrorInvalidValue);
  cudaError_t e = cudaMemcpyFromSymbol(host, hcgr::g_trace, n * sizeof(unsigned long long));
  if (e != cudaSuccess) return static_cast<int>(e);
  void* dev = nullptr;
  e = cudaGetSymbolAddress(&dev, hcgr::g_trace);
  if (e == cudaSuccess) e = cudaMemset(dev, 0, sizeof(hcgr::g_trace));
  return static_cast<int>(e);
}
#endif

// COMBINE on its own (aiter PR #5913, "Technical Details", the (COMBINE)
// bullet; the combine-only entry point of "Behavior and intent"):
//
//   R2[m, s, c] = bf16(R[m, s, c] + y[m, c] * 2 sigmoid(inj[m, s] / HC))
//
// for layers that run COMBINE apart from the mix.  The kernel streams R in,
// R2 out and y once per stream (from L2 after the first), so it is bound by
// HBM bandwidth: 4K + 2HS + 4HC bytes per token.  One thread handles one
// 16-byte chunk (8 channels) of one stream of one token; consecutive threads
// take consecutive chunks, so every warp access is a contiguous 512 bytes.
// The combine weight and the rounding are the fused kernels' own
// (combine_weight, fmaf, round-to-nearest-even), so R2 agrees with theirs
// bit for bit.
#include "hc_gr_internal.cuh"

namespace hcgr {
namespace {

constexpr int CB_THREADS = 256;
constexpr int CB_BATCH = 4;          // units whose loads are in flight together per thread
constexpr int CB_BLOCKS_PER_SM = 4;  // resident at <= 64 registers a thread

struct CombineParams {
  const bf16_t* R;
  const bf16_t* y;
  const float* inj;
  bf16_t* R2;
  int64_t ld_inj;
  int64_t units;     // M * HC * (HS / 8)
  int HC, n8;        // n8 = HS / 8 chunks per stream row
};

__global__ void __launch_bounds__(CB_THREADS, CB_BLOCKS_PER_SM) combine_kernel(const CombineParams p) {
  const float inv_hc = 1.0f / static_cast<float>(p.HC);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * CB_THREADS;
  const int64_t per_token = static_cast<int64_t>(p.HC) * p.n8;
#pragma unroll 1
  for (int64_t u0 = static_cast<int64_t>(blockIdx.x) * CB_THREADS + threadIdx.x; u0 < p.units;
       u0 += stride * CB_BATCH) {
    uint4 rv[CB_BATCH], yv[CB_BATCH];
    float iw[CB_BATCH];
    // all loads of the batch first, so that they are in flight together
#pragma unroll
    for (int b = 0; b < CB_BATCH; ++b) {
      const int64_t u = u0 + b * stride;
      if (u < p.units) {
        const int64_t m = u / per_token;
        const int64_t rem = u - m * per_token;
        const int s = static_cast<int>(rem / p.n8);
        const int c8 = static_cast<int>(rem - static_cast<int64_t>(s) * p.n8);
        rv[b] = __ldcs(reinterpret_cast<const uint4*>(p.R) + u);
        yv[b] = __ldg(reinterpret_cast<const uint4*>(p.y) + m * p.n8 + c8);
        iw[b] = __ldg(p.inj + m * p.ld_inj + s);
      }
    }
#pragma unroll
    for (int b = 0; b < CB_BATCH; ++b) {
      const int64_t u = u0 + b * stride;
      if (u < p.units) {
        const float w = combine_weight(iw[b], inv_hc);
        float r[8], yy[8];
        unpack8(rv[b], r);
        unpack8(yv[b], yy);
        uint4 o;
        o.x = pack2(fmaf(yy[0], w, r[0]), fmaf(yy[1], w, r[1]));
        o.y = pack2(fmaf(yy[2], w, r[2]), fmaf(yy[3], w, r[3]));
        o.z = pack2(fmaf(yy[4], w, r[4]), fmaf(yy[5], w, r[5]));
        o.w = pack2(fmaf(yy[6], w, r[6]), fmaf(yy[7], w, r[7]));
        __stcs(reinterpret_cast<uint4*>(p.R2) + u, o);
      }
    }
  }
}

}  // namespace

cudaError_t launch_combine(int64_t M, int HC, int HS, const bf16_t* R, const bf16_t* y,
                           const float* inj, int64_t ld_inj, bf16_t* R2, const Device& dev,
                           cudaStream_t stream) {
  CombineParams p;
  p.R = R;
  p.y = y;
  p.inj = inj;
  p.R2 = R2;
  p.ld_inj = ld_inj;
  p.HC = HC;
  p.n8 = HS / 8;
  p.units = M * HC * static_cast<int64_t>(p.n8);
  const int64_t need = (p.units + CB_THREADS - 1) / CB_THREADS;
  const int64_t cap = static_cast<int64_t>(dev.sms > 0 ? dev.sms : 1) * CB_BLOCKS_PER_SM;
  const int grid = static_cast<int>(need < cap ? need : cap);
  combine_kernel<<<grid, CB_THREADS, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace hcgr

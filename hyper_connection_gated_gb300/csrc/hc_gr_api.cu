// C ABI of the HC gated residual: argument validation, the handle's
// workspace, the M-based dispatch between the decode and prefill paths, and
// device status reporting.  The operation and the layouts are documented in
// include/hc_gr.h.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>

#include "hc_gr_internal.cuh"

struct hc_gr_ctx {
  hcgr::Device dev;
  hcgr::Workspace ws;
  int64_t max_M = 0;
  int K_max = 0;
  int n_out_max = 0;
  int HC_max = 0;
  int r_max = 0;
  char last_cuda[256] = {0};
};

namespace {

using hcgr::bf16_t;

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int id) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != id) cudaSetDevice(id);
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

int cuda_fail(hc_gr_ctx* h, cudaError_t e) {
  if (h) std::snprintf(h->last_cuda, sizeof(h->last_cuda), "%s", cudaGetErrorString(e));
  return HC_GR_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
};
Range span(const void* p, int64_t bytes) {   // NULL: the empty range
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return p ? Range{lo, lo + static_cast<uintptr_t>(bytes)} : Range{0, 0};
}
bool overlap(const Range& a, const Range& b) {
  return a.lo < b.hi && b.lo < a.hi && a.hi > a.lo && b.hi > b.lo;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Ticket and status word to zero, every exchange word to the empty marker.
cudaError_t reset_control(const hcgr::Workspace& ws, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(ws.ticket, 0, hcgr::CTL_BYTES, s);
  if (e == cudaSuccess && ws.xred_words)
    e = cudaMemsetAsync(ws.xred, 0xff, ws.xred_words * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws.xgat, 0xff, 2 * ws.xgat_words * 4, s);
  return e;
}

}  // namespace

extern "C" {

const char* hc_gr_strerror(int status) {
  switch (status) {
    case HC_GR_OK: return "ok";
    case HC_GR_ERR_INVALID_ARG: return "invalid argument";
    case HC_GR_ERR_UNSUPPORTED: return "unsupported shape or device";
    case HC_GR_ERR_ALIAS: return "an output overlaps another output or an input";
    case HC_GR_ERR_CUDA: return "CUDA error";
    case HC_GR_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

const char* hc_gr_last_cuda_error(hc_gr_handle h) { return h ? h->last_cuda : ""; }

int hc_gr_create(hc_gr_handle* out, int device, int64_t max_M, int HC, int HS, int r) {
  if (!out) return HC_GR_ERR_INVALID_ARG;
  *out = nullptr;
  if (max_M < 1 || HC < 1 || HS < 1 || r < 1 || device < 0) return HC_GR_ERR_INVALID_ARG;
  if (HS % 8 != 0 || r % 8 != 0) return HC_GR_ERR_UNSUPPORTED;
  if (max_M > HC_GR_MAX_TOKENS || static_cast<int64_t>(HC) * HS > HC_GR_MAX_WIDTH)
    return HC_GR_ERR_UNSUPPORTED;
  hc_gr_ctx* h = new (std::nothrow) hc_gr_ctx();
  if (!h) return HC_GR_ERR_CUDA;
  DeviceGuard guard(device);
  cudaDeviceProp prop;
  cudaError_t e = cudaGetDeviceProperties(&prop, device);
  if (e != cudaSuccess) {
    delete h;
    return HC_GR_ERR_CUDA;
  }
  if (!(prop.major == 10 && prop.minor == 3)) {
    delete h;
    return HC_GR_ERR_UNSUPPORTED;
  }
  h->dev.id = device;
  h->dev.sms = prop.multiProcessorCount;
  h->dev.smem_optin = static_cast<int>(prop.sharedMemPerBlockOptin);
  h->dev.l2_bytes = prop.l2CacheSize;
  h->max_M = max_M;
  h->K_max = HC * HS;
  h->HC_max = HC;
  h->r_max = r;
  h->n_out_max = r + HC;

  // one allocation: [ticket/err | reduce-scatter words | all-gather words (two
  // copies) | lora | prefill scratch]
  size_t xred_words = 0;
  for (int64_t M = 1; M <= std::min<int64_t>(max_M, hcgr::DECODE_MAX_M); ++M)
    xred_words = std::max(xred_words, hcgr::decode_xred_words(h->dev, M, HC, HS, r));
  const size_t xgat_words = hcgr::decode_xgat_words(r + HC);
  const size_t lora_f = static_cast<size_t>(max_M) * (r + HC);
  size_t off = 0;
  const size_t off_ctl = off;    off += hcgr::CTL_BYTES;
  const size_t off_xred = off;   off = align_up(off + xred_words * 4, 256);
  const size_t off_xgat = off;   off = align_up(off + 2 * xgat_words * 4, 256);
  const size_t off_lora = off;   off = align_up(off + lora_f * 4, 256);
  const size_t off_pre = off;    off = align_up(off + hcgr::prefill_ws_bytes(max_M, HC, HS, r), 256);
  void* base = nullptr;
  e = cudaMalloc(&base, off);
  if (e != cudaSuccess) {
    cudaGetLastError();   // leave no stale error for the caller's next CUDA call
    delete h;
    return HC_GR_ERR_CUDA;
  }
  unsigned char* b = static_cast<unsigned char*>(base);
  h->ws.base = base;
  h->ws.bytes = off;
  h->ws.ticket = reinterpret_cast<unsigned long long*>(b + off_ctl);
  h->ws.err = reinterpret_cast<int*>(b + off_ctl + hcgr::MAX_GRID * 8);
  h->ws.xred = reinterpret_cast<uint32_t*>(b + off_xred);
  h->ws.xred_words = xred_words;
  h->ws.xgat = reinterpret_cast<uint32_t*>(b + off_xgat);
  h->ws.xgat_words = xgat_words;
  h->ws.lora = reinterpret_cast<float*>(b + off_lora);
  h->ws.k1_part = reinterpret_cast<float*>(b + off_pre);
  h->ws.prefill_bytes = hcgr::prefill_ws_bytes(max_M, HC, HS, r);
  e = reset_control(h->ws, nullptr);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(base);
    delete h;
    return HC_GR_ERR_CUDA;
  }
  *out = h;
  return HC_GR_OK;
}

int hc_gr_destroy(hc_gr_handle h) {
  if (!h) return HC_GR_OK;
  int st = HC_GR_OK;
  {
    DeviceGuard guard(h->dev.id);
    cudaDeviceSynchronize();
    if (h->ws.base && cudaFree(h->ws.base) != cudaSuccess) st = HC_GR_ERR_CUDA;
  }
  delete h;
  return st;
}

int hc_gr_forward_ex(hc_gr_handle h, const hc_gr_args* a, struct CUstream_st* stream) {
  if (!h || !a) return HC_GR_ERR_INVALID_ARG;
  const int64_t M = a->M;
  const int HC = a->HC, HS = a->HS, r = a->r;
  if (M < 1 || HC < 1 || HS < 1 || r < 1) return HC_GR_ERR_INVALID_ARG;
  if (!(std::isfinite(a->eps) && a->eps > 0.0f)) return HC_GR_ERR_INVALID_ARG;
  if (a->force_path < HC_GR_PATH_AUTO || a->force_path > HC_GR_PATH_PREFILL)
    return HC_GR_ERR_INVALID_ARG;
  const int64_t ld_inj = a->ld_inj == 0 ? HC : a->ld_inj;
  if (ld_inj < HC) return HC_GR_ERR_INVALID_ARG;
  const bool merged = a->Wdi != nullptr;
  // y, inj and R2 all NULL: the mix alone (R is the combined residual)
  const bool mix_only = !a->y && !a->inj && !a->R2;
  if (!mix_only && (!a->y || !a->inj || !a->R2)) return HC_GR_ERR_INVALID_ARG;
  if (!a->R || !a->Wnorm || !a->Wu || !a->rrms || !a->inj_next || !a->x)
    return HC_GR_ERR_INVALID_ARG;
  if (!merged && (!a->Wd || !a->Wi)) return HC_GR_ERR_INVALID_ARG;
  const void* p16[] = {a->R, a->y, a->Wnorm, a->Wu, a->R2, a->x, a->lora,
                       merged ? a->Wdi : a->Wd, merged ? a->Wdi : a->Wi};
  for (const void* p : p16)
    if (!aligned(p, 16)) return HC_GR_ERR_INVALID_ARG;
  const void* p4[] = {a->inj, a->rrms, a->inj_next};
  for (const void* p : p4)
    if (!aligned(p, 4)) return HC_GR_ERR_INVALID_ARG;
  if (HS % 8 != 0 || r % 8 != 0) return HC_GR_ERR_UNSUPPORTED;
  const int64_t K = static_cast<int64_t>(HC) * HS;
  if (M > HC_GR_MAX_TOKENS || K > HC_GR_MAX_WIDTH) return HC_GR_ERR_UNSUPPORTED;
  if (M > h->max_M || K > h->K_max || r + HC > h->n_out_max) return HC_GR_ERR_UNSUPPORTED;
  if (merged && a->n_pad < r + HC) return HC_GR_ERR_UNSUPPORTED;
  if (a->force_path == HC_GR_PATH_DECODE && M > hcgr::DECODE_MAX_M) return HC_GR_ERR_UNSUPPORTED;

  // outputs must not overlap each other or any input
  const Range outs[] = {span(a->R2, M * K * 2), span(a->rrms, M * HC * 4),
                        span(a->inj_next, M * HC * 4), span(a->x, M * HS * 2),
                        a->lora ? span(a->lora, M * r * 4) : Range{0, 0}};
  const Range ins[] = {span(a->R, M * K * 2), span(a->y, M * HS * 2),
                       span(a->inj, ((M - 1) * ld_inj + HC) * 4),
                       span(a->Wnorm, (a->wnorm_hs ? HS : K) * 2),
                       span(a->Wu, K * r * 2),
                       merged ? span(a->Wdi, static_cast<int64_t>(a->n_pad) * K * 2)
                              : span(a->Wd, static_cast<int64_t>(r) * K * 2),
                       merged ? Range{0, 0} : span(a->Wi, static_cast<int64_t>(HC) * K * 2)};
  const int nouts = sizeof(outs) / sizeof(outs[0]);
  for (int i = 0; i < nouts; ++i) {
    for (int j = i + 1; j < nouts; ++j)
      if (overlap(outs[i], outs[j])) return HC_GR_ERR_ALIAS;
    for (const Range& in : ins)
      if (overlap(outs[i], in)) return HC_GR_ERR_ALIAS;
  }

  hcgr::Call c;
  c.M = M;
  c.HC = HC;
  c.HS = HS;
  c.r = r;
  c.K = static_cast<int>(K);
  c.n_out = r + HC;
  c.eps = a->eps;
  c.R = static_cast<const bf16_t*>(a->R);
  c.y = static_cast<const bf16_t*>(a->y);
  c.inj = a->inj;
  c.ld_inj = ld_inj;
  c.Wnorm = static_cast<const bf16_t*>(a->Wnorm);
  c.ld_wnorm = a->wnorm_hs ? 0 : HS;
  if (merged) {
    c.Wd = static_cast<const bf16_t*>(a->Wdi);
    c.Wi = c.Wd + static_cast<int64_t>(r) * K;
  } else {
    c.Wd = static_cast<const bf16_t*>(a->Wd);
    c.Wi = static_cast<const bf16_t*>(a->Wi);
  }
  c.fold = a->fold_w ? 1 : 0;
  c.Wu = static_cast<const bf16_t*>(a->Wu);
  c.R2 = static_cast<bf16_t*>(a->R2);
  c.rrms = a->rrms;
  c.inj_next = a->inj_next;
  c.x = static_cast<bf16_t*>(a->x);
  c.lora = a->lora ? a->lora : h->ws.lora;
  c.debug_fault = a->debug_fault;
  c.pdl = a->pdl ? 1 : 0;

  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceGuard guard(h->dev.id);
  // M-based dispatch (the page's split between a skinny decode path and the
  // tiled kernels, "Behavior and intent"): the weight-streaming decode kernel
  // up to the measured crossover (M <= DECODE_MAX_M and M * K <=
  // DECODE_AUTO_MAX_MK), the tensor-core prefill kernels above it (and for
  // shapes the decode kernel's plan cannot hold).
  cudaError_t e;
  if (a->force_path == HC_GR_PATH_DECODE) {
    e = hcgr::launch_decode(c, h->ws, h->dev, s);
  } else if (a->force_path == HC_GR_PATH_PREFILL || M > hcgr::DECODE_MAX_M ||
             M * c.K > hcgr::DECODE_AUTO_MAX_MK) {
    e = hcgr::launch_prefill(c, h->ws, h->dev, s);
  } else {
    e = hcgr::launch_decode(c, h->ws, h->dev, s);
    if (e == cudaErrorNotSupported) e = hcgr::launch_prefill(c, h->ws, h->dev, s);
  }
  if (e == cudaErrorNotSupported) return HC_GR_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return cuda_fail(h, e);
  return HC_GR_OK;
}

int hc_gr_combine(hc_gr_handle h, int64_t M, int HC, int HS, const void* R, const void* y,
                  const float* inj, int64_t ld_inj, void* R2, struct CUstream_st* stream) {
  if (!h || !R || !y || !inj || !R2) return HC_GR_ERR_INVALID_ARG;
  if (M < 1 || HC < 1 || HS < 1) return HC_GR_ERR_INVALID_ARG;
  if (ld_inj == 0) ld_inj = HC;
  if (ld_inj < HC) return HC_GR_ERR_INVALID_ARG;
  if (!aligned(R, 16) || !aligned(y, 16) || !aligned(R2, 16) || !aligned(inj, 4))
    return HC_GR_ERR_INVALID_ARG;
  if (HS % 8 != 0) return HC_GR_ERR_UNSUPPORTED;
  const int64_t K = static_cast<int64_t>(HC) * HS;
  if (M > HC_GR_MAX_TOKENS || K > HC_GR_MAX_WIDTH) return HC_GR_ERR_UNSUPPORTED;
  const Range out = span(R2, M * K * 2);
  if (overlap(out, span(R, M * K * 2)) || overlap(out, span(y, M * HS * 2)) ||
      overlap(out, span(inj, ((M - 1) * ld_inj + HC) * 4)))
    return HC_GR_ERR_ALIAS;
  DeviceGuard guard(h->dev.id);
  const cudaError_t e = hcgr::launch_combine(
      M, HC, HS, static_cast<const hcgr::bf16_t*>(R), static_cast<const hcgr::bf16_t*>(y), inj,
      ld_inj, static_cast<hcgr::bf16_t*>(R2), h->dev, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e);
  return HC_GR_OK;
}

int hc_gr_mix(hc_gr_handle h, int64_t M, int HC, int HS, int r, float eps, const void* R,
              const void* Wnorm, const void* Wd, const void* Wi, const void* Wu, float* rrms,
              float* inj_next, void* x, float* lora, struct CUstream_st* stream) {
  hc_gr_args a;
  std::memset(&a, 0, sizeof(a));
  a.M = M;
  a.HC = HC;
  a.HS = HS;
  a.r = r;
  a.eps = eps;
  a.R = R;
  a.Wnorm = Wnorm;
  a.Wd = Wd;
  a.Wi = Wi;
  a.Wu = Wu;
  a.rrms = rrms;
  a.inj_next = inj_next;
  a.x = x;
  a.lora = lora;
  return hc_gr_forward_ex(h, &a, stream);
}

int hc_gr_forward(hc_gr_handle h, int64_t M, int HC, int HS, int r, float eps, const void* R,
                  const void* y, const float* inj, const void* Wnorm, const void* Wd,
                  const void* Wi, const void* Wu, void* R2, float* rrms, float* inj_next,
                  void* x, float* lora, struct CUstream_st* stream) {
  hc_gr_args a;
  std::memset(&a, 0, sizeof(a));
  a.M = M;
  a.HC = HC;
  a.HS = HS;
  a.r = r;
  a.eps = eps;
  a.R = R;
  a.y = y;
  a.inj = inj;
  a.Wnorm = Wnorm;
  a.Wd = Wd;
  a.Wi = Wi;
  a.Wu = Wu;
  a.R2 = R2;
  a.rrms = rrms;
  a.inj_next = inj_next;
  a.x = x;
  a.lora = lora;
  return hc_gr_forward_ex(h, &a, stream);
}

int hc_gr_check(hc_gr_handle h, struct CUstream_st* stream) {
  if (!h) return HC_GR_ERR_INVALID_ARG;
  DeviceGuard guard(h->dev.id);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(h, e);
  int dev_status = 0;
  e = cudaMemcpy(&dev_status, h->ws.err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(h, e);
  if (dev_status == hcgr::DEV_OK) return HC_GR_OK;
  // clear the status, the ticket and the exchange buffers (a failed call can
  // leave values in them) so the handle can be used again
  e = reset_control(h->ws, s);
  if (e != cudaSuccess) return cuda_fail(h, e);
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(h, e);
  return HC_GR_ERR_TIMEOUT;
}

}  // extern "C"

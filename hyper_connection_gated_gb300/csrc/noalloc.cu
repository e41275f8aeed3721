// hc_gr_forward_noalloc: the decode kernel with its scratch memory in a
// fixed device array owned by the library, for callers that must not
// allocate device memory on their call path (see include/hc_gr.h).
//
// The scratch array is a file-scope __device__ array, so every GPU that loads
// the library holds it until the process exits.  In host code its name is
// only a host-side stand-in, never a device address: the device address is
// obtained once per device with cudaGetSymbolAddress (with that device
// current) and passed to the kernel.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "hc_gr_internal.cuh"

namespace hcgr {
namespace {

// Limits of this entry point: M <= NOALLOC_MAX_M tokens and r + HC <=
// NOALLOC_MAX_NOUT; everything else as for hc_gr_forward's decode path.
constexpr int NOALLOC_MAX_M = 8;
constexpr int NOALLOC_MAX_NOUT = 336;
constexpr size_t NOALLOC_SCRATCH_BYTES = 4u << 20;   // 4 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
struct PerDevice {
  bool ready = false;
  unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch
  Device dev;
};
PerDevice g_dev[MAX_DEVICES];
std::mutex g_mu;

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// Carve the scratch array into the decode kernel's workspace for a call that
// needs xred_words reduce-scatter words: [ticket/status | reduce-scatter |
// all-gather (two copies) | lora].
bool carve(unsigned char* base, size_t xred_words, Workspace& ws) {
  ws.base = base;
  ws.ticket = reinterpret_cast<unsigned long long*>(base);
  ws.err = reinterpret_cast<int*>(base + MAX_GRID * 8);
  size_t off = align256(CTL_BYTES);
  ws.xred = reinterpret_cast<uint32_t*>(base + off);
  ws.xred_words = xred_words;
  off = align256(off + xred_words * 4);
  ws.xgat = reinterpret_cast<uint32_t*>(base + off);
  ws.xgat_words = decode_xgat_words(NOALLOC_MAX_NOUT);
  off = align256(off + 2 * ws.xgat_words * 4);
  ws.lora = reinterpret_cast<float*>(base + off);
  off = align256(off + static_cast<size_t>(NOALLOC_MAX_M) * NOALLOC_MAX_NOUT * 4);
  ws.bytes = off;
  ws.k1_part = nullptr;
  ws.prefill_bytes = 0;
  return off <= NOALLOC_SCRATCH_BYTES;
}

bool overlap(uintptr_t a, size_t na, uintptr_t b, size_t nb) {
  return na && nb && a < b + nb && b < a + na;
}

}  // namespace
}  // namespace hcgr

extern "C" int hc_gr_forward_noalloc(int64_t M, int HC, int HS, int r, float eps, const void* R,
                                     const void* y, const float* inj, const void* Wnorm,
                                     const void* Wd, const void* Wi, const void* Wu, void* R2,
                                     float* rrms, float* inj_next, void* x, float* lora,
                                     struct CUstream_st* stream) {
  using namespace hcgr;
  if (M < 1 || HC < 1 || HS < 1 || r < 1 || !(std::isfinite(eps) && eps > 0.0f))
    return HC_GR_ERR_INVALID_ARG;
  if (!R || !y || !inj || !Wnorm || !Wd || !Wi || !Wu || !R2 || !rrms || !inj_next || !x)
    return HC_GR_ERR_INVALID_ARG;
  const void* p16[] = {R, y, Wnorm, Wd, Wi, Wu, R2, x, lora};
  for (const void* p : p16)
    if (reinterpret_cast<uintptr_t>(p) % 16) return HC_GR_ERR_INVALID_ARG;
  const void* p4[] = {inj, rrms, inj_next};
  for (const void* p : p4)
    if (reinterpret_cast<uintptr_t>(p) % 4) return HC_GR_ERR_INVALID_ARG;
  if (HS % 8 || r % 8) return HC_GR_ERR_UNSUPPORTED;
  if (M > NOALLOC_MAX_M || r + HC > NOALLOC_MAX_NOUT) return HC_GR_ERR_UNSUPPORTED;
  const int64_t K = static_cast<int64_t>(HC) * HS;
  const uintptr_t outs[5] = {reinterpret_cast<uintptr_t>(R2), reinterpret_cast<uintptr_t>(rrms),
                             reinterpret_cast<uintptr_t>(inj_next), reinterpret_cast<uintptr_t>(x),
                             reinterpret_cast<uintptr_t>(lora)};
  const size_t nouts[5] = {static_cast<size_t>(M * K * 2), static_cast<size_t>(M * HC * 4),
                           static_cast<size_t>(M * HC * 4), static_cast<size_t>(M * HS * 2),
                           lora ? static_cast<size_t>(M * r * 4) : 0};
  const uintptr_t ins[7] = {reinterpret_cast<uintptr_t>(R), reinterpret_cast<uintptr_t>(y),
                            reinterpret_cast<uintptr_t>(inj), reinterpret_cast<uintptr_t>(Wnorm),
                            reinterpret_cast<uintptr_t>(Wd), reinterpret_cast<uintptr_t>(Wi),
                            reinterpret_cast<uintptr_t>(Wu)};
  const size_t nins[7] = {static_cast<size_t>(M * K * 2), static_cast<size_t>(M * HS * 2),
                          static_cast<size_t>(M * HC * 4), static_cast<size_t>(K * 2),
                          static_cast<size_t>(r * K * 2), static_cast<size_t>(HC * K * 2),
                          static_cast<size_t>(K * r * 2)};
  for (int i = 0; i < 5; ++i) {
    for (int j = i + 1; j < 5; ++j)
      if (overlap(outs[i], nouts[i], outs[j], nouts[j])) return HC_GR_ERR_ALIAS;
    for (int j = 0; j < 7; ++j)
      if (overlap(outs[i], nouts[i], ins[j], nins[j])) return HC_GR_ERR_ALIAS;
  }

  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= MAX_DEVICES)
    return HC_GR_ERR_CUDA;
  PerDevice& pd = g_dev[device];
  {
    // once per device, with that device current: query it and resolve the
    // device address of the scratch array (its host-side name is not one)
    std::lock_guard<std::mutex> lock(g_mu);
    if (!pd.ready) {
      cudaDeviceProp prop;
      if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return HC_GR_ERR_CUDA;
      if (!(prop.major == 10 && prop.minor == 3)) return HC_GR_ERR_UNSUPPORTED;
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
        return HC_GR_ERR_CUDA;
      pd.scratch = static_cast<unsigned char*>(ptr);
      pd.dev.id = device;
      pd.dev.sms = prop.multiProcessorCount;
      pd.dev.smem_optin = static_cast<int>(prop.sharedMemPerBlockOptin);
      pd.dev.l2_bytes = prop.l2CacheSize;
      pd.ready = true;
    }
  }
  const size_t xred_words = decode_xred_words(pd.dev, M, HC, HS, r);
  Workspace ws;
  if (xred_words == 0 || !carve(pd.scratch, xred_words, ws)) return HC_GR_ERR_UNSUPPORTED;

  Call c;
  c.M = M;
  c.HC = HC;
  c.HS = HS;
  c.r = r;
  c.K = static_cast<int>(K);
  c.n_out = r + HC;
  c.eps = eps;
  c.R = static_cast<const bf16_t*>(R);
  c.y = static_cast<const bf16_t*>(y);
  c.inj = inj;
  c.ld_inj = HC;
  c.Wnorm = static_cast<const bf16_t*>(Wnorm);
  c.ld_wnorm = HS;
  c.Wd = static_cast<const bf16_t*>(Wd);
  c.Wi = static_cast<const bf16_t*>(Wi);
  c.fold = 0;
  c.Wu = static_cast<const bf16_t*>(Wu);
  c.R2 = static_cast<bf16_t*>(R2);
  c.rrms = rrms;
  c.inj_next = inj_next;
  c.x = static_cast<bf16_t*>(x);
  c.lora = lora ? lora : ws.lora;
  c.debug_fault = 0;
  c.pdl = 0;

  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The ticket starts at zero and every exchange word empty on every call
  // (the array keeps whatever the previous call left there, and a call that
  // timed out can leave values behind).  The status word is kept: a timeout
  // stays recorded until hc_gr_noalloc_check clears it.
  if (cudaMemsetAsync(ws.base, 0, MAX_GRID * 8, s) != cudaSuccess) return HC_GR_ERR_CUDA;
  const size_t xbytes = reinterpret_cast<unsigned char*>(ws.lora) -
                        reinterpret_cast<unsigned char*>(ws.xred);
  if (cudaMemsetAsync(ws.xred, 0xff, xbytes, s) != cudaSuccess) return HC_GR_ERR_CUDA;
  const cudaError_t e = launch_decode(c, ws, pd.dev, s);
  if (e == cudaErrorNotSupported) return HC_GR_ERR_UNSUPPORTED;
  return e == cudaSuccess ? HC_GR_OK : HC_GR_ERR_CUDA;
}

extern "C" int hc_gr_noalloc_check(struct CUstream_st* stream) {
  using namespace hcgr;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= MAX_DEVICES)
    return HC_GR_ERR_CUDA;
  unsigned char* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_dev[device].ready) scratch = g_dev[device].scratch;
  }
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return HC_GR_ERR_CUDA;
  if (!scratch) return HC_GR_OK;   // no call on this device yet
  int* err = reinterpret_cast<int*>(scratch + MAX_GRID * 8);
  int status = DEV_OK;
  if (cudaMemcpy(&status, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return HC_GR_ERR_CUDA;
  if (status == DEV_OK) return HC_GR_OK;
  if (cudaMemset(err, 0, sizeof(int)) != cudaSuccess) return HC_GR_ERR_CUDA;
  return HC_GR_ERR_TIMEOUT;
}

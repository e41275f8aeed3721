// Internal declarations shared by the HC-GR CUDA sources (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/hc_gr.h"

namespace hcgr {

using bf16_t = uint16_t;

// Device status word values (the handle's err word).
constexpr int DEV_OK = 0;
constexpr int DEV_TIMEOUT = 1;

// Workspace of a handle: all device memory the library owns.
struct Workspace {
  unsigned long long* ticket = nullptr;  // decode: call ticket (arrivals | epoch << 32)
  int* err = nullptr;         // device status word
  uint32_t* xred = nullptr;   // decode: reduce-scatter exchange words (empty = 0xffffffff)
  size_t xred_words = 0;
  uint32_t* xgat = nullptr;   // decode: all-gather words, two copies of xgat_words
  size_t xgat_words = 0;
  float* lora = nullptr;      // lora when the caller passes lora == NULL
  void* base = nullptr;       // single allocation holding everything above
  size_t bytes = 0;
  // prefill workspace
  float* k1_part = nullptr;   // prefill scratch: per-stream products, inject partials, h
  size_t prefill_bytes = 0;   // capacity of the prefill scratch
};

// Everything one forward call needs after validation.
struct Call {
  int64_t M;
  int HC, HS, r, K, n_out;
  float eps;
  const bf16_t* R;
  const bf16_t* y;    // NULL: mix only -- R holds the combined streams (R2 = R), inj unused
  const float* inj;
  int64_t ld_inj;
  const bf16_t* Wnorm;
  int64_t ld_wnorm;   // entries between two streams' Wnorm slices: HS, or 0 (one [HS] slice shared)
  const bf16_t* Wd;   // row n < r of the projection weight: Wd + n * K
  const bf16_t* Wi;   // row j < HC of the inject weight:   Wi + j * K
  int fold;
  const bf16_t* Wu;
  bf16_t* R2;         // NULL (mix only): not stored
  float* rrms;
  float* inj_next;
  bf16_t* x;
  float* lora;        // never NULL here (workspace substitute)
  int debug_fault;
  int pdl;            // decode: launched as a programmatic dependent of the previous kernel
};

struct Device {
  int id = 0;
  int sms = 0;
  int smem_optin = 0;
  int l2_bytes = 0;
};

// Raises a kernel's dynamic shared-memory limit on `device` (the current
// device).  The attribute belongs to the device, so it is set once per device:
// `done` holds one bit per device id below 64 (higher ids set it on every
// call).  Concurrent first calls may both set it, which is harmless.
inline cudaError_t smem_limit_once(const void* func, int bytes, int device,
                                   std::atomic<unsigned long long>& done) {
  const unsigned long long bit = device >= 0 && device < 64 ? 1ull << device : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Decode path (M <= DECODE_MAX_M): one persistent kernel.
constexpr int DECODE_MAX_M = 64;
// The M dispatch's threshold: the decode kernel while M <= DECODE_MAX_M and
// M * K <= DECODE_AUTO_MAX_MK, the prefill kernels above.  Measured on the
// GB300 (graph replay, weights from HBM, programmatic dependent launches):
// at HC=4, HS=2560, r=320 (K = 10240) decode takes 14.6 / 16.0 / 19.1 / 21.3 /
// 22.4 / 23.3 us at M = 24 / 32 / 40 / 48 / 56 / 64 against 23.1 - 23.6 us for
// prefill, so decode wins up to its 64-token limit; at HC=8, HS=4096, r=512
// (K = 32768) decode takes 38.3 / 41.9 / 49.9 us at M = 16 / 20 / 24 against
// 43.7 / 43.8 / 44.1 us, so the paths cross between 20 and 24 tokens.  Both
// crossovers sit at about the same M * K: the decode kernel's per-token work
// grows with the width K.
constexpr int64_t DECODE_AUTO_MAX_MK = 64LL * 10240;
constexpr int MAX_GRID = 256;            // largest prefill grid the scratch is sized for
constexpr int CTL_BYTES = MAX_GRID * 8 + 256;   // ticket at 0, status word at MAX_GRID * 8
// Exchange words the decode kernel needs for one call (0: shape unsupported).
size_t decode_xred_words(const Device& dev, int64_t M, int HC, int HS, int r);
size_t decode_xgat_words(int n_out_max);
cudaError_t launch_decode(const Call& c, const Workspace& ws, const Device& dev,
                          cudaStream_t stream);

// COMBINE alone: R2 = bf16(R + y * 2 sigmoid(inj / HC)), one streaming kernel.
cudaError_t launch_combine(int64_t M, int HC, int HS, const bf16_t* R, const bf16_t* y,
                           const float* inj, int64_t ld_inj, bf16_t* R2, const Device& dev,
                           cudaStream_t stream);

// Prefill path: tcgen05 tensor-core kernels.
cudaError_t launch_prefill(const Call& c, const Workspace& ws, const Device& dev,
                           cudaStream_t stream);
size_t prefill_ws_bytes(int64_t max_M, int HC, int HS, int r);

// ------------------------------------------------------------ device helpers
#if defined(__CUDACC__)

__device__ __forceinline__ float bf16_to_f32(bf16_t v) {
  return __uint_as_float(static_cast<uint32_t>(v) << 16);
}

// Round-to-nearest-even float -> bf16 (the cvt.rn conversion instructions).
__device__ __forceinline__ bf16_t f32_to_bf16(float f) {
  unsigned short r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

__device__ __forceinline__ void unpack8(const uint4 v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Two floats -> packed bf16x2 (a in the low half), round-to-nearest-even.
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}
__device__ __forceinline__ float lo_bf16(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t p) { return __uint_as_float(p & 0xffff0000u); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// --- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread may sleep up to suspend_ns inside the
// instruction while the phase is incomplete (it wakes when the phase
// completes), so waiting warps take few issue slots from working ones.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t suspend_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(bar), "r"(parity), "r"(suspend_ns) : "memory");
  return ok != 0;
}

// Non-blocking check of an mbarrier phase.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Time limits of the bounded waits are counted in SM clock cycles (clock64,
// cheap to read); limit_ns is converted at 2 cycles per ns, the upper end of
// the SM clock range, so a limit never expires early.
__device__ __forceinline__ long long wait_limit_cycles(uint64_t limit_ns) {
  return static_cast<long long>(limit_ns) * 2;
}

// Bounded wait on an mbarrier phase.  On expiry it records DEV_TIMEOUT in the
// status word and returns false; the caller then skips the dependent work.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, int* err,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_sleep(bar, parity, 1000u)) return true;
    if ((it & 15u) == 0) {
      if (clock64() - t0 > wait_limit_cycles(limit_ns)) {
        atomicCAS(err, DEV_OK, DEV_TIMEOUT);
        return false;
      }
      if (*((volatile int*)err) != DEV_OK) return false;
    }
  }
}

// 4-byte asynchronous copy global -> shared (cp.async, L1-allocating); the
// copies of a thread complete at its next cp_async_wait_all().
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;"
               ::"r"(smem_u32(smem_dst)), "l"(__cvta_generic_to_global(gsrc)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// 1-D bulk async copy global -> shared, completion counted on an mbarrier.
// src, dst 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// Tiled TMA loads global -> shared (the tensor map lives in kernel-parameter
// space, passed by generic address).  The destination is 128-byte aligned
// (1024 for 128-byte swizzled boxes); x * element size is a multiple of 16.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(bar) : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar) : "memory");
}

// ---------------------------------------------------------------- tcgen05
// Tensor-memory allocation (one full warp), MMA issue (one thread), commit to
// an mbarrier, and 32-lane loads of accumulator rows.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulator.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
// One lane of the (converged) warp; used for the single-thread tcgen05 issue.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n .reg .b32 r;\n .reg .pred p;\n elect.sync r|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(pred));
  return pred != 0;
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
      ::"r"(bar) : "memory");
}
// Tensor-memory loads.  Each thread of the warp reads N consecutive 32-bit
// columns of its lane (lane = 32 * (warp % 4) + laneid).  The load and the
// wait for its completion sit in one asm block: the destination registers
// are undefined until the wait, so no compiler-inserted move or spill may
// touch them in between.
__device__ __forceinline__ void tmem_ld8_wait(uint32_t t0, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
        "=r"(v[6]), "=r"(v[7])
      : "r"(t0)
      : "memory");
}
__device__ __forceinline__ void tmem_ld8x2_wait(uint32_t t0, uint32_t t1, uint32_t* v0, uint32_t* v1) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%16];\n"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%17];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v0[0]), "=r"(v0[1]), "=r"(v0[2]), "=r"(v0[3]), "=r"(v0[4]), "=r"(v0[5]),
        "=r"(v0[6]), "=r"(v0[7]), "=r"(v1[0]), "=r"(v1[1]), "=r"(v1[2]), "=r"(v1[3]),
        "=r"(v1[4]), "=r"(v1[5]), "=r"(v1[6]), "=r"(v1[7])
      : "r"(t0), "r"(t1)
      : "memory");
}
__device__ __forceinline__ void tmem_ld16_wait(uint32_t t0, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
        "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
        "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(t0)
      : "memory");
}
__device__ __forceinline__ void tmem_ld32_wait(uint32_t t0, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
        "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
        "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]),
        "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]),
        "=r"(v[30]), "=r"(v[31])
      : "r"(t0)
      : "memory");
}
// Generic-proxy writes to shared memory become visible to the async proxy
// (TMA, tcgen05.mma operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Shared-memory matrix descriptor for a K-major operand in the 128-byte
// swizzle layout that TMA writes for 64-element bf16 boxes: rows of 128 bytes,
// 8-row atoms 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t smem_addr) {
  return static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}
// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Hardware tanh approximation (one MUFU operation).
__device__ __forceinline__ float tanh_approx(float x) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(x));
  return t;
}

__device__ __forceinline__ void st_relaxed_u32(unsigned* p, unsigned v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Prefetch of `bytes` contiguous bytes into L2 only (no shared memory
// written, nothing to wait for).  src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}
// Exchange words: 0xffffffff marks an empty word; a value never equals it.
constexpr uint32_t XEMPTY = 0xffffffffu;

__device__ __forceinline__ uint4 ld_relaxed_v4(const uint32_t* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_v4(uint32_t* p, uint4 v) {
  asm volatile("st.relaxed.gpu.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ bool all_set(const uint4& v) {
  return v.x != XEMPTY && v.y != XEMPTY && v.z != XEMPTY && v.w != XEMPTY;
}
// A float as an exchange word (NaN canonicalised, so never the empty marker).
__device__ __forceinline__ uint32_t xword(float v) {
  return v != v ? 0x7fc00000u : __float_as_uint(v);
}
// Writes that an earlier grid made with ordinary stores, ordered before this
// thread's later async-proxy (TMA) reads of global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Programmatic dependent launch: wait for the grid this one depends on (a
// no-op without that dependency), and let the next grid start launching.
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 1 / (1 + e^-u) with the fast exponential and division (a few ulp);
// e^-u overflowing to +inf gives 0.
__device__ __forceinline__ float sigmoid_fast(float u) { return __fdividef(1.0f, 1.0f + __expf(-u)); }
// COMBINE weight iw = 2 sigmoid(inj / HC), inv_hc = 1 / HC.  Decode and
// prefill form it the same way, so their R2 agree bit for bit.
__device__ __forceinline__ float combine_weight(float inj, float inv_hc) {
  return 2.0f * sigmoid_fast(inj * inv_hc);
}
// 1 / sqrt(v): hardware estimate plus one Newton step (~1 ulp).
__device__ __forceinline__ float rsqrt_nr(float v) {
  const float y = rsqrtf(v);
  return y * fmaf(-0.5f * v * y, y, 1.5f);
}

#endif  // __CUDACC__

}  // namespace hcgr

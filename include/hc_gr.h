/*
 * hc_gr.h -- C ABI of the Hyper-Connection gated residual (HC-GR) for one
 * GB300 GPU (sm_103a).
 *
 * The operation (aiter PR #5913, "Two-stage Hyper-Connection Gated Residual
 * kernel", section "Technical Details"), per token, with HC residual streams
 * of width HS, K = HC * HS and low rank r:
 *
 *   (COMBINE) iw[s] = 2 * sigmoid(inj[s] / HC)
 *             R2[s, c] = R[s, c] + y[c] * iw[s]              -> stored in bf16
 *   (N)       rrms[s] = 1 / sqrt(mean_c R2[s, c]^2 + eps)
 *             xn[s, c] = R2[s, c] * rrms[s] * (1 + Wnorm[s * HS + c])
 *   (G1)      lora = xn . Wd^T            (r values, stored before SiLU)
 *             h = SiLU(lora / HC)
 *   (INJ)     inj_next = xn . Wi^T        (HC values, the next layer's logits)
 *   (G2)      G = sigmoid(h . Wu^T)       (K values, never stored)
 *   (MIX)     x[c] = (1 / HC) * sum_s G[s * HS + c] * xn[s * HS + c]
 *
 * R2 is rounded to bf16 before rrms and everything after it are computed, the
 * way the page's second kernel rebuilds xn from the stored R2 and rrms.
 *
 * Types and layouts (all row-major, contiguous unless a leading dimension is
 * given; M tokens):
 *   R, R2      [M, HC, HS] bf16        y, x      [M, HS] bf16
 *   inj        [M, HC] fp32 (row stride ld_inj >= HC in hc_gr_forward_ex)
 *   rrms, inj_next [M, HC] fp32        lora      [M, r] fp32
 *   Wnorm      [K] bf16 (or [HS], shared by the streams: hc_gr_args.wnorm_hs)
 *                                      Wd        [r, K] bf16
 *   Wi         [HC, K] bf16            Wu        [K, r] bf16
 *   Wdi        [n_pad, K] bf16 merged down/inject weight: rows 0..r-1 = Wd,
 *              rows r..r+HC-1 = Wi, rows r+HC..n_pad-1 are never read.  With
 *              fold_w = 1 every column k already carries the factor
 *              (1 + Wnorm[k]) (the "(1+w) folded in" weight of the page's
 *              Performance setup); Wnorm is then still read for the mix.
 * bf16 is passed as raw 16-bit storage (const void*).  Every pointer is a
 * device pointer owned by the caller; the library never frees or retains it
 * past the call.  bf16 tensors and lora are 16-byte aligned; inj, rrms and
 * inj_next need only 4-byte alignment.  HS and r are multiples of 8.  The
 * prefill kernels additionally need HS and r multiples of 64, r <= 512 and
 * HC <= 8; other shapes run on the decode kernel (M <= 64) or are rejected
 * with HC_GR_ERR_UNSUPPORTED.
 *
 * Streams and concurrency: hc_gr_forward* only enqueues work on `stream`
 * (a cudaStream_t; NULL is the legacy default stream) and returns.  A handle
 * owns one workspace (the decode kernel's cross-CTA exchange buffers and call
 * ticket, the prefill kernels' scratch and a device status word); calls on
 * one handle must be ordered on one stream.  Use one handle per concurrent
 * stream.
 *
 * Errors: every entry point returns an hc_gr_status.  Argument errors are
 * detected on the host before anything is enqueued and leave outputs
 * untouched.  A device-side failure (a bounded wait that expired) is
 * recorded in the handle and reported by hc_gr_check; the outputs of that
 * call, and of every later call on the handle until hc_gr_check has cleared
 * the status, are undefined.
 *
 * Size limits: M and max_M at most HC_GR_MAX_TOKENS, HC * HS at most
 * HC_GR_MAX_WIDTH (UNSUPPORTED beyond), so that every element offset the
 * kernels form stays inside their index types.
 */
#ifndef HC_GR_H_
#define HC_GR_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t == struct CUstream_st* */

typedef struct hc_gr_ctx* hc_gr_handle;

#define HC_GR_MAX_TOKENS (1LL << 30) /* largest M (and max_M) accepted */
#define HC_GR_MAX_WIDTH (1LL << 30)  /* largest K = HC * HS accepted */

/* Status codes.  The contract follows the page's "PR Self-Review", section
 * "Behavior and intent": the public entry points refuse what they cannot
 * compute correctly (unsupported architecture, widths the kernels cannot
 * tile, malformed or aliased buffers) instead of returning wrong results;
 * the review findings on strided injection and up-weight validation are
 * honoured by explicit strides and checks rather than rejected. */
typedef enum hc_gr_status {
  HC_GR_OK = 0,
  HC_GR_ERR_INVALID_ARG = 1, /* NULL pointer, M < 1, eps <= 0 or not finite,
                                misaligned pointer, ld_inj < HC, bad path */
  HC_GR_ERR_UNSUPPORTED = 2, /* shape outside what the handle was created for,
                                HS or r not a multiple of 8, n_pad < r + HC,
                                M or HC * HS above the size limits, a device
                                that is not sm_103 */
  HC_GR_ERR_ALIAS = 3,       /* an output overlaps another output or an input */
  HC_GR_ERR_CUDA = 4,        /* a CUDA call failed (launch, allocation, copy) */
  HC_GR_ERR_TIMEOUT = 5      /* a device-side bounded wait expired */
} hc_gr_status;

/* Dispatch between the two kernel families (the page's "Behavior and intent":
 * a skinny decode path for few tokens beside the tiled two-kernel path). */
typedef enum hc_gr_path {
  HC_GR_PATH_AUTO = 0,    /* M <= 64 and M * HC * HS <= 64 * 10240 (the
                             measured crossover: 64 tokens at HC=4, HS=2560;
                             20 at HC=8, HS=4096): decode kernel, otherwise
                             (or where its plan does not fit) prefill */
  HC_GR_PATH_DECODE = 1,  /* weight-streaming persistent kernel, M <= 64 */
  HC_GR_PATH_PREFILL = 2  /* tensor-core (tcgen05) two-stage kernels */
} hc_gr_path;

/* Full argument set of hc_gr_forward_ex.  Zero-initialise, then fill.
 * Wdi / n_pad / fold_w: the merged down/inject weight of the page's
 * "Performance" setup (336 rows with (1 + w) folded in); ld_inj: the strided
 * injection the review found a kernel ignoring ("Validation and unverified
 * scope": the strided combine case). */
typedef struct hc_gr_args {
  int64_t M;
  int32_t HC, HS, r;
  float eps;
  const void* R;
  const void* y;
  const float* inj;
  int64_t ld_inj;      /* row stride of inj in floats; 0 means HC */
  const void* Wnorm;
  const void* Wd;      /* separate down weight [r, K]; used when Wdi == NULL */
  const void* Wi;      /* separate inject weight [HC, K] */
  const void* Wdi;     /* merged [n_pad, K] weight, or NULL */
  int32_t n_pad;       /* rows of Wdi (>= r + HC); ignored without Wdi */
  int32_t fold_w;      /* 1: the projection weight carries (1 + Wnorm) */
  const void* Wu;
  void* R2;
  float* rrms;
  float* inj_next;
  void* x;
  float* lora;         /* may be NULL: lora is then kept in the workspace */
  int32_t force_path;  /* hc_gr_path */
  int32_t debug_fault; /* tests only: 1 = one CTA of the decode kernel writes
                          none of its partial sums, as if it had died, so the
                          others' bounded waits expire and hc_gr_check reports
                          TIMEOUT */
  int32_t pdl;         /* 1: launch as a programmatic dependent of the
                          previous kernel on `stream`.  Decode: its weight
                          copies (Wd and Wi or Wdi, and Wu) may start before
                          that kernel has finished, so that kernel must not
                          write them; activations are read and outputs written
                          only after it has finished.  Prefill: K1's prologue
                          overlaps the previous kernel (K1 touches memory
                          only after it has finished).  0: plain stream
                          order for the call's first kernel.  Inside a
                          prefill call the stream reduce is always a
                          dependent of K1 and K2 of the reduce, whatever this
                          field; each waits for its predecessor to finish
                          before it touches memory. */
  int32_t wnorm_hs;    /* 1: Wnorm has HS entries, one per channel, shared by
                          every stream (xn[s, c] = R2[s, c] rrms[s]
                          (1 + Wnorm[c])); 0: the full-width [K] layout.  A
                          folded Wdi then carries (1 + Wnorm[k mod HS]). */
} hc_gr_args;

/* Creates a handle bound to `device` and allocates its workspace for calls
 * with M <= max_M, HC * HS <= the given HC * HS and r + HC <= the given
 * r + HC.  Queries the device (SM count, shared memory) once.  (The page's
 * op keeps per-device state -- its skinny decode's arrival counters, "PR
 * Self-Review" -- in a process-wide cache; here that state is the handle's.)
 * Returns INVALID_ARG for out == NULL or non-positive sizes, UNSUPPORTED for
 * max_M or HC * HS above the size limits or a device that is not sm_103,
 * CUDA when the device query or the allocation fails (*out is then NULL in
 * every failure). */
int hc_gr_create(hc_gr_handle* out, int device, int64_t max_M, int HC, int HS, int r);

/* The whole forward pass for one batch of M tokens with separate, unfolded
 * Wd and Wi (see the layouts above): the (COMBINE), (N), (G1), (INJ), (G2)
 * and (MIX) bullets of the page's "Technical Details" in one call -- its
 * combine_and_mix entry point ("Behavior and intent").  lora may be NULL.
 * Asynchronous on `stream`. */
int hc_gr_forward(hc_gr_handle h, int64_t M, int HC, int HS, int r, float eps,
                  const void* R, const void* y, const float* inj, const void* Wnorm,
                  const void* Wd, const void* Wi, const void* Wu,
                  void* R2, float* rrms, float* inj_next, void* x, float* lora,
                  struct CUstream_st* stream);

/* Same operation ("Technical Details", as hc_gr_forward) with every option:
 * a merged (optionally folded) weight, a strided inj and a forced path.
 * With y, inj and R2 all NULL the call is the mix alone (see hc_gr_mix);
 * NULL in only some of them is INVALID_ARG. */
int hc_gr_forward_ex(hc_gr_handle h, const hc_gr_args* a, struct CUstream_st* stream);

/* COMBINE alone (the page's combine-only entry point, "Behavior and intent";
 * the formula of the (COMBINE) bullet): R2 = bf16(R + y * 2 sigmoid(inj /
 * HC)) for M tokens, nothing else.  For layers that apply COMBINE apart from
 * the mix.  R2 is bit-identical to the R2 hc_gr_forward stores for the same
 * inputs.
 *   R, R2 [M, HC, HS] bf16 (16-byte aligned), y [M, HS] bf16 (16-byte
 *   aligned), inj [M, HC] fp32 with row stride ld_inj >= HC floats (0 means
 *   HC; 4-byte aligned), so the strided inj_next of a previous call can be
 *   passed as it is.  Any M >= 1 and HC >= 1; HS a multiple of 8
 *   (UNSUPPORTED otherwise).  The handle supplies the device and keeps the
 *   last CUDA error; its workspace is not used and its size limits do not
 *   apply.  R2 must not overlap R, y or inj (ALIAS).  One kernel launch,
 *   asynchronous on `stream`. */
int hc_gr_combine(hc_gr_handle h, int64_t M, int HC, int HS, const void* R, const void* y,
                  const float* inj, int64_t ld_inj, void* R2, struct CUstream_st* stream);

/* The mix alone (the page's mix entry point, "Behavior and intent"): every
 * step after COMBINE -- (N), (G1), (INJ), (G2), (MIX) -- with R taken as
 * the already-combined streams (R2 = R; nothing is injected and R2 is not
 * written).  Outputs rrms, inj_next, x and lora (may be NULL) as in
 * hc_gr_forward, the same limits, layouts and paths.  Equivalent to
 * hc_gr_forward_ex with y = inj = R2 = NULL. */
int hc_gr_mix(hc_gr_handle h, int64_t M, int HC, int HS, int r, float eps, const void* R,
              const void* Wnorm, const void* Wd, const void* Wi, const void* Wu, float* rrms,
              float* inj_next, void* x, float* lora, struct CUstream_st* stream);

/* Waits for `stream`, then returns the device status recorded by the
 * handle's kernels since the last check (HC_GR_OK or HC_GR_ERR_TIMEOUT).
 * The status comes from the bounded cross-CTA waits that replace the page's
 * skinny-decode arrival counters ("Behavior and intent"); a wait that
 * expires reports instead of hanging.
 * After a TIMEOUT it clears the status and resets the exchange buffers and
 * the call ticket, so the handle is usable again.  Returns HC_GR_ERR_CUDA if
 * the stream reports a CUDA error. */
int hc_gr_check(hc_gr_handle h, struct CUstream_st* stream);

/* Releases the workspace.  Waits for the device first.  NULL is a no-op.
 * (No counterpart on the pages: their op owns no handle.) */
int hc_gr_destroy(hc_gr_handle h);

/* Static text for a status code.  (No counterpart on the pages.) */
const char* hc_gr_strerror(int status);

/* Text of the last CUDA error seen by this handle (static storage).  (No
 * counterpart on the pages.) */
const char* hc_gr_last_cuda_error(hc_gr_handle h);

/* hc_gr_forward without a handle and without any device allocation.  The
 * pages have no counterpart: this entry point exists for callers that may not
 * call cudaMalloc on their call path, for instance an engine whose memory
 * manager owns all device memory, or code that must not risk the implicit
 * device synchronisation of an allocation.  It runs the decode kernel with
 * its scratch memory (the cross-CTA exchange buffers, lora when lora is NULL,
 * the call ticket and the status word) in one fixed 4 MiB device array inside
 * the library, which every GPU that loads the library holds until the process
 * exits.
 *   - Limits: M <= 8 tokens and r + HC <= 336; larger sizes return
 *     HC_GR_ERR_UNSUPPORTED.  Other arguments, layouts and alignment as for
 *     hc_gr_forward; the current device is used.
 *   - The first call on a device queries the device and resolves the device
 *     address of the scratch array; make that first call before any stream
 *     capture.
 *   - Every call shares the one array: calls that overlap on the GPU (on
 *     different streams, or on several host threads) race and corrupt each
 *     other.  Each call first empties the exchange buffers and clears the
 *     call ticket (memsets on `stream`); the status word is left as it is,
 *     so a device-side timeout of any call stays recorded until
 *     hc_gr_noalloc_check reads and clears it (as with a handle, the outputs
 *     of the failed call and of every later call until then are undefined).
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 *     routine.  Asynchronous on `stream`. */
int hc_gr_forward_noalloc(int64_t M, int HC, int HS, int r, float eps,
                          const void* R, const void* y, const float* inj, const void* Wnorm,
                          const void* Wd, const void* Wi, const void* Wu,
                          void* R2, float* rrms, float* inj_next, void* x, float* lora,
                          struct CUstream_st* stream);

/* Status of the hc_gr_forward_noalloc calls on the current device.  The pages
 * have no counterpart.  Waits for `stream`, then reads the status word in the
 * fixed scratch array: HC_GR_OK, or HC_GR_ERR_TIMEOUT if a device-side bounded
 * wait of any call since the last check expired (the outputs of those calls
 * are undefined); a TIMEOUT is cleared by the check.  HC_GR_OK before the
 * first call on the device.  HC_GR_ERR_CUDA if the stream reports an error.
 * Allocates nothing. */
int hc_gr_noalloc_check(struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* HC_GR_H_ */

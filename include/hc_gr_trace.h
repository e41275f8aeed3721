/*
 * hc_gr_trace.h -- phase timeline of the decode kernel (diagnostic build).
 *
 * Not part of the library's ABI: the symbol exists only in
 * libhc_gr_trace.so, the same sources compiled with HCGR_TRACE defined
 * (hyper_connection_gated_gb300/build.py, build(trace=True)).  In that build
 * thread 0 of every decode CTA records %globaltimer (ns) at fixed points of
 * the kernel into a device array of 36 slots per CTA:
 *   0 start, 1 prologue done (weight copies issued, TMEM allocated),
 *   2 previous kernel finished (griddepcontrol.wait returned),
 *   down CTAs: 3 COMBINE done, 4 the first issuer's last weight box landed
 *              and its MMAs issued, 5 every down MMA complete, 6 the CTA's
 *              reduce-scatter pieces written;
 *   up CTAs:   7 first reduce-scatter block gathered, 8 every block reduced
 *              (h published), 9 all-gather of h done, 10 gate MMAs complete,
 *              11 x stored;
 *   12 end (tensor memory released), 13 the prologue's CTA barrier passed,
 *   14 thread 0's first weight box issued, 15 the first up issuer's gate
 *   MMAs issued, 16 (down) the last reduce-scatter store issued by any
 *   thread, 17 (up) the last word of its first block seen by any thread,
 *   18-23 sub-stamps of the reduce (18 piece loop left, 19 shuffle tree
 *   passed, 20 sum stored; latest thread), of the gate readback (21), of x
 *   (22) and of the first product readback (23); 24/25 the first down
 *   issuer's first box landed / its first MMAs issued; 26 (up) the last
 *   thread out of the all-gather loop; 27/28 the first up issuer's first
 *   chunk landed / its MMAs issued; 29 (up) the mix inputs landed;
 *   30 (down) the down MMAs' completion seen; 31 (up) the gate MMAs'
 *   completion seen; 32/33 thread 0 before / after the barrier
 *   initialisation; 34 the last thread at the prologue's CTA barrier;
 *   35 unused.
 * Slots a CTA does not pass read 0 (every read clears the array).
 */
#ifndef HC_GR_TRACE_H_
#define HC_GR_TRACE_H_

#ifdef __cplusplus
extern "C" {
#endif

/* Copies n <= 256 * 36 values ([CTA][36], CTA = blockIdx.x of the last
 * decode launch) to host memory, then zeroes the device array.  Returns the
 * CUDA status (0 = success). */
int hc_gr_trace_read(unsigned long long* host, int n);

#ifdef __cplusplus
}
#endif

#endif /* HC_GR_TRACE_H_ */

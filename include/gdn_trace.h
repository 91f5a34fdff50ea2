/*
 * Per-role clock trace of the tensor-core chunk kernel: exported only by the tracing
 * build of the library (libgdn_trace.so, compiled with -DGDN_TC_TRACE; the
 * package's build(trace=True) makes it). The regular library has none of this code.
 *
 * One CTA is traced: lane 0 of warp w records clock64() at point p (0-7) of the life
 * of each chunk c < 256 it handles, into slot [w][c][p] of a 16 x 256 x 8 array of
 * uint64 (0 = not reached); four more words hold {clock64, %globaltimer} at the CTA's
 * start and end, for the clock rate. Warps: 0 producer, 1 W' / U products, 2 state
 * products, 3 [K;Q] K^T and q norms, 4 (first of WG-A) chunk preparation, 12 (first of
 * WG-B) state step and epilogue. The points of each warp are listed by the package's
 * trace tool (gated_deltanet_linear_prefill_gb300/trace.py).
 *
 * Each returns a cudaError_t value (0 on success). Stamps are written by the kernel
 * launches that follow: clear, set the CTA, launch, then read.
 */
#ifndef GDN_TRACE_H_
#define GDN_TRACE_H_

#ifdef __cplusplus
extern "C" {
#endif

/* Selects the CTA (blockIdx.x) that later launches trace. */
int gdn_trace_set_cta(int cta);
/* Zeroes every stamp. */
int gdn_trace_clear(void);
/* Synchronises the device and copies the 16 * 2048 + 4 words to `host`. */
int gdn_trace_read(unsigned long long* host);

#ifdef __cplusplus
}
#endif

#endif

/*
 * ssb_peaks.h -- throughput probes of libssb (measurement only, not part of
 * the method).
 *
 * The batched scoring pass evaluates one sincos (two transcendental results)
 * per active (q, k, set) term, and the G build is float32 arithmetic; their
 * roofline fractions are taken against rates measured on the device in the
 * same run, not against datasheet figures.  These two kernels produce those
 * rates: each thread runs 8 independent dependency chains for `iters`
 * iterations, with `blocks` CTAs of 256 threads, asynchronously on `stream`
 * (a cudaStream_t passed as void*).  The caller times them (CUDA events on
 * the same stream) and divides the operation counts below by the time.
 *
 *   ssb_peak_sincos: per iteration and chain one __sincosf (2 transcendental
 *                    results, as in the scoring kernel) and one multiply-add
 *                    that feeds the next argument:
 *                    2 * 8 * 256 * blocks * iters transcendental results.
 *   ssb_peak_fma:    per iteration and chain one float32 fused multiply-add:
 *                    2 * 8 * 256 * blocks * iters floating-point operations.
 *
 * out_dev: device float[1], written only in a case that never occurs (it
 * keeps the chains live).  Returns 0 (SSB_OK), 1 for blocks or iters < 1 or a
 * NULL out_dev, 4 on a launch error (message in ssb_last_error()).
 */
#ifndef SSB_PEAKS_H
#define SSB_PEAKS_H

#ifdef __cplusplus
extern "C" {
#endif

int ssb_peak_sincos(float* out_dev, int blocks, int iters, void* stream);
int ssb_peak_fma(float* out_dev, int blocks, int iters, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SSB_PEAKS_H */

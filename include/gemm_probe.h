/*
 * gemm_probe.h -- peak probes of the GB300 GEMM library (C ABI).
 *
 * Throughput is reported against the roofline min(peak, I x HBM bandwidth)
 * ("GEMM on NVIDIA GPUs: from naive kernel to tiled pipeline", section 2
 * "GEMM arithmetic intensity"; "Understanding roofline and tiling through
 * matrix multiplication", section 8).  The pages give no GB300 peaks, so the
 * library carries two kernels that measure the arithmetic units with no
 * memory traffic, as a cross-check of the peaks the roofline divides by:
 *
 *   gemm_probe_tc_bf16  the tensor pipe: back-to-back BF16 tcgen05.mma
 *                       (FP32 accumulation) on operands resident in shared
 *                       memory -- the GEMM mainloop's MMA stream without its
 *                       loads;
 *   gemm_probe_fma_f32  the CUDA cores: chains of FP32 FMAs in registers
 *                       (the speed-of-light estimate of "Worklog: optimising
 *                       GEMM on NVIDIA H100", SM count x FP32 lanes x 2 x
 *                       clock).
 *
 * Both enqueue exactly one kernel on `stream` (asynchronous, like the GEMM
 * entry points), write the number of floating-point operations that kernel
 * performs to *flops before returning, and touch no caller memory on the
 * device.  The caller times the launch (for example with CUDA events on
 * `stream`) and divides.  The values the kernels compute are discarded.
 *
 * A third probe, gemm_probe_wait_timeout, exercises the kernels' failure
 * path (a bounded wait that runs out) without breaking a kernel.
 *
 * Errors (returned before any launch unless noted):
 *   GEMM_ERR_INVALID_VALUE       a count outside [1, 2^40], cta_group not 1
 *                                or 2, or flops == NULL
 *   GEMM_ERR_UNSUPPORTED_DEVICE  the current device is not sm_103
 *   GEMM_ERR_LAUNCH / _INTERNAL  the launch or its setup failed
 * gemm_probe_tc_bf16 waits for its MMAs with a bounded wait (at least 1 s,
 * and 4x the time the MMAs take at 2 PFLOP/s); if it runs out, the device
 * status word reads GEMM_ERR_TIMEOUT (gemm_last_device_status).
 */
#ifndef DENSE_GEMM_08_GB300_GEMM_PROBE_H
#define DENSE_GEMM_08_GB300_GEMM_PROBE_H

#include <stdint.h>

#include "gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * cta_group 1: one CTA per SM issues n_mma MMAs of 128 x 256 x 16
 *   (2^20 FLOPs each);
 * cta_group 2: one CTA pair per two SMs (as many pairs as can be resident)
 *   issues n_mma MMAs of 256 x 256 x 16 (2^21 FLOPs each).
 * *flops = FLOPs per MMA x n_mma x CTA groups launched.
 */
gemm_status_t gemm_probe_tc_bf16(int cta_group, int64_t n_mma, double *flops,
                                 cudaStream_t stream);

/*
 * 8 CTAs of 256 threads per SM; each thread runs 8 independent chains of
 * 16 x trips dependent FP32 FMAs.  *flops = 2 x 8 x 16 x trips x threads.
 */
gemm_status_t gemm_probe_fma_f32(int64_t trips, double *flops, cudaStream_t stream);

/*
 * The kernels' failure path, exercised without breaking a kernel: one thread
 * waits, with the same bounded wait the GEMM kernels use, on a barrier that
 * nothing completes; after timeout_ns (1 us .. 10 s) it gives up and sets the
 * device status word, so that gemm_last_device_status returns
 * GEMM_ERR_TIMEOUT (and clears the word).  Nothing else is in flight and the
 * CUDA context stays usable.  Enqueues one kernel on `stream`.
 * Errors: GEMM_ERR_INVALID_VALUE (timeout out of range),
 * GEMM_ERR_UNSUPPORTED_DEVICE, GEMM_ERR_LAUNCH.
 */
gemm_status_t gemm_probe_wait_timeout(uint64_t timeout_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_GEMM_08_GB300_GEMM_PROBE_H */

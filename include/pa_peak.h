/*
 * pa_peak.h - tensor-core throughput probe (libpa_peak.so), the measured
 * denominator of the "fraction of the dense int8 tensor roofline" that the
 * benchmark reports ("int8 tensor-core prefill attention", section "Summary":
 * the attention moves to int8 tensor cores; sm_103a has no integer tcgen05
 * MMA, so the int8 tensor rate of this GPU is that of the warp-level
 * mma.sync s8 instruction).  Not part of the attention library.
 */
#ifndef PA_PEAK_H
#define PA_PEAK_H

#ifdef __cplusplus
extern "C" {
#endif

#define PA_PEAK_S8 0   /* mma.sync.m16n8k32 s8 x s8 -> s32 */
#define PA_PEAK_F16 1  /* mma.sync.m16n8k16 f16 x f16 -> f32 */

/* Run `iters` rounds of eight independent MMAs per warp, eight warps per
 * block, blocks_per_sm (1..8) blocks per SM of the current device, and report
 * the rate in tera-ops per second (2 M N K per MMA) and the kernel's time in
 * milliseconds (ms may be NULL).  Allocates and frees its own small buffers;
 * synchronous.  Returns 0, -1 for a bad argument, -3 if a CUDA call failed. */
int pa_peak_mma_sync(int kind, int blocks_per_sm, long long iters, double* tops, double* ms);

#ifdef __cplusplus
}
#endif

#endif /* PA_PEAK_H */

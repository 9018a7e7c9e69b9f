/*
 * w12_debug.h -- test hooks of the W12 library (not for production use).
 *
 * These exist so that the failure paths of the kernels can be exercised
 * without faulting the GPU: every wait inside the kernels is bounded, and a
 * test can make one wait run out on purpose.
 */
#ifndef W12_DEBUG_H
#define W12_DEBUG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Process-wide debug settings applied to every later launch.
 *   flags bit 0: in the next GEMM launches, CTA 0's producer announces its
 *                first record but never copies it, so that CTA's consumers
 *                time out; the kernel records W12_E_TIMEOUT in the workspace
 *                status word and every CTA returns with no copy in flight.
 *                In the recurrent layer's tensor-memory WY kernel (trees of
 *                several requests), CTA (0, 0) never copies its first
 *                request's state: its splitters' wait runs out, both warp
 *                roles stop, W12_E_TIMEOUT is recorded and tensor memory is
 *                released.
 *   flags bit 1: run every GEMM on the tensor-memory (tcgen05) kernel.
 *   flags bit 2: run every GEMM on the warp-MMA kernel (64 rows per pass).
 *                Without either bit the library picks by row count.
 *   flags bit 3: w12_verify_step launches one kernel per GEMM (the default).
 *   flags bit 4: w12_verify_step runs all its GEMMs (every linear, then the
 *                LM head) as one persistent tensor-memory GEMM chain: one
 *                launch per up to 144 GEMMs, each GEMM's activations read
 *                once every CTA has finished the previous GEMM.  Bits 2 and
 *                3 take precedence.
 *   timeout_ns:  limit of every bounded wait inside the kernels
 *                (0 restores the default of 2 seconds).
 * Not thread-safe; meant to be set between launches by a test.
 */
void w12_debug_set(int32_t flags, uint64_t timeout_ns);

/*
 * Per-launch timing of w12_verify_step for benchmarks.  While enabled, the
 * step records a CUDA event before its first launch and after every launch
 * (which also serialises the launches, so steps timed this way lose the
 * overlap between consecutive kernels).  w12_debug_profile_read synchronises
 * on the last event and writes the elapsed milliseconds of each launch of the
 * most recent step (GEMM launches in order, then the argmax reduction, then
 * acceptance) to ms[0..max); it returns the number of launches, or a
 * negative status.
 */
void w12_debug_profile(int32_t enable);
int32_t w12_debug_profile_read(float *ms, int32_t max);

/*
 * The CUDA error behind the most recent W12_E_CUDA returned by this library
 * (0 if none): its code, and its name copied into buf (len bytes, may be NULL).
 */
int32_t w12_debug_last_cuda_error(char *buf, int32_t len);

/* Number of SMs the kernels size their persistent grids for (current device). */
int32_t w12_debug_num_sms(void);

/*
 * Per-GEMM timing inside the verify step's GEMM chain (one persistent launch
 * for all linears and the LM head, split into w12_debug_chain_parts(n) launches
 * for n GEMMs).  While dev_words (device, n_words 64-bit words) is set, every
 * CTA of a chain launch covering GEMMs [j0, j0 + m) writes the global timer
 * (ns) when it starts, at word ((j0 + part) + m) * S + cta, and when it has
 * written its last output of GEMM j, at word (j + part) * S + cta, with S the
 * SM count and part the launch's index.  GEMM j ends when the last CTA
 * stamps it.  Too small a buffer disables the stamps.  NULL turns it off.
 */
void w12_debug_chain_trace(void *dev_words, size_t n_words);
int32_t w12_debug_chain_parts(int32_t n_gemms);

#ifdef __cplusplus
}
#endif

#endif /* W12_DEBUG_H */

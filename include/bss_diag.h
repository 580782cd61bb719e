/*
 * bss_diag.h -- diagnostic entry point of the block-sparse attention library.
 *
 * Not an operation of the method (the blog has no counterpart): a one-tile
 * self-test of the tensor-core building blocks the attention kernel is made
 * of -- TMA loads into 128-byte swizzled shared memory, the shared-memory and
 * instruction descriptors, tcgen05.mma with both operands in shared memory and
 * with the A operand in tensor memory, and tcgen05 loads/stores -- so a wrong
 * descriptor shows up as a wrong matrix product, isolated from the softmax.
 */
#ifndef BSS_DIAG_H_
#define BSS_DIAG_H_

#include "bss.h"

#ifdef __cplusplus
extern "C" {
#endif

/* One CTA computes, with the attention kernel's own code paths,
 *   S = A B^T          A, B: device bf16 [128][d]     -> S: device float [128][128]
 *   O = P V            P: device bf16 [128][128] (written into tensor memory
 *                      row by row, as the softmax does), V: device bf16 [128][d]
 *                                                     -> O: device float [128][d]
 * d = 64 or 128; all pointers 16-byte aligned.  Asynchronous on `stream`.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA; timeouts via bss_get_device_status. */
bss_status bss_diag_mma_tile(const void* A, const void* B, const void* P, const void* V, float* S, float* O,
                             int32_t d, cudaStream_t stream);

/* Failure-detection check of the bounded waits every kernel uses: one CTA
 * initialises an mbarrier that nothing ever arrives on and waits on it with
 * the same bounded wait as the attention kernel, giving up after limit_ns
 * nanoseconds (1e3 .. 1e9).  The wait records BSS_ERR_TIMEOUT in the device
 * status word and the kernel returns normally, so the context stays usable;
 * the host reads the status with bss_get_device_status.  *waited_ns (device
 * int64, may be NULL) receives the time the wait took.
 * Errors: INVALID_ARG (limit out of range, misaligned pointer), CUDA. */
bss_status bss_diag_wait_timeout(int64_t limit_ns, int64_t* waited_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BSS_DIAG_H_ */

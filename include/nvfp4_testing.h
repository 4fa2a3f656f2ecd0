/*
 * nvfp4_testing.h -- test support entry points of libnvfp4.
 *
 * The pages have no counterpart for these.  The first exists so that a test
 * can make one of the GEMM's bounded waits run out on a real GPU, without a
 * fault, and check the library's failure path (the status word read by
 * nvfp4_device_error in nvfp4.h, and that the next call still works).  The
 * other two serve the library's debug build (libnvfp4_debug.so, compiled
 * with NVFP4_BOUNDS_CHECK): there every store of a code, a scale byte or an
 * output element (dequantize, and the GEMM epilogue's stores that do not go
 * through TMA, whose tensor maps bound their own stores) first checks that
 * its bytes lie in the range the call declared for that buffer (from its
 * first byte to the last byte its shape and leading dimension reach), and a
 * store outside is skipped and counted instead of written.  The tensor
 * amax, s_g and workspace words are single words and are not checked.
 * Production code has no reason to call any of them.
 */
#ifndef NVFP4_TESTING_H
#define NVFP4_TESTING_H

#include "nvfp4.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * nvfp4_testing_arm_gemm_timeout -- arm a fault for the next GEMM launch of
 * this process (the next nvfp4_gemm, nvfp4_gemm_amax, nvfp4_gemm_lora or
 * nvfp4_gemm_axpby call on any thread; the arm is consumed by that launch).
 *  wait_limit_us  every mbarrier wait of that launch gives up after this
 *                 many microseconds instead of 2 s; 1000 .. 2000000.
 * In that launch the leader CTA of every CTA pair leaves out one arrival on
 * the barrier that releases its first K stage to the MMA issuer, so the
 * issuer's wait runs out: the kernel sets the status word's timeout bit,
 * waits (bounded) for its copies and MMAs in flight, frees its tensor
 * memory and returns; its output is not written.  nvfp4_device_error then
 * returns NVFP4_ERR_TIMEOUT (and clears the word).  Use a GEMM of one
 * 256 x 256 output tile, so that one CTA pair runs.
 * Returns NVFP4_ERR_INVALID_ARG for a limit outside the range, else NVFP4_OK.
 */
NVFP4_API nvfp4_status nvfp4_testing_arm_gemm_timeout(uint32_t wait_limit_us);

/*
 * nvfp4_testing_bounds_violations -- the number of stores the debug build's
 * bounds check skipped since the previous call (the count is then cleared).
 *  count  host pointer, receives the number.
 * Synchronizes the device first.  Returns NVFP4_ERR_UNSUPPORTED in the
 * regular build (the check is not compiled in; *count is not written),
 * NVFP4_ERR_INVALID_ARG for a null count, NVFP4_ERR_CUDA if reading the
 * device counters fails.
 */
NVFP4_API nvfp4_status nvfp4_testing_bounds_violations(uint64_t* count);

/*
 * nvfp4_testing_bounds_shrink -- debug build: every call made after this
 * one declares each output buffer `bytes` bytes shorter than its shape says
 * (0 restores the true ranges), so that the check fires on stores that are
 * in fact inside the caller's allocation: a test of the check itself that
 * touches no memory outside any buffer.  0 <= bytes <= 4096, else
 * NVFP4_ERR_INVALID_ARG; NVFP4_ERR_UNSUPPORTED in the regular build.  The
 * setting is process-wide.
 */
NVFP4_API nvfp4_status nvfp4_testing_bounds_shrink(int64_t bytes);

#ifdef __cplusplus
}
#endif
#endif

/*
 * nvfp4_testing.h -- test support entry point of libnvfp4.
 *
 * The pages have no counterpart for this: it exists so that a test can make
 * one of the GEMM's bounded waits run out on a real GPU, without a fault,
 * and check the library's failure path (the status word read by
 * nvfp4_device_error in nvfp4.h, and that the next call still works).
 * Production code has no reason to call it.
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

#ifdef __cplusplus
}
#endif
#endif

/*
 * mla_testing.h -- test hooks of the GB300 MLA library.  Not part of the operations in
 * mla.h and never needed by a user: they exist so that tests can drive the library's
 * failure handling without faulting a GPU.
 */
#ifndef MLA_GB300_TESTING_H_
#define MLA_GB300_TESTING_H_

#ifdef __cplusplus
extern "C" {
#endif

/*
 * mla_testing_decode_stall -- make later mla_decode calls that take the transposed kernel
 * (fp8 cache, q_len * H <= 32) leave the pipeline unit numbered `skip_unit` (counted per CTA
 * from 0) unloaded, and give every device-side pipeline wait `wait_limit_cycles` SM clocks
 * before it gives up.  The stage that waits for the missing unit then runs out: the kernel
 * latches MLA_ERR_TIMEOUT in the device error word (read by mla_check_device_error), every
 * role of the CTA leaves its loop, lets its own copies and MMAs in flight finish, and the
 * CTA frees its tensor memory and exits.  The outputs of such a call are undefined.
 * skip_unit < 0 restores normal calls; wait_limit_cycles <= 0 restores the default limit
 * (about 0.5 s of SM clocks).  Process-wide; not thread-safe with respect to calls in flight.
 */
void mla_testing_decode_stall(int skip_unit, long long wait_limit_cycles);

/*
 * mla_testing_bounds_checked -- 1 when this library is the bounds-checked build (compiled
 * with MLA_DEBUG): every store of an output, LSE or workspace element is checked against
 * its buffer; one that falls outside is skipped and latches MLA_ERR_DEVICE_CHECK in the
 * device error word.  0 for the normal build, which has no such checks.
 */
int mla_testing_bounds_checked(void);

/*
 * mla_testing_bounds_shrink -- make later launches report the output buffer `out` to the
 * store checks as `bytes` smaller than it is (0 restores the true size), so that a test can
 * see the bounds-checked build catch the stores of the last rows without any store leaving
 * the real buffer.  No effect on the normal build.  Process-wide.
 */
void mla_testing_bounds_shrink(long long bytes);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_TESTING_H_ */

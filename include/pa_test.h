/*
 * Test hooks of libpa_test.so, a build of the same sources with
 * -DPA_TEST_HOOKS for the tests of failure detection.  The product library
 * (libpa.so) does not export them.
 */
#ifndef PA_TEST_H_
#define PA_TEST_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * pa_test_set_wait_fault: from the next launch of the 16-bit paged decode
 * kernel on (pa_decode, pa_decode_split, pa_decode_step), the TMA producer of
 * the CTA with linear index `cta` (x fastest over the grid (sequences, KV
 * heads, partitions); -1: none) issues no tile from its tile `tile` on: no
 * expect_tx and no copy, so no bulk copy is in flight when the CTA ends.
 * Every pipeline wait of that kernel gives up after wait_limit_ns (> 0;
 * product builds use one second), so the consumers' waits for the withheld
 * tiles run out, set PA_DEVERR_WAIT_TIMEOUT in the device error word and
 * end.  The results of that launch are not defined; the fused step's
 * counters must be zeroed again before the next step.  Returns PA_OK, or
 * PA_ERR_INVALID_ARG for a zero limit.
 */
int pa_test_set_wait_fault(int32_t cta, int32_t tile, unsigned long long wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* PA_TEST_H_ */

/*
 * pa_test.h -- test hooks of libpa.so. NOT part of the attention boundary
 * (include/pa.h): they exist so the tests can make a bounded device wait run
 * out on purpose and check that the library reports it and stays usable,
 * without faulting, trapping or hanging the GPU.
 *
 * ("P3: native paged-KV continuous-batching sampler", Review (adversarial
 *  pass): a failure must surface as an error the caller sees, not wedge the
 *  engine. Every wait inside libpa's kernels gives up after a limit, sets
 *  PA_FLAG_TIMEOUT in the status word, lets the copies it started land and
 *  returns.)
 *
 * Both settings are process-wide and are read when a call builds its launch
 * parameters: calls running concurrently in other threads see them too, so
 * set them only around a test's own calls, and put them back (a value <= 0
 * restores the default wait limit, a negative item turns the skip off).
 */
#ifndef PA_TEST_H
#define PA_TEST_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Every bounded wait of later calls' kernels gives up after `cycles` SM clock
 * cycles (default 2e9, about one second; <= 0 restores it). */
void pa_test_set_wait_cycles(int64_t cycles);

/* In later calls the bf16 split-KV kernel issues no copy for the first 16-key
 * chunk of split item `item` (items are (row, split, kv head) triples in the
 * order the kernel hands them out; item 0 is always taken), so the warp that
 * owns it waits for data that never comes, gives up after the wait limit,
 * raises PA_FLAG_TIMEOUT and leaves that item and its queued ones unfinished
 * (their rows' outputs are then unspecified). A negative item (the default)
 * turns this off. */
void pa_test_skip_split_item(int64_t item);

#ifdef __cplusplus
}
#endif

#endif /* PA_TEST_H */

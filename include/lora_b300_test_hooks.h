/*
 * lora_b300_test_hooks.h — test-only entry point of liblora_b300_testhooks.so,
 * the library built from the same sources with -DLORA_TEST_HOOKS.  The product
 * library (liblora_b300.so) does not export it; the pages have no counterpart.
 *
 * Every device-side wait of the library is bounded and, past its limit,
 * records LORA_DEVSTAT_TIMEOUT in the call's status word and unwinds.  This
 * hook lets a test make one such wait run out without faulting anything: the
 * stream-K rank pass's flag wait (a finisher CTA polling another CTA's flag
 * in global memory, with no copy of its own in flight).
 */
#ifndef LORA_B300_TEST_HOOKS_H
#define LORA_B300_TEST_HOOKS_H

#include "lora_b300.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Set, on the current device, the limit of the stream-K flag wait in
 * nanoseconds (the product value is 1e9) and the index of one CTA of every
 * later stream-K launch that parks its partial without raising its flag
 * (-1: none).  Synchronous; LORA_ERR_CUDA if the device symbols cannot be
 * written. */
lora_status_t lora_test_stream_k_hooks(unsigned long long wait_limit_ns, int skip_flag_cta);

#ifdef __cplusplus
}
#endif

#endif /* LORA_B300_TEST_HOOKS_H */

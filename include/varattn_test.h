/*
 * varattn test hooks -- for the library's own test-suite, not for users.
 *
 * The host code of libvarattn reaches the CUDA runtime only through one
 * internal function table.  These hooks swap that table for a mock that fakes
 * a device (device 0, 148 SMs), runs no kernel, and counts its calls; the call
 * whose count equals fail_at returns a CUDA error.  A test can so drive every
 * VAR_ERR_CUDA branch of the C ABI on a machine without a GPU: count the calls
 * an entry point makes with fail_at = 0, then make each of them fail in turn.
 *
 * While the mock is on, the library's per-device caches (status-word address,
 * SM count, kernel attributes) are neither read nor filled.  Turn it on only in
 * a process that makes no real CUDA call through this library.
 */
#ifndef VARATTN_TEST_H
#define VARATTN_TEST_H

#include <stdint.h>

#include "varattn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* enable != 0: use the mock and reset its call count; fail_at > 0 makes the
 * fail_at-th call (1-based) fail, 0 never.  enable = 0 restores the runtime.
 * Returns VAR_OK. */
VAR_API int var_test_mock_cuda(int32_t enable, int64_t fail_at);

/* Mock calls made since the last var_test_mock_cuda. */
VAR_API int64_t var_test_mock_calls(void);

#ifdef __cplusplus
}
#endif

#endif /* VARATTN_TEST_H */

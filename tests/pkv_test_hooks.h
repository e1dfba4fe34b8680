/*
 * pkv_test_hooks.h - entry points that exist only in test builds of libpagedkv (compiled with
 * -DPKV_TEST_HOOKS; tests/test_gpu_failure.py builds that variant next to the product library).
 * The product library neither exports them nor carries the checks they drive.
 */
#ifndef PKV_TEST_HOOKS_H
#define PKV_TEST_HOOKS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* In the attention launches that follow (process-wide), every CTA's producer skips its tile
   `tile` (0-based within the CTA's block list): it neither loads it nor signals it, so the
   consumer's bounded wait on it expires (PKV_FLAG_TIMEOUT) and the CTA takes its abort path --
   drain, void result, release, return -- with no fault and no hang.  -1 switches it off (the
   default); returns the previous value.  Results are void while it is set. */
int64_t pkv_debug_withhold_tile(int64_t tile);

#ifdef __cplusplus
}
#endif
#endif /* PKV_TEST_HOOKS_H */

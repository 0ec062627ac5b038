/*
 * moe_test_hooks.h -- the one extra function of the test build of the library,
 * libmoe_b300_testhooks.so (the same sources compiled with MOE_TEST_HOOKS). The
 * product library, libmoe_b300.so, does not export it. The pages have no
 * counterpart: it exists so that a test can make a device-side bounded wait give up
 * without faulting or hanging the GPU.
 *
 * moe_test_withhold_gemm_load(kchunk): from the next launch on, the bf16 expert
 * GEMM on single-CTA (128-row) tiles has its first CTA withhold the TMA loads of
 * k-chunk `kchunk` (64 elements of K) of its first work item, and the expected byte
 * count of that stage. The MMA thread's wait on that stage gives up after its time
 * limit (2 s), the kernel sets status bit 1 and returns after draining what it issued;
 * the call then reports MOE_EDEVICE through moe_get_status. -1 (the initial value)
 * withholds nothing. Not thread-safe; call it between launches.
 */
#ifndef MOE_B300_TEST_HOOKS_H
#define MOE_B300_TEST_HOOKS_H

#ifdef __cplusplus
extern "C" {
#endif

void moe_test_withhold_gemm_load(int kchunk);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_TEST_HOOKS_H */

/*
 * fa_selftest.h -- self-test of the library's bounded on-device waits.
 *
 * Not part of the attention computation: this entry point lets a test
 * exercise the failure path that every kernel of the library shares (a
 * bounded mbarrier wait that runs out, sets the device status word and
 * returns) without faulting or hanging the GPU.
 */
#ifndef FA_SELFTEST_H_
#define FA_SELFTEST_H_

#include "fa.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * fa_selftest_wait_timeout -- enqueue one small kernel whose threads wait on
 * an mbarrier phase that nothing completes, with the kernels' own bounded
 * wait and a limit of timeout_ns (1 us .. 1 s).  The wait gives up, records
 * a timeout in the device status word and the kernel returns; a following
 * fa_last_device_error() then reports FA_ERR_DEVICE_TIMEOUT (and clears it).
 * Returns FA_ERR_SHAPE for a limit out of range, FA_ERR_CUDA if the launch
 * fails.
 */
FA_API fa_status fa_selftest_wait_timeout(unsigned long long timeout_ns,
                                          fa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_SELFTEST_H_ */

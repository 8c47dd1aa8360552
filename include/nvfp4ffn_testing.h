/*
 * nvfp4ffn_testing.h -- testing hooks of libnvfp4ffn.so.  Not part of the
 * decode API: they exist so that a test suite can exercise paths that normal
 * inputs never reach.  The pages have no counterpart of them.
 */
#ifndef NVFP4FFN_TESTING_H
#define NVFP4FFN_TESTING_H

#include "nvfp4ffn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Process-wide switch for testing the bounded waits.  With enable != 0, every
 * later nvfp4_gemv / ffn_gate_up_nvfp4 / ffn_swiglu_nvfp4(_noalloc) launch
 * runs with a producer that issues no weight copies, and with its bounded
 * waits limited to wait_limit_ns (1000 .. 1e9 ns, else NVFP4_ERR_RANGE): each
 * consumer's first wait runs out, the kernel sets its device status word and
 * returns, and the call's outputs are left unwritten.  The kernel still ends
 * every wait and leaves no copy in flight.  enable == 0 restores normal
 * operation (1 s limit).  Not synchronised with launches on other threads.
 */
nvfp4_status nvfp4_testing_inject_stall(int enable, unsigned long long wait_limit_ns);

/*
 * Host-only check of the GEMV kernel's shared-memory plan for a problem
 * (streams = 1: one projection [N, K]; 2: the gate/up pair [N = I, K = H]) on
 * a device with num_sms SMs: 1 if every offset has the alignment the kernel's
 * accesses assume and the plan fits the per-block limit, 0 if not (such a
 * launch is refused), -1 for invalid arguments.  Needs no GPU.
 */
int nvfp4_testing_plan_aligned(int streams, int M, int N, int K, int num_sms);
/* The same check for the block-scaled FP8 kernels (w8a16_gemv, ffn_swiglu_w8a16). */
int nvfp4_testing_plan_aligned_w8a16(int streams, int M, int N, int K, int num_sms);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4FFN_TESTING_H */

/*
 * bsa_selftest.h - self-test entry points of libbsa.so.  They check two
 * building blocks of bsa_forward on the device and are meant for test
 * suites, not for the attention path.  Conventions as in bsa.h.
 */
#ifndef BSA_SELFTEST_H
#define BSA_SELFTEST_H

#include <stdint.h>

#include "bsa.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * bsa_selftest_exp2 - evaluate, for each x[i] (device fp32 [n]), the three
 * 2^x used or mirrored by the softmax: y_fma (the FMA-pipe polynomial that
 * bsa_forward uses for part of its exponentials: Cody-Waite reduction plus a
 * fitted degree-3 minimax polynomial), y_mufu (the hardware ex2.approx) and
 * y_ref (CUDA's exp2f).  All outputs device fp32 [n].  The polynomial is
 * specified for -125 <= x <= 127 (below, clamped to -125).
 */
bsa_status bsa_selftest_exp2(const float* x, float* y_fma, float* y_mufu, float* y_ref, int64_t n,
                             void* stream);

/*
 * bsa_selftest_wait_timeout - launch one thread that waits, bounded by
 * limit_ns (1 us .. 1 s), on an mbarrier that nothing completes, using the
 * same bounded wait as bsa_forward.  When the limit expires the kernel
 * records BSA_ERR_TIMEOUT in the device status word and returns; read it with
 * bsa_device_status().  Nothing faults, traps or hangs.
 */
bsa_status bsa_selftest_wait_timeout(int64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BSA_SELFTEST_H */

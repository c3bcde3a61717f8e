/*
 * gdn_testing.h -- test hooks of libgdn.  Not for production use: they exist so that tests can
 * drive the failure paths of the kernels without faulting or hanging a GPU.
 *
 * Failure detection in the tensor-core kernels of the chunked prefill works through bounded
 * waits: every wait on an mbarrier (a tensor-core product or a bulk copy completing) gives up
 * after a wall-clock limit, ORs GDN_STATUS_WAIT_TIMEOUT into the call's status word, waits (again
 * with the limit) for the products and copies that block still has in flight, frees its tensor
 * memory and returns ("[XE2] Support MTP of QWEN model", review notes: problems are reported,
 * never undefined behaviour).  The hook below makes one of those waits run out on purpose.
 */
#ifndef GDN_TESTING_H
#define GDN_TESTING_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Settings for every later launch of the chunked prefill's kernels in this process (all
 * devices, all host threads; a launch reads them when it is enqueued):
 *   wait_ns          wall-clock limit of each bounded wait, in nanoseconds of the GPU's global
 *                    timer; 0 restores the default of one second;
 *   drop_copy_chunk  a chunk index whose record the scan kernel does not copy in (no copy and
 *                    no expected byte count is issued for it), so that the wait for that chunk
 *                    runs out with nothing in flight; < 0 for none (the default).
 * A row whose wait ran out produces no outputs past that chunk and stores no state.  Always
 * returns 0 (GDN_OK).  Reset with gdn_testing_set_prefill_faults(0, -1).
 */
int gdn_testing_set_prefill_faults(uint64_t wait_ns, int32_t drop_copy_chunk);

#ifdef __cplusplus
}
#endif

#endif /* GDN_TESTING_H */

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

#include "gdn.h"

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

/*
 * Which kernels gdn_mixed_batch runs for the token-recurrence rows (spec and decode rows, and
 * every non-spec row when no prefill row takes the chunked path), for every later call in this
 * process:
 *   0  by size (the default): when the layer allows it (dk = 128, dv a multiple of 32,
 *      (dv / 32) * (Hv / Hk) in {4, 8}), the batch has no chunked prefill rows and the fused
 *      kernel's grid fits in one wave of the GPU, the fused kernel (conv update and recurrence
 *      in one launch); otherwise the conv kernel, then the recurrence;
 *   1  always the conv kernel, then the recurrence;
 *   2  the fused kernel whenever the layer and batch allow it, whatever the grid size.
 * Both give the same results bit for bit; the setting only exists so that tests can run each
 * on any batch.  Returns 0, or GDN_ERR_SHAPE (-3) for another value.
 */
int gdn_testing_set_verify_path(int32_t path);

/*
 * The path gdn_mixed_batch would take for the token-recurrence rows of this batch on the current
 * device under the current setting: 1 (conv kernel, then recurrence) or 2 (fused kernel);
 * GDN_ERR_SHAPE (-3) for invalid descriptors.  Host only: reads no device memory.
 */
int gdn_testing_verify_path_of(const gdn_layer_desc* layer, const gdn_rows* non_spec, int32_t num_prefills,
                               const gdn_rows* spec);

#ifdef __cplusplus
}
#endif

#endif /* GDN_TESTING_H */

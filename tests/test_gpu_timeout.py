"""Failure detection in the chunked prefill's tensor-core kernels, driven without a GPU fault.

Every wait of those kernels on an mbarrier is bounded by wall-clock time; when one runs out the
kernel ORs GDN_STATUS_WAIT_TIMEOUT into the status word, waits (bounded) for whatever that block
still has in flight, frees its tensor memory and returns ("[XE2] Support MTP of QWEN model",
review notes: problems are reported, never undefined behaviour).  The test hook in
include/gdn_testing.h leaves one chunk's record copy out on purpose, so the scan's wait for that
chunk runs out while nothing else is in flight (the forced wait is placed where every product
and copy issued before it has been waited for).  Each test checks that the call returned, that
the status says so, which outputs were written, and that a normal call right after it on the same
stream matches the oracle -- which also shows the tensor memory was freed (an allocation on the
same SMs would otherwise never succeed).
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_spec_gb300 as gdn
from gated_deltanet_linear_spec_gb300.device_batch import to_device
from gated_deltanet_linear_spec_gb300.workloads import LayerShape, RowSpec, build_batch
from tests.gpu_compare import BF16_TOL, assert_parity, run_gpu
from tests.oracle_run import act_to_f64, np_act, run_oracle

pytestmark = pytest.mark.gpu

SHORT_WAIT_NS = 20_000_000  # 20 ms instead of the default second


def prefill_batch(length: int, seed: int):
    layer = LayerShape(1, 2, 128, 128, 4, 3, torch.bfloat16)
    return build_batch(layer, [RowSpec("prefill", length)], num_slots=8, seed=seed)


@pytest.fixture
def faults():
    def set_faults(wait_ns, drop_chunk):
        gdn.gdn_testing_set_prefill_faults(wait_ns, drop_chunk)
    yield set_faults
    gdn.gdn_testing_set_prefill_faults(0, -1)


@pytest.mark.parametrize("length,drop", [(50, 0), (200, 2)])
def test_a_wait_that_runs_out_is_reported_and_the_next_call_is_clean(faults, length, drop):
    batch = prefill_batch(length, seed=70 + drop)
    db = to_device(batch)
    ssm_before = db.pools.ssm_pool.clone()
    faults(SHORT_WAIT_NS, drop)
    db.run()  # returns normally: the failure is only visible in the status word
    torch.cuda.synchronize()
    faults(0, -1)
    assert int(db.status.item()) & gdn.STATUS_WAIT_TIMEOUT
    # no final state for the row; its slot (and every other one) keeps its prior bits
    assert torch.equal(db.pools.ssm_pool, ssm_before)
    out = act_to_f64(np_act(db.out.cpu()))
    ref = run_oracle(batch)
    # the chunks before the one whose record never came had their outputs stored up to one
    # chunk behind (a chunk's outputs leave while the next chunk runs); nothing from the dropped
    # chunk on was written
    done = 64 * max(0, drop - 1)
    assert np.all(out[done:] == 0.0)
    if done:
        r = ref.out_f64[:done]
        assert np.all(np.abs(out[:done] - r) <= BF16_TOL + BF16_TOL * np.abs(r))
    # the next call on the same stream, with the default limit and no copy left out
    gpu = run_gpu(batch)
    assert_parity(batch, gpu, ref)


def test_a_short_limit_alone_changes_nothing(faults):
    faults(SHORT_WAIT_NS, -1)  # a short limit alone changes nothing when every copy arrives
    batch = prefill_batch(200, seed=75)
    gpu = run_gpu(batch)
    assert_parity(batch, gpu, run_oracle(batch))

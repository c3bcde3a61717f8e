"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the named workloads.

Every workload runs the whole path (gdn_mixed_batch) once on the GPU and once in the oracle on
the same seeded inputs, then compares outputs and states within the stated tolerances, the conv
ring bit for bit, and the set of written slots exactly.
"""
import pytest
import torch

from gated_deltanet_linear_spec_gb300 import workloads as W
from tests.gpu_compare import assert_parity, run_gpu
from tests.oracle_run import run_oracle

pytestmark = pytest.mark.gpu


def _parity(batch, heads=None):
    gpu = run_gpu(batch)
    ref = run_oracle(batch, heads=heads)
    worst = assert_parity(batch, gpu, ref, heads)
    torch.cuda.empty_cache()
    return worst


def test_tiny():
    _parity(W.tiny())


@pytest.mark.parametrize("seed", [0, 1, 2, 3, 4, 5])
def test_tiny_seeds(seed):
    _parity(W.tiny(seed))


def test_non_spec_decode():
    _parity(W.non_spec_decode())


def test_spec_verify():
    _parity(W.spec_verify())


def test_mixed():
    _parity(W.mixed())


@pytest.mark.parametrize("batch", [1, 8, 64, 256, 512])
@pytest.mark.parametrize("drafts", [1, 2, 4])
def test_sweep_point(drafts, batch):
    # full-size inputs and launch; the oracle recomputes eight of the 32 v-heads (a different
    # run of eight per point, so that the points together cover every head)
    h0 = (drafts * 7 + batch * 3) % 25
    _parity(W.sweep_point(drafts, batch, seed=4 + drafts * 10 + batch), heads=(h0, h0 + 8))


def test_long_prefill():
    # every v-head of the 8192-token row (128 chunks on the tensor-core path)
    _parity(W.long_prefill(8192))

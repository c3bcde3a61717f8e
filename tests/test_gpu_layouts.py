"""GPU parity for the two alternative layouts: per-k-head x ("[GDN] Spec-decoding-aware attention
kernel", Test Plan: reorder_input=False) and per-slot conv snapshots ("[XE2] Support MTP of QWEN
model", review thread on the conv state layout), each against the oracle, plus the per-k-head
path against the packed path on the GPU (only load addresses differ, so bit for bit)."""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_spec_gb300 import workloads as W
from gated_deltanet_linear_spec_gb300.workloads import RowSpec, build_batch, uniform_accepts, with_layouts
from tests.gpu_compare import assert_parity, run_gpu
from tests.oracle_run import run_oracle

pytestmark = pytest.mark.gpu


def _parity(batch, heads=None):
    gpu = run_gpu(batch)
    assert_parity(batch, gpu, run_oracle(batch, heads=heads), heads)
    torch.cuda.empty_cache()
    return gpu


@pytest.mark.parametrize("qkv,conv", [(1, 0), (0, 1), (1, 1)])
def test_mixed_small_layouts(qkv, conv):
    _parity(with_layouts(W.mixed_small(8), qkv_layout=qkv, conv_layout=conv))


@pytest.mark.parametrize("qkv,conv", [(1, 0), (0, 1)])
def test_tiny_layouts(qkv, conv):
    _parity(with_layouts(W.tiny(3), qkv_layout=qkv, conv_layout=conv))


def test_spec_verify_per_slot():
    _parity(with_layouts(W.spec_verify(seed=12), conv_layout=1), heads=(9, 11))


def test_per_slot_more_drafts_than_the_rolled_ring_holds():
    # state_len = W - 1 = 3 with 6 verify tokens per row: only the per-slot layout accepts it
    k = 6
    acc = uniform_accepts(64, k, 77)
    rows = [RowSpec("spec", k if i % 9 else k - 3, min(acc[i], k if i % 9 else k - 3)) for i in range(64)]
    b = build_batch(W.big_layer(3), rows, num_slots=512, spec_cols=k, seed=78, null_frac=0.05)
    _parity(with_layouts(b, conv_layout=1), heads=(20, 22))


def test_per_khead_equals_packed_bit_for_bit():
    b = W.spec_verify(seed=13)
    packed = run_gpu(b)
    per_khead = run_gpu(with_layouts(b, qkv_layout=1))
    assert packed.status == 0 and per_khead.status == 0
    assert np.array_equal(packed.out, per_khead.out)
    assert np.array_equal(packed.conv_pool, per_khead.conv_pool)
    assert np.array_equal(packed.ssm_pool.view(np.uint32), per_khead.ssm_pool.view(np.uint32))


def test_long_prefill_per_khead():
    # the chunked path reads the post-conv q|k|v, which is packed in both layouts
    _parity(with_layouts(W.long_prefill(1000), qkv_layout=1), heads=(4, 6))

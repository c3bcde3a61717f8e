"""The fused verify kernel (conv update and gated delta rule in one launch) against the
two-kernel path and the oracle.

gdn_mixed_batch runs the recurrence rows of small batches (one wave of the GPU) on layers with
dk = 128 through one kernel whose CTAs of a (row, k-head) form a thread-block cluster and
exchange the q|k conv outputs through distributed shared memory; larger batches take the conv
kernel and then the recurrence.  The test hook in include/gdn_testing.h forces either path, so
every batch here runs both ways: the results must agree bit for bit (the same fp32 conv outputs
feed the same recurrence arithmetic), and the fused results must match the oracle within the
stated tolerances.  Covered: clusters of 8 (two v-heads per k-head, four dv tiles) and of 4 (one
v-head per k-head, or dv = 64), conv widths 2-4 with a bias, fp32 activations (prefill rows then
run the token recurrence, many token batches per row), the per-k-head x layout, the per-slot conv
layout, acceptance-aware rows, spec rows longer than one token batch, ragged rows, NULL slots,
the metric's full batch, and the automatic choice at one wave.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_spec_gb300 as gdn
import gated_deltanet_linear_spec_gb300.device_batch  # noqa: F401
from gated_deltanet_linear_spec_gb300 import workloads as W
from gated_deltanet_linear_spec_gb300.workloads import LayerShape, RowSpec, build_batch, with_layouts
from tests.gpu_compare import assert_parity, run_gpu
from tests.oracle_run import run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture
def path():
    yield gdn.gdn_testing_set_verify_path
    gdn.gdn_testing_set_verify_path(0)


def check(batch, path):
    path(2)
    fused = run_gpu(batch)
    path(1)
    two = run_gpu(batch)
    assert np.array_equal(fused.out, two.out), "outputs differ from the two-kernel path"
    assert np.array_equal(fused.conv_pool, two.conv_pool), "conv ring differs from the two-kernel path"
    assert np.array_equal(fused.ssm_pool.view(np.uint32), two.ssm_pool.view(np.uint32)), "states differ"
    assert_parity(batch, fused, run_oracle(batch))


def test_spec_verify_big_layer(path):
    # the metric's batch: clusters of 8 (2 v-heads x 4 dv tiles per k-head), width 4, 5% NULL
    check(W.spec_verify(), path)


@pytest.mark.parametrize("width", [2, 3, 4])
def test_cluster_of_four_one_v_head_per_k_head(width, path):
    layer = LayerShape(2, 2, 128, 128, width, width - 2 + 5, torch.bfloat16)
    rows = [RowSpec("spec", 5, 1 + i % 5) for i in range(5)] + [RowSpec("spec", 2, 2), RowSpec("decode", 1),
                                                                RowSpec("decode", 1, has_initial_state=False)]
    check(build_batch(layer, rows, num_slots=64, spec_cols=5, seed=110 + width, shuffle_from=0,
                      spec_nulls=[(0, 2), (3, 0)], conv_bias=True), path)


def test_cluster_of_four_with_dv_64(path):
    layer = LayerShape(1, 2, 128, 64, 4, 6, torch.bfloat16)
    rows = [RowSpec("spec", 4, 3), RowSpec("spec", 4, 1), RowSpec("decode", 1), RowSpec("prefill", 40)]
    check(build_batch(layer, rows, num_slots=24, spec_cols=4, seed=117, shuffle_from=0), path)


def test_long_spec_rows_span_several_token_batches(path):
    layer = LayerShape(1, 2, 128, 128, 4, 2 + 20, torch.bfloat16)
    rows = [RowSpec("spec", 20, 7), RowSpec("spec", 13, 20), RowSpec("spec", 9, 1), RowSpec("decode", 1)]
    check(build_batch(layer, rows, num_slots=80, spec_cols=20, seed=118, shuffle_from=0, spec_nulls=[(0, 9)]), path)


def test_fp32_layer_runs_prefill_rows_through_the_fused_kernel(path):
    layer = LayerShape(2, 4, 128, 128, 4, 6, torch.float32)
    rows = [RowSpec("spec", 4, 2), RowSpec("decode", 1), RowSpec("prefill", 100),
            RowSpec("prefill", 17, has_initial_state=False)]
    check(build_batch(layer, rows, num_slots=32, spec_cols=4, seed=119, shuffle_from=0), path)


@pytest.mark.parametrize("qkv_layout,conv_layout", [(1, 0), (0, 1), (1, 1)])
def test_layouts(qkv_layout, conv_layout, path):
    base = build_batch(LayerShape(2, 4, 128, 128, 4, 6, torch.bfloat16),
                       [RowSpec("spec", 4, 1 + i % 4) for i in range(6)] + [RowSpec("decode", 1)],
                       num_slots=64, spec_cols=4, seed=120, shuffle_from=0, spec_nulls=[(1, 1)])
    check(with_layouts(base, qkv_layout=qkv_layout, conv_layout=conv_layout), path)


def test_acceptance_aware_rows(path):
    layer = LayerShape(1, 2, 128, 128, 4, 6, torch.bfloat16)
    rows = [RowSpec("spec", 4, 2), RowSpec("decode", 1, num_accepted=3, aware=True),
            RowSpec("decode", 1, num_accepted=1, aware=True), RowSpec("decode", 1, num_accepted=4, aware=True)]
    check(build_batch(layer, rows, num_slots=48, spec_cols=4, seed=121, shuffle_from=0), path)


def test_one_wave_batches_take_the_fused_kernel_by_default(path):
    # 8 rows x 32 v-heads x 4 dv tiles = 1024 CTAs: one wave on the GB300's SMs, so the default
    # choice is the fused kernel; its results equal the forced two-kernel path bit for bit
    batch = W.spec_verify(batch=8)
    d = gdn.device_batch.to_device(batch)
    assert gdn.gdn_testing_verify_path_of(d.layer, d.non_spec, d.num_prefills, d.spec) == 2
    big = gdn.device_batch.to_device(W.spec_verify())
    assert gdn.gdn_testing_verify_path_of(big.layer, big.non_spec, big.num_prefills, big.spec) == 1
    del d, big
    path(0)
    auto = run_gpu(batch)
    path(1)
    two = run_gpu(batch)
    assert np.array_equal(auto.out, two.out) and np.array_equal(auto.conv_pool, two.conv_pool)
    assert np.array_equal(auto.ssm_pool.view(np.uint32), two.ssm_pool.view(np.uint32))
    assert_parity(batch, auto, run_oracle(batch))

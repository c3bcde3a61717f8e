"""GPU parity for acceptance-aware non-spec rows ("[Bugfix] Align Qwen GDN gates with speculative
tokens", the second mechanism in the reachability comment: a verify row cut to a prefix by the
batch budget and scheduled as a plain row, continuing from what its previous verify step
accepted).  Decode rows run in the token recurrence, prefill rows in the chunked tensor-core
path; both conv layouts."""
import copy

import numpy as np
import pytest
import torch

import gated_deltanet_linear_spec_gb300 as gdn
from gated_deltanet_linear_spec_gb300 import workloads as W
from gated_deltanet_linear_spec_gb300.workloads import LayerShape, RowSpec, build_batch, uniform_accepts, with_layouts
from tests.gpu_compare import assert_outputs_close, assert_parity, run_gpu
from tests.oracle_run import np_act, run_oracle

pytestmark = pytest.mark.gpu

LAYER = LayerShape(1, 2, 128, 128, 4, 6, torch.bfloat16)


def _mixed_aware(seed):
    acc = uniform_accepts(8, 4, seed)
    rows = [RowSpec("decode", 1, acc[0], aware=True), RowSpec("decode", 1),
            RowSpec("decode", 1, acc[1], aware=True), RowSpec("decode", 1, acc[2], has_initial_state=False, aware=True)]
    rows += [RowSpec("spec", 4 if i != 1 else 3, acc[3 + i]) for i in range(4)]
    rows += [RowSpec("prefill", 70, acc[7], aware=True), RowSpec("prefill", 130, 3, has_initial_state=False, aware=True),
             RowSpec("prefill", 65)]
    return build_batch(LAYER, rows, num_slots=96, spec_cols=4, seed=seed, shuffle_from=4, spec_nulls=[(2, 1)])


@pytest.mark.parametrize("conv_layout", [0, 1])
@pytest.mark.parametrize("seed", [31, 32])
def test_mixed_batch_with_aware_rows(seed, conv_layout):
    b = with_layouts(_mixed_aware(seed), conv_layout=conv_layout)
    assert b.non_spec.num_accepted_tokens is not None and not b.non_spec.is_spec
    assert_parity(b, run_gpu(b), run_oracle(b))


def test_aware_decode_rows_big_layer():
    acc = uniform_accepts(96, 4, 5)
    rows = [RowSpec("decode", 1, acc[i], aware=True) for i in range(64)]
    rows += [RowSpec("spec", 4, acc[64 + i]) for i in range(32)]
    b = build_batch(W.big_layer(6), rows, num_slots=512, spec_cols=4, seed=6, shuffle_from=0)
    assert_parity(b, run_gpu(b), run_oracle(b, heads=(7, 9)), heads=(7, 9))


def test_aware_row_with_bad_num_accepted_is_skipped():
    b = _mixed_aware(33)
    bad = copy.copy(b)
    bad.non_spec = copy.copy(b.non_spec)
    na = b.non_spec.num_accepted_tokens.clone()
    na[0] = 0                    # the first decode row (aware)
    na[b.num_decodes] = 9        # the first prefill row (aware, chunked path)
    bad.non_spec.num_accepted_tokens = na
    gpu = run_gpu(bad)
    assert gpu.status & gdn.STATUS_NUM_ACCEPTED
    ref = run_oracle(b)          # the same batch with valid acceptance
    ns = b.non_spec
    q = ns.query_start_loc.tolist()
    tok = ns.token_indx if ns.token_indx is not None else torch.arange(ns.num_tokens)
    mask = np.ones(b.num_actual_tokens, bool)
    skipped_tokens = []
    for r in (0, b.num_decodes):
        skipped_tokens += tok[q[r]: q[r + 1]].tolist()
    mask[skipped_tokens] = False
    assert_outputs_close(gpu.out, ref, True, rows_mask=mask)
    assert (gpu.out[skipped_tokens] == 0).all()   # outputs start as zeros and stay so
    pre_ssm, pre_conv = b.ssm_pool.numpy(), np_act(b.conv_pool)
    for r in (0, b.num_decodes):
        s = int(ns.state_indices[r])
        assert np.array_equal(gpu.ssm_pool[s], pre_ssm[s])
        assert np.array_equal(gpu.conv_pool[s], pre_conv[s])

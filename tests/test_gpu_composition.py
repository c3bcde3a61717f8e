"""GPU tests of gdn_mixed_batch as the composition of the single-step entry points.

A mixed call with decode and prefill rows must be bit-identical to gdn_conv_update over the
non-spec rows (fp32 post-conv rows), then gdn_recurrent_step on the decode rows and
gdn_chunk_prefill on the prefill rows, and match the oracle: every conv width, both x layouts,
both conv layouts with acceptance-aware rows, rows shorter than the conv history, a fresh row, a
NULL slot, gathered and identity token order, and a second call continuing from the first."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_spec_gb300 as gdn
from gated_deltanet_linear_spec_gb300.device_batch import to_device
from gated_deltanet_linear_spec_gb300.workloads import LayerShape, RowSpec, build_batch, uniform_accepts
from tests.gpu_compare import assert_parity, run_gpu
from tests.oracle_run import np_act, run_oracle

pytestmark = pytest.mark.gpu

LENGTHS = [1, 2, 3, 64, 65, 130]


def _batch(width, qkv_layout, conv_layout, aware, seed):
    layer = LayerShape(1, 2, 128, 128, width, width + 3, torch.bfloat16, qkv_layout, conv_layout)
    acc = uniform_accepts(len(LENGTHS) + 1, 4, seed)
    rows = [RowSpec("decode", 1), RowSpec("decode", 1, acc[0], aware=aware)]
    rows += [RowSpec("prefill", L, acc[1 + i] if aware else 1, has_initial_state=(i != 4), aware=aware)
             for i, L in enumerate(LENGTHS)]
    # non-spec row 3 (a prefill row; their order is seeded) gets a NULL conv and state slot
    return build_batch(layer, rows, num_slots=48, spec_cols=4 if aware else 0, seed=seed, shuffle_from=2,
                       non_spec_nulls=[3], conv_bias=(seed % 2 == 0), force_token_indx=True)


def _sl(t, lo, hi):
    return None if t is None else t[lo:hi].contiguous()


def _separate_calls(batch):
    """Conv kernel over every non-spec row, then the token recurrence on the decode rows and the
    chunked prefill on the prefill rows."""
    d = to_device(batch)
    ns, nd = d.non_spec, batch.num_decodes
    y = torch.empty((ns.num_tokens, batch.layer.channels), dtype=torch.float32, device="cuda")
    gdn.gdn_conv_update(d.layer, d.params, d.pools, d.x, ns, y, d.status)
    q = ns.query_start_loc
    split = int(q[nd])
    if nd:
        dec = gdn.Rows(q[: nd + 1].contiguous(), split, _sl(ns.token_indx, 0, split), _sl(ns.state_indices, 0, nd),
                       _sl(ns.has_initial_state, 0, nd), _sl(ns.spec_state_indices, 0, nd),
                       _sl(ns.num_accepted_tokens, 0, nd))
        gdn.gdn_recurrent_step(d.layer, d.params, d.pools, y[:split].contiguous(), d.a, d.b, dec, d.out, d.status)
    n = ns.num_seqs
    pre = gdn.Rows((q[nd:] - split).contiguous(), ns.num_tokens - split, _sl(ns.token_indx, split, ns.num_tokens),
                   _sl(ns.state_indices, nd, n), _sl(ns.has_initial_state, nd, n), _sl(ns.spec_state_indices, nd, n),
                   _sl(ns.num_accepted_tokens, nd, n))
    gdn.gdn_chunk_prefill(d.layer, d.params, d.pools, y[split:].contiguous(), d.a, d.b, pre, d.out, status=d.status)
    torch.cuda.synchronize()
    return d


def _assert_mixed_equals_separate(batch):
    mixed = run_gpu(batch)
    assert mixed.status == 0, f"device status {mixed.status:#x}"
    d = _separate_calls(batch)
    assert int(d.status.item()) == 0
    assert np.array_equal(np_act(d.out.cpu()), mixed.out), "outputs differ"
    assert np.array_equal(np_act(d.pools.conv_pool.cpu()), mixed.conv_pool), "conv slots differ"
    assert np.array_equal(d.pools.ssm_pool.cpu().numpy().view(np.uint32), mixed.ssm_pool.view(np.uint32)), \
        "states differ"
    return mixed


@pytest.mark.parametrize("layouts", [(0, False), (0, True), (1, True)], ids=["rolled", "rolled-aware", "per-slot-aware"])
@pytest.mark.parametrize("qkv_layout", [0, 1], ids=["packed", "per-khead"])
@pytest.mark.parametrize("width", [2, 3, 4])
def test_mixed_call_equals_conv_then_recurrence_and_prefill(width, qkv_layout, layouts):
    conv_layout, aware = layouts
    batch = _batch(width, qkv_layout, conv_layout, aware, seed=40 + 7 * width + 3 * qkv_layout + conv_layout)
    mixed = _assert_mixed_equals_separate(batch)
    assert_parity(batch, mixed, run_oracle(batch))


def test_prefill_row_in_identity_token_order():
    """One 200-token row in identity order (no token_indx) continuing a prior state, then the
    same row in a second call: the rolled slot of the first call is the second call's history."""
    layer = LayerShape(1, 2, 128, 128, 4, 3, torch.bfloat16)
    batch = build_batch(layer, [RowSpec("prefill", 200)], num_slots=4, seed=51)
    assert batch.non_spec.token_indx is None
    mixed = _assert_mixed_equals_separate(batch)
    assert_parity(batch, mixed, run_oracle(batch))
    d = to_device(batch)
    for _ in range(2):
        d.run()
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    ref = run_oracle(batch)
    ref2 = run_oracle(batch, conv_pool=ref.conv_pool, ssm_pool=ref.ssm_pool)
    assert np.array_equal(np_act(d.pools.conv_pool.cpu()), ref2.conv_pool)

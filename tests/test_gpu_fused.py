"""The fused verify kernel (conv update and gated delta rule in one launch) against the
two-kernel path and the oracle.

gdn_mixed_batch runs the spec and decode rows of layers with dk = 128 through one kernel whose
CTAs of a (row, k-head) form a thread-block cluster and exchange the q|k conv outputs through
distributed shared memory.  The separate entry points (gdn_conv_update into an fp32 buffer, then
gdn_recurrent_step, and gdn_chunk_prefill for prefill rows) compute the same thing in two
launches; the results must agree bit for bit (the same fp32 conv outputs feed the same
recurrence arithmetic), and both must match the oracle within the stated tolerances.  Covered:
clusters of 8 (two v-heads per k-head, four dv tiles) and of 4 (one v-head per k-head, or dv =
64), conv widths 2-4, fp32 activations (prefill rows then run the token recurrence inside the
fused kernel, many token batches per row), the per-k-head x layout, the per-slot conv layout,
acceptance-aware rows, spec rows longer than one token batch, ragged rows and NULL slots.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_spec_gb300 as gdn
from gated_deltanet_linear_spec_gb300 import workloads as W
from gated_deltanet_linear_spec_gb300.device_batch import to_device
from gated_deltanet_linear_spec_gb300.workloads import LayerShape, RowSpec, build_batch, with_layouts
from tests.gpu_compare import assert_parity, run_gpu
from tests.oracle_run import np_act, run_oracle

pytestmark = pytest.mark.gpu


def two_kernel_path(batch):
    """The batch through the separate entry points: conv per subset into fp32, the token
    recurrence on the spec rows and the decode rows (every non-spec row when the layer has no
    chunked path), the chunked prefill on the prefill rows."""
    d = to_device(batch)
    C = batch.layer.channels
    chunked = batch.layer.act_dtype == torch.bfloat16 and batch.layer.head_k_dim == 128 \
        and batch.layer.head_v_dim == 128
    ys = {}
    for name in ("spec", "non_spec"):
        rows = getattr(d, name)
        if rows is None:
            continue
        ys[name] = torch.empty((rows.num_tokens, C), dtype=torch.float32, device="cuda")
        gdn.gdn_conv_update(d.layer, d.params, d.pools, d.x, rows, ys[name], d.status)
    if d.spec is not None:
        gdn.gdn_recurrent_step(d.layer, d.params, d.pools, ys["spec"], d.a, d.b, d.spec, d.out, d.status)
    ns = d.non_spec
    if ns is not None:
        nd = batch.num_decodes if chunked else ns.num_seqs
        q = ns.query_start_loc
        split = int(q[nd])

        def part(lo, hi, t0, t1):
            cut = lambda t: None if t is None else t[lo:hi].contiguous()  # noqa: E731
            ssi = None if ns.spec_state_indices is None else ns.spec_state_indices[lo:hi].contiguous()
            return gdn.Rows((q[lo:hi + 1] - t0).contiguous(), t1 - t0, ns.token_indx[t0:t1].contiguous()
                            if ns.token_indx is not None else None, cut(ns.state_indices), cut(ns.has_initial_state),
                            ssi, cut(ns.num_accepted_tokens))

        if nd:
            gdn.gdn_recurrent_step(d.layer, d.params, d.pools, ys["non_spec"][:split].contiguous(), d.a, d.b,
                                   part(0, nd, 0, split), d.out, d.status)
        if nd < ns.num_seqs:
            gdn.gdn_chunk_prefill(d.layer, d.params, d.pools, ys["non_spec"][split:].contiguous(), d.a, d.b,
                                  part(nd, ns.num_seqs, split, ns.num_tokens), d.out, status=d.status)
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    return np_act(d.out.cpu()), np_act(d.pools.conv_pool.cpu()), d.pools.ssm_pool.cpu().numpy()


def check(batch):
    fused = run_gpu(batch)
    out, conv, ssm = two_kernel_path(batch)
    assert np.array_equal(fused.out, out), "outputs differ from the two-kernel path"
    assert np.array_equal(fused.conv_pool, conv), "conv ring differs from the two-kernel path"
    assert np.array_equal(fused.ssm_pool.view(np.uint32), ssm.view(np.uint32)), "states differ"
    assert_parity(batch, fused, run_oracle(batch))


def test_spec_verify_big_layer():
    # the metric's batch: clusters of 8 (2 v-heads x 4 dv tiles per k-head), width 4, 5% NULL
    check(W.spec_verify(batch=16))


@pytest.mark.parametrize("width", [2, 3, 4])
def test_cluster_of_four_one_v_head_per_k_head(width):
    layer = LayerShape(2, 2, 128, 128, width, width - 2 + 5, torch.bfloat16)
    rows = [RowSpec("spec", 5, 1 + i % 5) for i in range(5)] + [RowSpec("spec", 2, 2), RowSpec("decode", 1),
                                                                RowSpec("prefill", 70)]
    check(build_batch(layer, rows, num_slots=64, spec_cols=5, seed=110 + width, shuffle_from=0,
                      spec_nulls=[(0, 2), (3, 0)], conv_bias=True))


def test_cluster_of_four_with_dv_64():
    layer = LayerShape(1, 2, 128, 64, 4, 6, torch.bfloat16)
    rows = [RowSpec("spec", 4, 3), RowSpec("spec", 4, 1), RowSpec("decode", 1), RowSpec("prefill", 40)]
    check(build_batch(layer, rows, num_slots=24, spec_cols=4, seed=117, shuffle_from=0))


def test_long_spec_rows_span_several_token_batches():
    layer = LayerShape(1, 2, 128, 128, 4, 2 + 20, torch.bfloat16)
    rows = [RowSpec("spec", 20, 7), RowSpec("spec", 13, 20), RowSpec("spec", 9, 1), RowSpec("decode", 1)]
    check(build_batch(layer, rows, num_slots=80, spec_cols=20, seed=118, shuffle_from=0, spec_nulls=[(0, 9)]))


def test_fp32_layer_runs_prefill_rows_through_the_fused_kernel():
    layer = LayerShape(2, 4, 128, 128, 4, 6, torch.float32)
    rows = [RowSpec("spec", 4, 2), RowSpec("decode", 1), RowSpec("prefill", 100),
            RowSpec("prefill", 17, has_initial_state=False)]
    check(build_batch(layer, rows, num_slots=32, spec_cols=4, seed=119, shuffle_from=0))


@pytest.mark.parametrize("qkv_layout,conv_layout", [(1, 0), (0, 1), (1, 1)])
def test_layouts(qkv_layout, conv_layout):
    base = build_batch(LayerShape(2, 4, 128, 128, 4, 6, torch.bfloat16),
                       [RowSpec("spec", 4, 1 + i % 4) for i in range(6)] + [RowSpec("decode", 1), RowSpec("prefill", 65)],
                       num_slots=64, spec_cols=4, seed=120, shuffle_from=0, spec_nulls=[(1, 1)])
    check(with_layouts(base, qkv_layout=qkv_layout, conv_layout=conv_layout))


def test_acceptance_aware_rows():
    layer = LayerShape(1, 2, 128, 128, 4, 6, torch.bfloat16)
    rows = [RowSpec("spec", 4, 2), RowSpec("decode", 1, num_accepted=3, aware=True),
            RowSpec("decode", 1, num_accepted=1, aware=True), RowSpec("prefill", 5, num_accepted=4, aware=True)]
    check(build_batch(layer, rows, num_slots=48, spec_cols=4, seed=121, shuffle_from=0))

"""The entry point for callers that cannot allocate device memory.

gdn_mixed_batch_static_workspace runs gdn_mixed_batch with the library's own fixed device
scratch, for callers (plain C hosts, plugins inside frameworks that own every allocation, serving
loops that must not call cudaMalloc) that have no way to pass a workspace.  This file is
collected last so that a stop-at-first-failure run has already run every other test; it must
pass on its own in a fresh process as well.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_spec_gb300 as gdn
from gated_deltanet_linear_spec_gb300 import workloads as W
from gated_deltanet_linear_spec_gb300.device_batch import to_device
from tests.gpu_compare import BF16_TOL, STATE_REL
from tests.oracle_run import act_to_f64, np_act

pytestmark = pytest.mark.gpu


def _next_step_inputs(db, seed):
    """New activations and acceptance counts for a second step on the same pools."""
    g = torch.Generator().manual_seed(seed)
    T, C, Hv = db.x.shape[0], db.x.shape[1], db.a.shape[1]
    x = torch.randn((T, C), generator=g).to(db.x.dtype).cuda()
    a = torch.randn((T, Hv), generator=g).to(db.a.dtype).cuda()
    b = torch.randn((T, Hv), generator=g).to(db.b.dtype).cuda()
    na = torch.randint(1, db.spec.spec_state_indices.shape[1] + 1, (db.spec.num_seqs,), generator=g)
    return x, a, b, na.to(torch.int32).cuda()


def _assert_close(out_static, out_ref, ssm_static, ssm_ref, conv_static, conv_ref):
    g, r = act_to_f64(np_act(out_static.cpu())), act_to_f64(np_act(out_ref.cpu()))
    assert np.all(np.abs(g - r) <= BF16_TOL + BF16_TOL * np.abs(r))
    d = (ssm_static - ssm_ref).double().flatten(2).norm(dim=2)
    n = ssm_ref.double().flatten(2).norm(dim=2).clamp_min(1e-30)
    assert float((d / n).max()) <= STATE_REL
    assert torch.equal(conv_static, conv_ref)


def test_static_workspace_matches_mixed_batch_on_two_calls_in_a_row():
    batch = W.spec_verify()
    ref = to_device(batch)    # the existing entry point, with a caller-allocated workspace
    stat = to_device(batch)   # the new one, on its own copy of the pools
    assert gdn.gdn_workspace_bytes(stat.layer, stat.non_spec, stat.spec) <= gdn.STATIC_WORKSPACE_BYTES
    for call in range(2):
        if call == 1:
            x, a, b, na = _next_step_inputs(ref, seed=99)
            for d in (ref, stat):
                d.x.copy_(x); d.a.copy_(a); d.b.copy_(b); d.spec.num_accepted_tokens.copy_(na)
        ref.run()
        gdn.gdn_mixed_batch_static_workspace(stat.layer, stat.params, stat.pools, stat.x, stat.a, stat.b,
                                             stat.non_spec, stat.num_decodes, stat.num_prefills, stat.spec,
                                             stat.out, stat.status)
        torch.cuda.synchronize()
        assert int(stat.status.item()) == 0 and int(ref.status.item()) == 0
        _assert_close(stat.out, ref.out, stat.pools.ssm_pool, ref.pools.ssm_pool,
                      stat.pools.conv_pool, ref.pools.conv_pool)


def test_static_workspace_rejects_a_batch_that_does_not_fit():
    batch = W.mixed()  # 1672 tokens x 8192 fp32 channels of scratch > 16 MiB
    d = to_device(batch)
    assert gdn.gdn_workspace_bytes(d.layer, d.non_spec, d.spec) > gdn.STATIC_WORKSPACE_BYTES
    before = d.out.clone()
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_mixed_batch_static_workspace(d.layer, d.params, d.pools, d.x, d.a, d.b, d.non_spec, d.num_decodes,
                                             d.num_prefills, d.spec, d.out, d.status)
    assert e.value.name == "WORKSPACE"
    torch.cuda.synchronize()
    assert torch.equal(d.out, before)


def test_static_workspace_with_chunked_prefill_rows_matches_mixed_batch():
    # a small bf16 layer (dk = dv = 128, so prefill rows take the tensor-core path and their
    # chunk records live in the fixed array too): decode, spec and prefill rows of 70 and 130
    batch = W.mixed_small()
    ref = to_device(batch)
    stat = to_device(batch)
    need = gdn.gdn_workspace_bytes(stat.layer, stat.non_spec, stat.spec) + \
        gdn.gdn_prefill_workspace_bytes(stat.layer, stat.non_spec, stat.num_prefills)
    assert gdn.gdn_prefill_workspace_bytes(stat.layer, stat.non_spec, stat.num_prefills) > 0
    assert need <= gdn.STATIC_WORKSPACE_BYTES
    for call in range(2):
        if call == 1:
            x, a, b, na = _next_step_inputs(ref, seed=98)
            for d in (ref, stat):
                d.x.copy_(x); d.a.copy_(a); d.b.copy_(b); d.spec.num_accepted_tokens.copy_(na)
        ref.run()
        gdn.gdn_mixed_batch_static_workspace(stat.layer, stat.params, stat.pools, stat.x, stat.a, stat.b,
                                             stat.non_spec, stat.num_decodes, stat.num_prefills, stat.spec,
                                             stat.out, stat.status)
        torch.cuda.synchronize()
        assert int(stat.status.item()) == 0 and int(ref.status.item()) == 0
        _assert_close(stat.out, ref.out, stat.pools.ssm_pool, ref.pools.ssm_pool,
                      stat.pools.conv_pool, ref.pools.conv_pool)


def test_static_workspace_counts_the_prefill_records():
    # one 130-token prefill row of the 8192-channel layer: its post-conv scratch (4.3 MB) fits,
    # but with its three chunks of 32 records (15.9 MB) the batch does not
    batch = W.build_batch(W.big_layer(3), [W.RowSpec("prefill", 130)], num_slots=4, seed=12)
    d = to_device(batch)
    base = gdn.gdn_workspace_bytes(d.layer, d.non_spec, d.spec)
    assert base <= gdn.STATIC_WORKSPACE_BYTES
    assert base + gdn.gdn_prefill_workspace_bytes(d.layer, d.non_spec, d.num_prefills) > gdn.STATIC_WORKSPACE_BYTES
    out0, ssm0, conv0 = d.out.clone(), d.pools.ssm_pool.clone(), d.pools.conv_pool.clone()
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_mixed_batch_static_workspace(d.layer, d.params, d.pools, d.x, d.a, d.b, d.non_spec, d.num_decodes,
                                             d.num_prefills, d.spec, d.out, d.status)
    assert e.value.name == "WORKSPACE"
    torch.cuda.synchronize()
    assert torch.equal(d.out, out0) and torch.equal(d.pools.ssm_pool, ssm0) and torch.equal(d.pools.conv_pool, conv0)

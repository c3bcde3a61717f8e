"""Graph-padded inputs and CUDA-graph capture of the whole path (SURVEY "next" row 1; the pages:
"[GDN] Spec-decoding-aware attention kernel", Related issues -- the size(0) == num_actual_tokens
precondition under piecewise graph capture; "[XE2] Support MTP of QWEN model" -- graph-padded spec
metadata).  The library never reads device memory on the host, synchronises or allocates, so
gdn_mixed_batch can be captured once and replayed with new inputs; padded rows (no tokens, NULL
slots) and padded token rows past num_actual_tokens are left alone."""
import copy

import numpy as np
import pytest
import torch

import gated_deltanet_linear_spec_gb300 as gdn
from gated_deltanet_linear_spec_gb300 import workloads as W
from gated_deltanet_linear_spec_gb300.device_batch import to_device
from gated_deltanet_linear_spec_gb300.workloads import Subset
from tests.gpu_compare import assert_parity, run_gpu
from tests.oracle_run import np_act, run_oracle

pytestmark = pytest.mark.gpu


def _new_step(batch, seed):
    """The same rows with fresh activations and acceptance counts (the next decoding step)."""
    g = torch.Generator().manual_seed(seed)
    nb = copy.copy(batch)
    nb.x = torch.randn(batch.x.shape, generator=g).to(batch.x.dtype)
    nb.a = torch.randn(batch.a.shape, generator=g).to(batch.a.dtype)
    nb.b = torch.randn(batch.b.shape, generator=g).to(batch.b.dtype)
    if batch.spec is not None:
        nb.spec = copy.copy(batch.spec)
        k = batch.spec.spec_cols
        nb.spec.num_accepted_tokens = torch.randint(1, k + 1, (batch.spec.num_seqs,), generator=g).to(torch.int32)
    return nb


@pytest.mark.parametrize("workload", ["mixed_small", "spec_verify"])
def test_captured_step_replays_like_eager_calls(workload):
    batch = getattr(W, workload)()
    steps = [batch] + [_new_step(batch, 100 + i) for i in range(3)]
    eager = to_device(batch)
    graphed = to_device(batch)
    graphed.run()            # first call outside capture (one-time kernel attribute set-up)
    torch.cuda.synchronize()
    graphed.pools.conv_pool.copy_(eager.pools.conv_pool)
    graphed.pools.ssm_pool.copy_(eager.pools.ssm_pool)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        graphed.run()
    for st in steps:
        for name in ("x", "a", "b"):
            getattr(eager, name).copy_(getattr(st, name))
            getattr(graphed, name).copy_(getattr(st, name))
        if st.spec is not None:
            eager.spec.num_accepted_tokens.copy_(st.spec.num_accepted_tokens)
            graphed.spec.num_accepted_tokens.copy_(st.spec.num_accepted_tokens)
        eager.run()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(graphed.out, eager.out)
        assert torch.equal(graphed.pools.ssm_pool, eager.pools.ssm_pool)
        assert torch.equal(graphed.pools.conv_pool, eager.pools.conv_pool)
    assert int(graphed.status.item()) == 0


def _pad(batch, extra_tokens=5, extra_rows=3):
    """Pad x/a/b with garbage token rows and the spec subset with empty rows of NULL slots."""
    nb = copy.copy(batch)
    g = torch.Generator().manual_seed(7)
    pad = lambda t: torch.cat([t, torch.randn((extra_tokens,) + tuple(t.shape[1:]), generator=g).to(t.dtype)])  # noqa
    nb.x, nb.a, nb.b = pad(batch.x), pad(batch.a), pad(batch.b)
    s = batch.spec
    qsl = torch.cat([s.query_start_loc, s.query_start_loc[-1:].repeat(extra_rows)])
    ssi = torch.cat([s.spec_state_indices, torch.zeros((extra_rows, s.spec_cols), dtype=torch.int32)])
    na = torch.cat([s.num_accepted_tokens, torch.zeros(extra_rows, dtype=torch.int32)])
    nb.spec = Subset(qsl, s.token_indx, spec_state_indices=ssi, num_accepted_tokens=na)
    return nb


def test_padded_batch_equals_the_unpadded_one():
    batch = W.mixed_small(21)
    real_T = batch.num_actual_tokens
    ref = run_gpu(batch)
    padded = _pad(batch)
    d = to_device(padded)
    d.out.fill_(1.5)
    gdn.gdn_mixed_batch(d.layer, d.params, d.pools, d.x, d.a, d.b, d.non_spec, d.num_decodes, d.num_prefills,
                        d.spec, d.out, d.workspace, d.status, num_actual_tokens=real_T)
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    out = np_act(d.out.cpu())
    assert np.array_equal(out[:real_T], ref.out)
    assert (d.out[real_T:].float() == 1.5).all()
    assert np.array_equal(np_act(d.pools.conv_pool.cpu()), ref.conv_pool)
    assert np.array_equal(d.pools.ssm_pool.cpu().numpy().view(np.uint32), ref.ssm_pool.view(np.uint32))
    assert_parity(batch, ref, run_oracle(batch))

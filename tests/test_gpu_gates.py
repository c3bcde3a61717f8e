"""GPU parity at the extremes of the gates, on both recurrence paths.

The gates are g = -exp(A_log) softplus(a + dt_bias) and beta = sigmoid(b) ("[GDN]
Spec-decoding-aware attention kernel", the closing note on FLA's fused sigmoid-gated
recurrence).  The seeded workloads draw a, b ~ N(0, 1), which never reaches the branches tested
here: beta = 0 (b = -inf, pure decay), beta = 1 (b = +inf), the linear branch of softplus
(a + dt_bias > 20), and decays strong enough that gamma_t = e^{G_t} is 0 in fp32 inside a
64-token chunk -- everywhere, or only at some tokens, so that the cumulative log-decay of a chunk
is large while the differences G_t - G_s that weight its later tokens stay small.

Every batch mixes spec rows and a decode row (the token recurrence) with prefill rows of 200 and
130 tokens on a dk = dv = 128 bf16 layer (the tcgen05 chunked path), and is compared element by
element with the oracle at the stated tolerances.  For beta = 0 the stored states are also
checked against the closed form S_t = e^{g_1 + .. + g_t} S_0.
"""
import math

import numpy as np
import pytest
import torch

from gated_deltanet_linear_spec_gb300.workloads import LayerShape, RowSpec, build_batch
from tests.gpu_compare import STATE_REL, assert_parity, run_gpu
from tests.oracle_run import run_oracle

pytestmark = pytest.mark.gpu


def gate_batch(case: str, seed: int = 61):
    layer = LayerShape(1, 2, 128, 128, 4, 6, torch.bfloat16)
    rows = [RowSpec("spec", 4, 2), RowSpec("spec", 4, 4), RowSpec("spec", 3, 1), RowSpec("decode", 1),
            RowSpec("prefill", 200), RowSpec("prefill", 130, has_initial_state=False)]
    b = build_batch(layer, rows, num_slots=48, spec_cols=4, seed=seed, shuffle_from=0)
    g = torch.Generator().manual_seed(seed + 1000)
    T, Hv = b.a.shape
    small_A = torch.log(torch.empty(Hv).uniform_(1e-3, 1e-2, generator=g)).float()
    if case == "beta0":      # b = -inf: beta = 0, pure decay (mild, so the states stay non-zero)
        b.b = torch.full((T, Hv), float("-inf")).to(torch.bfloat16)
        b.A_log = small_A
    elif case == "beta1":    # b = +inf: beta = 1
        b.b = torch.full((T, Hv), float("inf")).to(torch.bfloat16)
    elif case == "softplus_linear":  # a + dt_bias in (21, 40): softplus(x) = x
        b.a = torch.empty((T, Hv)).uniform_(21.0, 40.0, generator=g).to(torch.bfloat16)
        b.A_log = small_A
    elif case == "decay_flush":      # g ~ -16 * 7.5 per token: gamma_t underflows after one token
        b.A_log = torch.full((Hv,), math.log(16.0))
        b.a = torch.empty((T, Hv)).uniform_(5.0, 10.0, generator=g).to(torch.bfloat16)
    elif case == "decay_some_tokens":  # every 8th token decays by ~e^-160, the others by ~e^-10
        b.A_log = torch.full((Hv,), math.log(16.0))
        a = torch.randn((T, Hv), generator=g)
        a[::8] = 10.0
        b.a = a.to(torch.bfloat16)
    else:
        raise ValueError(case)
    return b


@pytest.mark.parametrize("case", ["beta0", "beta1", "softplus_linear", "decay_flush", "decay_some_tokens"])
def test_gate_extremes_match_the_oracle(case):
    batch = gate_batch(case)
    assert batch.num_prefills == 2 and batch.spec is not None
    gpu = run_gpu(batch)
    assert_parity(batch, gpu, run_oracle(batch))


def _g(batch, gt: int, h: int) -> float:
    """g of global token gt at v-head h, in float64 from the batch's own inputs."""
    a = float(batch.a[gt, h].float()) + float(batch.dt_bias[h])
    sp = a if a > 20.0 else math.log1p(math.exp(a))
    return -math.exp(float(batch.A_log[h])) * sp


def test_beta_zero_is_pure_decay_on_both_paths():
    batch = gate_batch("beta0")
    gpu = run_gpu(batch)
    assert gpu.status == 0
    pool0 = batch.ssm_pool.double().numpy()
    Hv = batch.layer.num_v_heads
    checked = 0
    worst = 0.0

    def check(slot, prior, gts):
        nonlocal checked, worst
        for h in range(Hv):
            decay = math.exp(sum(_g(batch, gt, h) for gt in gts))
            ref = decay * (pool0[prior, h] if prior > 0 else 0.0)
            d = np.linalg.norm(gpu.ssm_pool[slot, h].astype(np.float64) - ref)
            nr = np.linalg.norm(ref)
            worst = max(worst, d / (nr if nr > 0 else 1.0))
            checked += 1

    sp = batch.spec
    qsl, tok = sp.query_start_loc.tolist(), sp.token_indx.tolist()
    for n in range(sp.num_seqs):
        na = int(sp.num_accepted_tokens[n])
        prior = int(sp.spec_state_indices[n, na - 1])
        gts = tok[qsl[n]:qsl[n + 1]]
        for t in range(len(gts)):
            slot = int(sp.spec_state_indices[n, t])
            if slot > 0:
                check(slot, prior, gts[:t + 1])
    ns = batch.non_spec
    qsl, tok = ns.query_start_loc.tolist(), ns.token_indx.tolist()
    for n in range(ns.num_seqs):
        slot = int(ns.state_indices[n])
        prior = slot if int(ns.has_initial_state[n]) else 0
        if slot > 0:
            check(slot, prior, tok[qsl[n]:qsl[n + 1]])
    assert checked > 0
    assert worst <= STATE_REL, f"pure decay off by {worst:.3e}"

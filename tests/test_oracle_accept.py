"""Pins of acceptance-aware non-spec rows in the oracle (CPU only).

A verify row cut to a prefix by the batch token budget is scheduled as a plain row ("[Bugfix]
Align Qwen GDN gates with speculative tokens", the second mechanism in the reachability
comment).  Given the acceptance of its previous verify step, such a row must continue from
what that step accepted.  Pinned three ways, all bit for bit:
  - a one-token aware row is a one-token verify row over the same slots;
  - an aware row of any length after a verify step equals the rollback path: a plain run over
    the accepted prefix, then a plain row (both conv layouts);
  - accepting one token with column 0 as the row's own slot changes nothing against a plain
    row, and has_initial_state = 0 still starts from zeros.
"""
import copy

import numpy as np
import pytest
import torch

from gated_deltanet_linear_spec_gb300.workloads import (LayerShape, RowSpec, Subset, build_batch, uniform_accepts,
                                                        with_layouts)
from tests.oracle_run import np_act, run_oracle

SMALL = LayerShape(2, 4, 16, 16, 4, 6, torch.bfloat16)
SMALL_F32 = LayerShape(2, 4, 16, 16, 4, 6, torch.float32)


@pytest.mark.parametrize("conv_layout", [0, 1])
@pytest.mark.parametrize("layer", [SMALL, SMALL_F32])
def test_one_token_aware_row_is_a_one_token_verify_row(layer, conv_layout):
    k = 4
    acc = uniform_accepts(6, k, 3)
    rows = [RowSpec("decode", 1, acc[i], aware=True) for i in range(6)]
    b = with_layouts(build_batch(layer, rows, num_slots=64, spec_cols=k, seed=9), conv_layout=conv_layout)
    ns = b.non_spec
    assert ns.num_accepted_tokens.tolist() == acc and not ns.is_spec
    spec = Subset(ns.query_start_loc, ns.token_indx, spec_state_indices=ns.spec_state_indices.clone(),
                  num_accepted_tokens=ns.num_accepted_tokens.clone())
    v = copy.copy(b)
    v.spec, v.non_spec, v.num_decodes = spec, None, 0
    r1, r2 = run_oracle(b), run_oracle(v)
    assert np.array_equal(r1.out, r2.out)
    assert np.array_equal(r1.ssm_pool, r2.ssm_pool)
    assert np.array_equal(r1.conv_pool, r2.conv_pool)


def _rollback_pair(layer, n_acc, Lb, seed, conv_layout, k=4, prev_acc=2):
    """Verify step A over k tokens, then an aware row B of Lb tokens with num_accepted = n_acc;
    against: a plain run A2 over the first n_acc tokens from the same history and state into a
    fresh slot, then a plain row B2 of the same Lb tokens from that slot."""
    gen = torch.Generator().manual_seed(seed)
    A = with_layouts(build_batch(layer, [RowSpec("spec", k, prev_acc)], num_slots=24, spec_cols=k, seed=seed),
                     conv_layout=conv_layout)
    ssi = A.spec.spec_state_indices
    used = set(ssi.view(-1).tolist())
    c = [p for p in range(1, 24) if p not in used][0]
    W = layer.conv_width
    conv, ssm = np_act(A.conv_pool), np_act(A.ssm_pool)
    if conv_layout == 0:
        hist = conv[int(ssi[0, 0]), prev_acc - 1: prev_acc - 1 + W - 1]
    else:
        hist = conv[int(ssi[0, prev_acc - 1]), : W - 1]
    conv2, ssm2 = conv.copy(), ssm.copy()
    conv2[c, : W - 1] = hist
    ssm2[c] = ssm[int(ssi[0, prev_acc - 1])]

    C, Hv, act = layer.channels, layer.num_v_heads, layer.act_dtype
    xB = torch.randn((Lb, C), generator=gen).to(act)
    aB = torch.randn((Lb, Hv), generator=gen).to(act)
    bB = torch.randn((Lb, Hv), generator=gen).to(act)
    q = lambda n: torch.tensor([0, n], dtype=torch.int32)  # noqa: E731
    one = torch.tensor([1], dtype=torch.int32)
    kind = (1, 0) if Lb == 1 else (0, 1)

    B = copy.copy(A)
    B.x, B.a, B.b, B.spec = xB, aB, bB, None
    B.non_spec = Subset(q(Lb), None, state_indices=ssi[:, 0].clone(), has_initial_state=one,
                        spec_state_indices=ssi.clone(), num_accepted_tokens=torch.tensor([n_acc], dtype=torch.int32))
    B.num_decodes, B.num_prefills = kind
    A2 = copy.copy(A)
    A2.x, A2.a, A2.b, A2.spec = A.x[:n_acc].clone(), A.a[:n_acc].clone(), A.b[:n_acc].clone(), None
    A2.non_spec = Subset(q(n_acc), None, state_indices=torch.tensor([c], dtype=torch.int32), has_initial_state=one)
    A2.num_decodes, A2.num_prefills = (1, 0) if n_acc == 1 else (0, 1)
    B2 = copy.copy(B)
    B2.non_spec = Subset(q(Lb), None, state_indices=torch.tensor([c], dtype=torch.int32), has_initial_state=one)

    ra = run_oracle(A, conv_pool=conv.copy(), ssm_pool=ssm.copy())
    rb = run_oracle(B, conv_pool=ra.conv_pool, ssm_pool=ra.ssm_pool)
    ra2 = run_oracle(A2, conv_pool=conv2, ssm_pool=ssm2)
    rb2 = run_oracle(B2, conv_pool=ra2.conv_pool, ssm_pool=ra2.ssm_pool)
    return ra, rb, ra2, rb2, int(ssi[0, 0]), c


@pytest.mark.parametrize("conv_layout", [0, 1])
@pytest.mark.parametrize("Lb", [1, 5])
@pytest.mark.parametrize("n_acc", [1, 2, 3, 4])
def test_aware_row_equals_the_rollback_path(n_acc, Lb, conv_layout):
    ra, rb, ra2, rb2, s0, c = _rollback_pair(SMALL, n_acc, Lb, 50 + 7 * n_acc + Lb, conv_layout)
    assert np.array_equal(ra.out[:n_acc], ra2.out)
    assert np.array_equal(rb.out, rb2.out)
    assert np.array_equal(rb.ssm_pool[s0], rb2.ssm_pool[c])
    W = SMALL.conv_width
    assert np.array_equal(rb.conv_pool[s0, : W - 1], rb2.conv_pool[c, : W - 1])


def test_aware_rows_that_accepted_one_token_are_plain_rows():
    rows = [RowSpec("decode", 1), RowSpec("decode", 1), RowSpec("prefill", 7), RowSpec("prefill", 3)]
    plain = build_batch(SMALL, rows, num_slots=40, spec_cols=3, seed=12)
    aware_rows = [RowSpec(r.kind, r.length, 1, aware=True) for r in rows]
    aware = build_batch(SMALL, aware_rows, num_slots=40, spec_cols=3, seed=12)
    assert torch.equal(aware.non_spec.state_indices, plain.non_spec.state_indices)
    assert torch.equal(aware.non_spec.spec_state_indices[:, 0], plain.non_spec.state_indices)
    for layout in (0, 1):
        r1 = run_oracle(with_layouts(plain, conv_layout=layout))
        r2 = run_oracle(with_layouts(aware, conv_layout=layout))
        assert np.array_equal(r1.out, r2.out)
        assert np.array_equal(r1.ssm_pool, r2.ssm_pool)
        assert np.array_equal(r1.conv_pool, r2.conv_pool)


def test_aware_row_without_initial_state_starts_from_zeros():
    rows = [RowSpec("prefill", 6, 3, has_initial_state=False, aware=True)]
    b = build_batch(SMALL, rows, num_slots=16, spec_cols=4, seed=14)
    zero = copy.copy(b)
    conv, ssm = b.conv_pool.clone(), b.ssm_pool.clone()
    src = int(b.non_spec.spec_state_indices[0, 2])
    own = int(b.non_spec.state_indices[0])
    conv[own].zero_()
    ssm[src].zero_()
    zero.conv_pool, zero.ssm_pool = conv, ssm
    zero.non_spec = copy.copy(b.non_spec)
    zero.non_spec.has_initial_state = torch.ones(1, dtype=torch.int32)
    r1, r2 = run_oracle(b), run_oracle(zero)
    assert np.array_equal(r1.out, r2.out)
    assert np.array_equal(r1.ssm_pool[own], r2.ssm_pool[own])

"""Pins of the oracle's speculative-decoding semantics and mixed-batch split (CPU only).

Speculative state contract ("[GDN] Spec-decoding-aware attention kernel", Changes,
gated_delta_rule.hpp bullet; Test Result: "K=N aligned-ring == non-spec native decode",
"NULL_BLOCK_ID suppresses pool I/O"): load from spec_state_indices[n, num_accepted-1], store
per token to spec_state_indices[n, t], slot <= 0 is NULL.
Mixed split ("[Bugfix] Align Qwen GDN gates with speculative tokens", Purpose and the
reachability comment): q|k|v and the a/b gates are gathered with the same index.
"""
import json
import os

import numpy as np
import pytest
import torch

from gated_deltanet_linear_spec_gb300.workloads import LayerShape, RowSpec, Subset, build_batch, tiny
from tests.oracle_run import run_oracle
from tests.scenarios import accepted_prefix_pair, p3_layout, relocate, with_subsets

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SMALL = LayerShape(2, 4, 16, 16, 4, 6, torch.bfloat16)
SMALL_F32 = LayerShape(2, 4, 16, 16, 4, 6, torch.float32)


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _changed_slots(pre, post):
    return {p for p in range(pre.shape[0]) if not np.array_equal(pre[p], post[p])}


@pytest.mark.parametrize("layer", [SMALL, SMALL_F32])
def test_single_verify_token_equals_non_spec_decode(layer):
    rows = [RowSpec("spec", 1, 1) for _ in range(5)]
    spec_batch = build_batch(layer, rows, num_slots=32, spec_cols=1, seed=31)
    ns = Subset(spec_batch.spec.query_start_loc, None, state_indices=spec_batch.spec.spec_state_indices[:, 0].clone(),
                has_initial_state=torch.ones(5, dtype=torch.int32))
    ns_batch = with_subsets(spec_batch, non_spec=ns, num_decodes=5)
    r1, r2 = run_oracle(spec_batch), run_oracle(ns_batch)
    assert np.array_equal(r1.out, r2.out)
    assert np.array_equal(r1.ssm_pool, r2.ssm_pool)
    assert np.array_equal(r1.conv_pool, r2.conv_pool)


@pytest.mark.parametrize("n_acc", [1, 2, 3, 4])
@pytest.mark.parametrize("layer", [SMALL, SMALL_F32])
def test_accepted_prefix_reproduces_non_spec_run(layer, n_acc):
    A, B, A2, B2 = accepted_prefix_pair(layer, n_acc, seed=40 + n_acc)
    ra = run_oracle(A)
    rb = run_oracle(B, conv_pool=ra.conv_pool, ssm_pool=ra.ssm_pool)
    ra2 = run_oracle(A2)
    rb2 = run_oracle(B2, conv_pool=ra2.conv_pool, ssm_pool=ra2.ssm_pool)
    assert np.array_equal(ra.out[:n_acc], ra2.out)
    assert np.array_equal(rb.out, rb2.out)
    for t in range(4):
        s, s2 = int(B.spec.spec_state_indices[0, t]), int(B2.spec.spec_state_indices[0, t])
        assert np.array_equal(rb.ssm_pool[s], rb2.ssm_pool[s2])


def test_null_load_slot_means_zero_prior():
    layer = SMALL_F32
    rows = [RowSpec("spec", 3, 2), RowSpec("spec", 3, 2)]
    batch = build_batch(layer, rows, num_slots=32, spec_cols=3, seed=50, spec_nulls=[(0, 1)])
    zero = batch.ssm_pool.clone()
    zero[int(batch.spec.spec_state_indices[1, 1])] = 0.0
    r_null = run_oracle(batch)
    # row 1 with an all-zero prior slot must equal row 0's NULL behaviour on the same values:
    # swap rows' values by building a batch whose row 0 reads the zeroed slot
    ssi = batch.spec.spec_state_indices.clone()
    ssi[0, 1] = ssi[1, 1]
    ssi[1, 1] = 0
    b2 = with_subsets(batch, spec=Subset(batch.spec.query_start_loc, None, spec_state_indices=ssi,
                                          num_accepted_tokens=batch.spec.num_accepted_tokens))
    b2.ssm_pool = zero
    r_zero = run_oracle(b2)
    assert np.array_equal(r_null.out[:3], r_zero.out[:3])


def test_null_store_slot_writes_nothing_and_other_slots_stay_untouched():
    layer = SMALL
    rows = [RowSpec("spec", 4, 3), RowSpec("spec", 2, 1), RowSpec("spec", 0, 1), RowSpec("spec", 4, 4)]
    batch = build_batch(layer, rows, num_slots=40, spec_cols=4, seed=51, spec_nulls=[(0, 2), (3, 0)])
    r = run_oracle(batch)
    pre_ssm = batch.ssm_pool.numpy()
    ssi = batch.spec.spec_state_indices.numpy()
    expect = set()
    for n, row in enumerate(rows):
        expect |= {int(ssi[n, t]) for t in range(row.length) if ssi[n, t] > 0}
    assert _changed_slots(pre_ssm, r.ssm_pool) == expect
    pre_conv = batch.conv_pool.view(torch.int16).numpy()
    post_conv = r.conv_pool.view(np.int16)
    expect_conv = {int(ssi[n, 0]) for n, row in enumerate(rows) if row.length > 0 and ssi[n, 0] > 0}
    assert _changed_slots(pre_conv, post_conv) == expect_conv
    assert np.array_equal(r.ssm_pool[0], pre_ssm[0]) and np.array_equal(post_conv[0], pre_conv[0])


def test_tiny_workload_touches_exactly_its_store_slots():
    batch = tiny()
    r = run_oracle(batch)
    ssi = batch.spec.spec_state_indices.numpy()
    assert (ssi == 0).sum() == 1 and len(set(ssi[ssi > 0].tolist())) == 8
    assert _changed_slots(batch.ssm_pool.numpy(), r.ssm_pool) == {int(s) for s in ssi.reshape(-1) if s > 0}
    assert np.isfinite(r.out_f64).all()


def test_p3_worked_example_interleaving_changes_nothing():
    g = _golden("p3_worked_example.json")
    rows = [RowSpec("spec", 3, 2), RowSpec("decode", 1)]
    # the page's layout: the non-spec row at token 0, the spec row at tokens 1..3
    page = build_batch(SMALL, rows, num_slots=32, spec_cols=3, seed=60, starts=[1, 0], force_token_indx=True)
    assert page.spec.token_indx.tolist() == g["spec_token_indx"]
    assert page.non_spec.token_indx.tolist() == g["non_spec_token_indx"]
    lead = relocate(page, [0, 3])  # spec tokens first
    r_page, r_lead = run_oracle(page), run_oracle(lead)
    m = lead.new_of_old.numpy()
    assert np.array_equal(r_lead.out[m], r_page.out)
    assert np.array_equal(r_lead.ssm_pool, r_page.ssm_pool)
    assert np.array_equal(r_lead.conv_pool, r_page.conv_pool)


def test_p3_reachability_layout_gate_gather():
    """Correct gathering: every token's output is independent of the interleaving.  The page's
    bug (gates read from the first T_spec rows): exactly the sixth spec row's 4 tokens move."""
    g = _golden("p3_reachability_layout.json")
    batch = p3_layout(SMALL, g, seed=61)
    tok = batch.spec.token_indx.numpy()
    first = int(np.argmax(tok != np.arange(len(tok))))
    assert first == g["first_misordered_token"]
    assert int((tok != np.arange(len(tok))).sum()) == g["max_displaced_spec_tokens"]

    good = run_oracle(batch)
    # interleaving-independence: put the non-spec row last
    lead = relocate(batch, [0, 4, 8, 12, 16, 20, 24])
    r_lead = run_oracle(lead)
    assert np.array_equal(r_lead.out[lead.new_of_old.numpy()], good.out)

    # planted mistake: the spec subset's gate for local token i is row i of a/b
    bug = with_subsets(batch, spec=batch.spec, non_spec=batch.non_spec,
                       num_decodes=batch.num_decodes, num_prefills=batch.num_prefills)
    a2, b2 = batch.a.clone(), batch.b.clone()
    a2[torch.from_numpy(tok).long()] = batch.a[: len(tok)]
    b2[torch.from_numpy(tok).long()] = batch.b[: len(tok)]
    bug.a, bug.b = a2, b2
    r_bug = run_oracle(bug)
    differs = [t for t in range(batch.num_actual_tokens) if not np.array_equal(r_bug.out[t], good.out[t])]
    assert differs == [int(t) for t in tok[g["first_misordered_token"]:]]

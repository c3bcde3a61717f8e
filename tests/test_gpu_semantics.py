"""GPU tests of the path's invariants (through the C ABI), each also held against the oracle.

- 10 repeated runs are byte-equal ("[GDN] Spec-decoding-aware attention kernel", Test Plan:
  determinism, 10x byte-equal core_attn_out + conv_state + ssm_state).
- A speculative row with one verify token equals a non-spec decode, bit for bit (same page,
  UT list: "K=N aligned-ring == non-spec native decode (bit-exact)").
- Rollback: a verify step with num_accepted = n followed by the next step equals a non-spec
  run over the n accepted tokens followed by the same step (the column-0 contract).
- Moving rows between interleaved token slots changes no token's output ("[Bugfix] Align Qwen
  GDN gates with speculative tokens"); the mixed call equals one call per subset ("[GDN]
  Spec-decoding-aware attention kernel", Test Plan: mixed batch matches per subset).
- Bad device data sets status bits, touches nothing it should not, and leaves the other rows
  exact; empty rows and all-NULL rows behave as the contract says.
"""
import copy

import numpy as np
import pytest
import torch

import gated_deltanet_linear_spec_gb300 as gdn
from gated_deltanet_linear_spec_gb300 import workloads as W
from gated_deltanet_linear_spec_gb300.device_batch import rows_to_device, to_device
from gated_deltanet_linear_spec_gb300.workloads import LayerShape, RowSpec, Subset, build_batch
from tests.gpu_compare import assert_outputs_close, assert_parity, assert_states_close, changed_slots, run_gpu
from tests.oracle_run import np_act, run_oracle
from tests.scenarios import accepted_prefix_pair, p3_layout, relocate, with_subsets

pytestmark = pytest.mark.gpu
SMALL = LayerShape(2, 4, 64, 64, 4, 6, torch.bfloat16)


def test_ten_runs_are_byte_equal():
    batch = W.spec_verify()
    first = run_gpu(batch)
    for _ in range(9):
        again = run_gpu(batch)
        assert np.array_equal(again.out, first.out)
        assert np.array_equal(again.conv_pool, first.conv_pool)
        assert np.array_equal(again.ssm_pool.view(np.uint32), first.ssm_pool.view(np.uint32))


@pytest.mark.parametrize("layer", [SMALL, W.big_layer(3)])
def test_single_verify_token_equals_non_spec_decode_bitwise(layer):
    rows = [RowSpec("spec", 1, 1) for _ in range(8)]
    sb = build_batch(layer, rows, num_slots=32, spec_cols=1, seed=71, spec_nulls=[(3, 0)])
    ns = Subset(sb.spec.query_start_loc, None, state_indices=sb.spec.spec_state_indices[:, 0].clone(),
                has_initial_state=torch.ones(8, dtype=torch.int32))
    nb = with_subsets(sb, non_spec=ns, num_decodes=8)
    g1, g2 = run_gpu(sb), run_gpu(nb)
    assert np.array_equal(g1.out, g2.out)
    assert np.array_equal(g1.conv_pool, g2.conv_pool)
    assert np.array_equal(g1.ssm_pool.view(np.uint32), g2.ssm_pool.view(np.uint32))
    assert_parity(sb, g1, run_oracle(sb))


def _run_chain(first, second):
    d1 = to_device(first)
    d1.run()
    torch.cuda.synchronize()
    d1.ssm_after = d1.pools.ssm_pool.cpu().numpy().copy()
    d2 = to_device(second, pools=d1.pools)
    d2.run()
    torch.cuda.synchronize()
    return d1, d2


@pytest.mark.parametrize("n_acc", [1, 2, 3, 4])
def test_rollback_to_accepted_prefix(n_acc):
    A, B, A2, B2 = accepted_prefix_pair(SMALL, n_acc, seed=80 + n_acc)
    a, b = _run_chain(A, B)
    a2, b2 = _run_chain(A2, B2)
    assert torch.equal(a.out[:n_acc], a2.out)
    assert torch.equal(b.out, b2.out)
    for t in range(4):
        s, s2 = int(B.spec.spec_state_indices[0, t]), int(B2.spec.spec_state_indices[0, t])
        assert torch.equal(b.pools.ssm_pool[s], b2.pools.ssm_pool[s2])
    # and the chain itself matches the oracle
    ra = run_oracle(A)
    rb = run_oracle(B, conv_pool=ra.conv_pool.copy(), ssm_pool=ra.ssm_pool.copy())
    assert_outputs_close(np_act(b.out.cpu()), rb, bf16=True)
    gpu_final = b.pools.ssm_pool.cpu().numpy()
    # step B writes the same slots on both sides (each side judged against its own pool after A)
    assert changed_slots(a.ssm_after, gpu_final) == changed_slots(ra.ssm_pool, rb.ssm_pool)
    # and every slot either step wrote agrees within the state tolerance
    assert_states_close(A.ssm_pool.numpy(), gpu_final, rb.ssm_pool)
    assert np.array_equal(np_act(b.pools.conv_pool.cpu()), rb.conv_pool)


def test_p3_layout_interleaving_is_invisible():
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "p3_reachability_layout.json")) as f:
        g = json.load(f)
    page = p3_layout(SMALL, g, seed=90)
    lead = relocate(page, [0, 4, 8, 12, 16, 20, 24])
    gp, gl = run_gpu(page), run_gpu(lead)
    assert np.array_equal(gl.out[lead.new_of_old.numpy()], gp.out)
    assert np.array_equal(gl.ssm_pool.view(np.uint32), gp.ssm_pool.view(np.uint32))
    assert_parity(page, gp, run_oracle(page))


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_interleavings_of_a_mixed_batch(seed):
    base = W.mixed_small(seed)
    rng = np.random.default_rng(seed)
    order = list(range(len(base.rows)))
    rng.shuffle(order)
    starts, pos = [0] * len(order), 0
    for i in order:
        starts[i] = pos
        pos += base.rows[i].length
    moved = relocate(base, starts)
    g0, g1 = run_gpu(base), run_gpu(moved)
    assert np.array_equal(g1.out[moved.new_of_old.numpy()], g0.out)
    assert np.array_equal(g1.conv_pool, g0.conv_pool)
    assert np.array_equal(g1.ssm_pool.view(np.uint32), g0.ssm_pool.view(np.uint32))
    assert_parity(moved, g1, run_oracle(moved))


def test_mixed_call_equals_one_call_per_subset():
    """gdn_mixed_batch == conv per subset, then the token recurrence on spec and decode rows and
    the chunked prefill on the prefill rows, bit for bit."""
    batch = W.mixed_small(5)
    whole = run_gpu(batch)
    d = to_device(batch)
    C = batch.layer.channels
    ys = {}
    for name, rows in (("spec", d.spec), ("non_spec", d.non_spec)):
        ys[name] = torch.empty((rows.num_tokens, C), dtype=torch.float32, device="cuda")
        gdn.gdn_conv_update(d.layer, d.params, d.pools, d.x, rows, ys[name], d.status)
    gdn.gdn_recurrent_step(d.layer, d.params, d.pools, ys["spec"], d.a, d.b, d.spec, d.out, d.status)
    ns, nd = d.non_spec, batch.num_decodes
    q = ns.query_start_loc
    split = int(q[nd])
    dec = gdn.Rows(q[: nd + 1].contiguous(), split, ns.token_indx[:split].contiguous(),
                   ns.state_indices[:nd].contiguous(), ns.has_initial_state[:nd].contiguous())
    pre = gdn.Rows((q[nd:] - split).contiguous(), ns.num_tokens - split, ns.token_indx[split:].contiguous(),
                   ns.state_indices[nd:].contiguous(), ns.has_initial_state[nd:].contiguous())
    gdn.gdn_recurrent_step(d.layer, d.params, d.pools, ys["non_spec"][:split].contiguous(), d.a, d.b, dec, d.out,
                           d.status)
    gdn.gdn_chunk_prefill(d.layer, d.params, d.pools, ys["non_spec"][split:].contiguous(), d.a, d.b, pre, d.out,
                          status=d.status)
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    assert np.array_equal(np_act(d.out.cpu()), whole.out)
    assert np.array_equal(np_act(d.pools.conv_pool.cpu()), whole.conv_pool)
    assert torch.equal(d.pools.ssm_pool.cpu(), torch.from_numpy(whole.ssm_pool))


def test_conv_update_alone_matches_oracle_in_both_output_types():
    batch = W.mixed_small(6)
    ref = run_oracle(batch)
    for ydt in (torch.float32, torch.bfloat16):
        d = to_device(batch)
        for name, rows in (("spec", d.spec), ("non_spec", d.non_spec)):
            y = torch.empty((rows.num_tokens, batch.layer.channels), dtype=ydt, device="cuda")
            gdn.gdn_conv_update(d.layer, d.params, d.pools, d.x, rows, y, d.status)
            torch.cuda.synchronize()
            yr = ref.y[name]
            tol = 1e-5 if ydt == torch.float32 else 8e-3
            assert np.all(np.abs(y.double().cpu().numpy() - yr) <= tol * (1 + np.abs(yr)))
        assert np.array_equal(np_act(d.pools.conv_pool.cpu()), ref.conv_pool)
        assert int(d.status.item()) == 0


def test_recurrent_step_with_bf16_qkv_input():
    """gdn_recurrent_step on a bf16 post-conv activation: the oracle gets the same bf16 values."""
    batch = W.mixed_small(8)
    ref_conv = run_oracle(batch)  # only for y
    d = to_device(batch)
    rows = d.spec
    y32 = torch.from_numpy(ref_conv.y["spec"]).to(torch.float32)
    ybf = y32.to(torch.bfloat16)
    gdn.gdn_recurrent_step(d.layer, d.params, d.pools, ybf.cuda(), d.a, d.b, rows, d.out, d.status)
    torch.cuda.synchronize()
    import oracle
    from tests.oracle_run import oracle_layer, oracle_rows
    sp = np_act(batch.ssm_pool)
    out = np.zeros(tuple(d.out.shape), np.uint16)
    of = np.full(tuple(d.out.shape), np.nan)
    oracle.recurrent(oracle_layer(batch), np_act(batch.A_log), np_act(batch.dt_bias), sp,
                     ybf.double().numpy(), np_act(batch.a), np_act(batch.b), batch.num_actual_tokens,
                     oracle_rows(batch.spec), out, of, None, 8)
    res = type("R", (), {"out_f64": of})
    assert_outputs_close(np_act(d.out.cpu()), res, bf16=True)
    assert_states_close(batch.ssm_pool.numpy(), d.pools.ssm_pool.cpu().numpy(), sp)


def _drop_spec_row(s: Subset, n: int) -> Subset:
    qsl = s.query_start_loc.tolist()
    tok = s.token_indx if s.token_indx is not None else torch.arange(s.num_tokens, dtype=torch.int32)
    keep = [i for i in range(s.num_seqs) if i != n]
    lens = [qsl[i + 1] - qsl[i] for i in keep]
    new_qsl = torch.tensor([0] + np.cumsum(lens).tolist(), dtype=torch.int32)
    new_tok = torch.cat([tok[qsl[i]:qsl[i + 1]] for i in keep]).to(torch.int32)
    return Subset(new_qsl, new_tok, spec_state_indices=s.spec_state_indices[keep].clone(),
                  num_accepted_tokens=s.num_accepted_tokens[keep].clone())


def _bad_row_case(mutate, expect_bit, row=2):
    batch = W.mixed_small(11)
    bad = copy.copy(batch)
    bad.spec = copy.copy(batch.spec)
    mutate(bad.spec, row)
    gpu = run_gpu(bad)
    assert gpu.status & expect_bit, f"status {gpu.status:#x} lacks {expect_bit:#x}"
    good = with_subsets(batch, spec=_drop_spec_row(batch.spec, row), non_spec=batch.non_spec,
                        num_decodes=batch.num_decodes, num_prefills=batch.num_prefills)
    ref = run_oracle(good)
    tok = batch.spec.token_indx
    q = batch.spec.query_start_loc
    mask = np.ones(batch.num_actual_tokens, bool)
    mask[tok[int(q[row]):int(q[row + 1])].numpy()] = False
    assert_outputs_close(gpu.out, ref, bf16=True, rows_mask=mask)
    return batch, gpu, ref, mask


def test_num_accepted_out_of_range_skips_the_row():
    def mut(s, n):
        s.num_accepted_tokens = s.num_accepted_tokens.clone()
        s.num_accepted_tokens[n] = 0
    batch, gpu, ref, mask = _bad_row_case(mut, gdn.STATUS_NUM_ACCEPTED)
    assert np.array_equal(gpu.conv_pool, ref.conv_pool)
    assert_states_close(batch.ssm_pool.numpy(), gpu.ssm_pool, ref.ssm_pool)
    assert not gpu.out[~mask].any()  # the skipped row's outputs were never written


def test_slot_out_of_range_sets_status_and_skips_the_store():
    batch = W.mixed_small(11)
    s = batch.spec
    q = s.query_start_loc.tolist()
    n = next(i for i in range(s.num_seqs) if q[i + 1] - q[i] == 4)
    load_col = int(s.num_accepted_tokens[n]) - 1
    store_col = next(c for c in (3, 2, 1) if c != load_col)  # a store-only column, not the conv column 0
    bad = copy.copy(batch)
    bad.spec = copy.copy(s)
    bad.spec.spec_state_indices = s.spec_state_indices.clone()
    bad.spec.spec_state_indices[n, store_col] = 10_000
    gpu = run_gpu(bad)
    assert gpu.status & gdn.STATUS_SLOT_RANGE
    ref = run_oracle(batch)
    # every slot the oracle wrote, except the one redirected out of range, is written the same
    dropped = int(s.spec_state_indices[n, store_col])
    exp = changed_slots(batch.ssm_pool.numpy(), ref.ssm_pool) - {dropped}
    assert changed_slots(batch.ssm_pool.numpy(), gpu.ssm_pool) == exp
    assert_outputs_close(gpu.out, ref, bf16=True)


def test_token_index_out_of_range_sets_status():
    batch = W.mixed_small(12)
    bad = copy.copy(batch)
    bad.spec = copy.copy(batch.spec)
    bad.spec.token_indx = batch.spec.token_indx.clone()
    bad.spec.token_indx[0] = 1 << 20
    gpu = run_gpu(bad)
    assert gpu.status & gdn.STATUS_TOKEN_RANGE


def test_non_monotone_query_start_loc_sets_status():
    def mut(s, n):
        s.query_start_loc = s.query_start_loc.clone()
        s.query_start_loc[n + 1] = s.query_start_loc[n] - 1
    batch = W.mixed_small(13)
    bad = copy.copy(batch)
    bad.spec = copy.copy(batch.spec)
    mut(bad.spec, 1)
    gpu = run_gpu(bad)
    assert gpu.status & gdn.STATUS_ROW_RANGE


def test_empty_rows_and_all_null_rows():
    rows = [RowSpec("spec", 0, 1), RowSpec("spec", 4, 2), RowSpec("spec", 3, 3), RowSpec("spec", 0, 4)]
    nulls = [(2, c) for c in range(4)]
    batch = build_batch(SMALL, rows, num_slots=40, spec_cols=4, seed=14, spec_nulls=nulls)
    gpu = run_gpu(batch)
    ref = run_oracle(batch)
    assert_parity(batch, gpu, ref)
    ssi = batch.spec.spec_state_indices.numpy()
    expect = {int(ssi[1, t]) for t in range(4)}
    assert changed_slots(batch.ssm_pool.numpy(), gpu.ssm_pool) == expect


def test_batch_without_tokens_is_a_no_op():
    batch = W.mixed_small(15)
    d = to_device(batch)
    empty = rows_to_device(Subset(torch.zeros(1, dtype=torch.int32)), "cuda")
    gdn.gdn_mixed_batch(d.layer, d.params, d.pools, d.x[:0], d.a[:0], d.b[:0], None, 0, 0, None, d.out[:0],
                        d.workspace, d.status)
    gdn.gdn_recurrent_step(d.layer, d.params, d.pools, d.x[:0].float(), d.a, d.b,
                           gdn.Rows(empty.query_start_loc, 0, state_indices=d.non_spec.state_indices[:0]),
                           d.out, d.status)
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    assert torch.equal(d.pools.ssm_pool.cpu(), batch.ssm_pool)

"""Pins of the oracle's causal conv1d and conv-ring contract (CPU only).

The conv output is checked against torch's float64 ``conv1d`` (an independent library
routine); the ring contents against the placement the pages state for the speculative
staging buffer ("[GDN] Spec-decoding-aware attention kernel", Changes, pass 1: token t goes
to column state_len - K_call + t; earlier columns are a shift copy of the pre-state) and the
column-0 rolled-history contract with load offset num_accepted - 1 (same page, Problem and
the IS_SPEC load bullet; "[XE2] Support MTP of QWEN model", review thread).
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from gated_deltanet_linear_spec_gb300.workloads import LayerShape, RowSpec, build_batch
from tests.oracle_run import act_to_f64, np_act, oracle_layer, oracle_rows

SMALL = LayerShape(2, 4, 16, 16, 4, 6, torch.float32)
SMALL_BF16 = LayerShape(2, 4, 16, 16, 4, 6, torch.bfloat16)


def _torch_conv_silu(hist: np.ndarray, xs: np.ndarray, w: np.ndarray, bias) -> np.ndarray:
    """SiLU(conv1d) over [hist ; xs] (time-major, [*, C]), valid positions only, float64."""
    seq = torch.from_numpy(np.concatenate([hist, xs], 0).T[None].copy())      # [1, C, W-1+L]
    wt = torch.from_numpy(w[:, None, :].copy())                                 # [C, 1, W]
    bt = None if bias is None else torch.from_numpy(bias.copy())
    y = F.conv1d(seq, wt, bt, groups=w.shape[0])                                # [1, C, L]
    return F.silu(y)[0].T.numpy()


def _run_conv(batch, which):
    L = oracle_layer(batch)
    rows = oracle_rows(getattr(batch, which))
    pool = np_act(batch.conv_pool)
    pre = pool.copy()
    cb = None if batch.conv_b is None else np_act(batch.conv_b)
    y = oracle.conv_update(L, np_act(batch.conv_w), cb, pool, np_act(batch.x), batch.num_actual_tokens, rows)
    return pre, pool, y, rows


@pytest.mark.parametrize("layer", [SMALL, SMALL_BF16])
@pytest.mark.parametrize("bias", [False, True])
def test_fresh_prefill_row_equals_zero_padded_conv1d(layer, bias):
    rows = [RowSpec("prefill", 37, has_initial_state=False), RowSpec("prefill", 5)]
    batch = build_batch(layer, rows, num_slots=8, seed=11, conv_bias=bias)
    pre, pool, y, r = _run_conv(batch, "non_spec")
    x = act_to_f64(np_act(batch.x))
    w = act_to_f64(np_act(batch.conv_w))
    bb = None if batch.conv_b is None else act_to_f64(np_act(batch.conv_b))
    C, W = layer.channels, layer.conv_width
    # row 0: has_initial_state = 0 -> zero history, i.e. torch's zero padding of W-1
    tok0 = np.asarray(r.token_indx if r.token_indx is not None else np.arange(r.num_tokens))
    ref0 = _torch_conv_silu(np.zeros((W - 1, C)), x[tok0[:37]], w, bb)
    np.testing.assert_allclose(y[:37], ref0, rtol=1e-13, atol=1e-13)
    # row 1: continues from the slot's first W-1 columns
    slot1 = int(r.state_indices[1])
    hist = act_to_f64(pre[slot1, : W - 1])
    ref1 = _torch_conv_silu(hist, x[tok0[37:]], w, bb)
    np.testing.assert_allclose(y[37:], ref1, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("layer", [SMALL, SMALL_BF16])
def test_spec_row_reads_history_at_num_accepted_minus_one(layer):
    # state_len 6 with W = 4 holds K_call = 4 verify tokens; one row per anchor 0..3
    rows = [RowSpec("spec", 4, na) for na in (1, 2, 3, 4)]
    batch = build_batch(layer, rows, num_slots=32, spec_cols=4, seed=5)
    pre, pool, y, r = _run_conv(batch, "spec")
    x = act_to_f64(np_act(batch.x))
    w = act_to_f64(np_act(batch.conv_w))
    W = layer.conv_width
    for n, na in enumerate((1, 2, 3, 4)):
        slot = int(r.spec_state_indices[n, 0])
        hist = act_to_f64(pre[slot, na - 1: na - 1 + W - 1])
        ref = _torch_conv_silu(hist, x[4 * n: 4 * n + 4], w, None)
        np.testing.assert_allclose(y[4 * n: 4 * n + 4], ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("layer", [SMALL, SMALL_BF16])
def test_spec_ring_placement_matches_staging_formula(layer):
    """Full rows (L = K_call): column state_len-K_call+t holds x_t bit for bit, and the
    first state_len-K_call columns are the pre-state shifted from the anchor."""
    k_call, W, SL = 4, layer.conv_width, layer.conv_state_len
    rows = [RowSpec("spec", k_call, na) for na in (1, 3, 4, 2)]
    batch = build_batch(layer, rows, num_slots=40, spec_cols=k_call, seed=9)
    pre, pool, y, r = _run_conv(batch, "spec")
    x = np_act(batch.x)
    for n, row in enumerate(rows):
        slot = int(r.spec_state_indices[n, 0])
        a = row.num_accepted - 1
        for t in range(k_call):
            assert np.array_equal(pool[slot, SL - k_call + t], x[k_call * n + t])
        for j in range(SL - k_call):
            assert np.array_equal(pool[slot, j], pre[slot, a + 1 + j])
        # the other K-1 slots of the row keep their conv contents (column-0 contract)
        for c in range(1, k_call):
            other = int(r.spec_state_indices[n, c])
            assert np.array_equal(pool[other], pre[other])


def test_ragged_spec_row_leaves_tail_columns_untouched():
    layer = SMALL_BF16
    W, SL = layer.conv_width, layer.conv_state_len
    rows = [RowSpec("spec", 2, 3), RowSpec("spec", 1, 1), RowSpec("spec", 4, 4)]
    batch = build_batch(layer, rows, num_slots=40, spec_cols=4, seed=13)
    pre, pool, y, r = _run_conv(batch, "spec")
    x = np_act(batch.x)
    starts = [0, 2, 3]
    for n, row in enumerate(rows):
        slot = int(r.spec_state_indices[n, 0])
        a, L = row.num_accepted - 1, row.length
        ncols = W - 2 + L
        for j in range(W - 2):
            assert np.array_equal(pool[slot, j], pre[slot, a + 1 + j])
        for t in range(L):
            assert np.array_equal(pool[slot, W - 2 + t], x[starts[n] + t])
        for j in range(ncols, SL):
            assert np.array_equal(pool[slot, j], pre[slot, j])


def test_non_spec_ring_keeps_last_inputs():
    layer = SMALL_BF16
    W = layer.conv_width
    rows = [RowSpec("decode", 1), RowSpec("prefill", 2), RowSpec("prefill", 9, has_initial_state=False)]
    batch = build_batch(layer, rows, num_slots=10, seed=17)
    pre, pool, y, r = _run_conv(batch, "non_spec")
    x = np_act(batch.x)
    tok = np.asarray(r.token_indx) if r.token_indx is not None else np.arange(r.num_tokens)
    qsl = r.query_start_loc
    for n in range(3):
        slot = int(r.state_indices[n])
        L = int(qsl[n + 1] - qsl[n])
        hist = pre[slot, : W - 1] if (n < 2) else np.zeros_like(pre[slot, : W - 1])
        H = np.concatenate([hist, x[tok[qsl[n]: qsl[n + 1]]]], 0)
        assert np.array_equal(pool[slot, : W - 1], H[L: L + W - 1])
        assert np.array_equal(pool[slot, W - 1:], pre[slot, W - 1:])


def test_null_conv_slot_reads_zero_and_writes_nothing():
    layer = SMALL
    rows = [RowSpec("spec", 3, 2), RowSpec("spec", 3, 3)]
    batch = build_batch(layer, rows, num_slots=20, spec_cols=4, seed=21, spec_nulls=[(0, 0)])
    pre, pool, y, r = _run_conv(batch, "spec")
    # slot 0 (NULL) is never written, and row 0 sees a zero history
    assert np.array_equal(pool[0], pre[0])
    x = act_to_f64(np_act(batch.x))
    w = act_to_f64(np_act(batch.conv_w))
    ref = _torch_conv_silu(np.zeros((3, layer.channels)), x[:3], w, None)
    np.testing.assert_allclose(y[:3], ref, rtol=1e-13, atol=1e-13)
    # only the conv slot of row 1 changed
    changed = [p for p in range(pool.shape[0]) if not np.array_equal(pool[p], pre[p])]
    assert changed == [int(r.spec_state_indices[1, 0])]


def test_empty_row_touches_nothing():
    layer = SMALL
    rows = [RowSpec("spec", 0, 2), RowSpec("spec", 2, 1)]
    batch = build_batch(layer, rows, num_slots=20, spec_cols=4, seed=23)
    pre, pool, y, r = _run_conv(batch, "spec")
    slot0 = int(r.spec_state_indices[0, 0])
    assert np.array_equal(pool[slot0], pre[slot0])
    assert y.shape[0] == 2

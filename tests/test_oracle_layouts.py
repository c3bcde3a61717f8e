"""Pins of the oracle's two alternative layouts (CPU only).

Per-k-head x ("[GDN] Spec-decoding-aware attention kernel", Test Plan: the reorder_input=False
projection order): x holds, for each k-head g in turn, q_g, k_g and the v of the Hv/Hk v-heads
of group g.  Only where the conv reads x changes, so a run on the permuted x must reproduce the
packed run bit for bit.

Per-slot conv snapshots ("[XE2] Support MTP of QWEN model", review thread on the conv state
layout): a spec row reads its history from column 0 of spec_state_indices[n, num_accepted-1]
and, after token t, stores the last W-1 inputs to spec_state_indices[n, t].  Pinned by the
closed form of what each written slot must hold, and by a two-step chain whose outputs equal
the rolled layout's outputs once the history is the same.
"""
import copy

import numpy as np
import pytest
import torch

from gated_deltanet_linear_spec_gb300.workloads import LayerShape, RowSpec, build_batch, per_khead_order, with_layouts
from tests.oracle_run import act_to_f64, np_act, run_oracle

SMALL = LayerShape(2, 4, 16, 16, 4, 6, torch.bfloat16)
SMALL_F32 = LayerShape(2, 4, 16, 16, 4, 6, torch.float32)


def test_per_khead_order_by_hand():
    # Hk = 2, Hv = 4 (G = 2), dk = 2, dv = 3: a group is q_g(2) k_g(2) v(3) v(3) = 10 channels
    L = LayerShape(2, 4, 2, 3, 4, 3, torch.float32)
    expected = ([0, 1, 10, 11] +                            # q0, q1
                [2, 3, 12, 13] +                            # k0, k1
                [4, 5, 6, 7, 8, 9, 14, 15, 16, 17, 18, 19])  # v0, v1 (group 0), v2, v3 (group 1)
    assert per_khead_order(L).tolist() == expected
    # G = 1 keeps one v-head per group
    L1 = LayerShape(2, 2, 2, 2, 4, 3, torch.float32)
    assert per_khead_order(L1).tolist() == [0, 1, 6, 7, 2, 3, 8, 9, 4, 5, 10, 11]
    # a single k-head is one group: the per-k-head order is the packed order
    assert per_khead_order(LayerShape(1, 4, 2, 3, 4, 3, torch.float32)).tolist() == list(range(16))


def _mixed_rows():
    return ([RowSpec("decode", 1), RowSpec("decode", 1)] +
            [RowSpec("spec", 4, 1 + i % 4) for i in range(4)] +
            [RowSpec("prefill", 9), RowSpec("prefill", 3, has_initial_state=False)])


@pytest.mark.parametrize("layer", [SMALL, SMALL_F32, LayerShape(2, 8, 16, 32, 3, 4, torch.bfloat16)])
def test_per_khead_x_reproduces_packed_run(layer):
    b = build_batch(layer, _mixed_rows(), num_slots=32, spec_cols=4, seed=11, shuffle_from=2,
                    spec_nulls=[(1, 2)], conv_bias=True)
    bk = with_layouts(b, qkv_layout=1)
    assert not torch.equal(bk.x, b.x)
    r, rk = run_oracle(b), run_oracle(bk)
    assert np.array_equal(r.out, rk.out)
    assert np.array_equal(r.ssm_pool, rk.ssm_pool)
    assert np.array_equal(r.conv_pool, rk.conv_pool)
    for name in r.y:
        assert np.array_equal(r.y[name], rk.y[name])


def _raw(t):
    return np_act(t)


@pytest.mark.parametrize("layer,k", [(SMALL, 4), (SMALL_F32, 4),
                                     (LayerShape(2, 4, 16, 16, 4, 3, torch.bfloat16), 6),
                                     (LayerShape(2, 4, 16, 16, 2, 1, torch.float32), 5)])
def test_per_slot_snapshots_closed_form(layer, k):
    # the per-slot layout needs only W-1 columns, so spec_cols may exceed state_len - W + 2
    acc = [1 + (3 * i) % k for i in range(6)]
    rows = [RowSpec("spec", k if i != 4 else k - 2, acc[i] if i != 4 else min(acc[i], k)) for i in range(6)]
    b = build_batch(layer, rows, num_slots=64, spec_cols=k, seed=23, spec_nulls=[(2, 0), (3, k - 1), (5, acc[5] - 1)])
    b = with_layouts(b, conv_layout=1)
    pre = _raw(b.conv_pool)
    r = run_oracle(b)
    W, C = layer.conv_width, layer.channels
    x = _raw(b.x)
    ssi = b.spec.spec_state_indices.numpy()
    na = b.spec.num_accepted_tokens.numpy()
    qsl = b.spec.query_start_loc.numpy()
    tok = b.spec.token_indx.numpy() if b.spec.token_indx is not None else np.arange(b.spec.num_tokens)
    expect = pre.copy()
    for n in range(len(rows)):
        L = qsl[n + 1] - qsl[n]
        src = ssi[n, na[n] - 1]
        hist = pre[src, :W - 1] if src > 0 else np.zeros((W - 1, C), dtype=pre.dtype)
        H = np.concatenate([hist, x[tok[qsl[n]: qsl[n + 1]]]], axis=0)
        for t in range(L):
            if ssi[n, t] > 0:
                expect[ssi[n, t], :W - 1] = H[t + 1: t + W]
    assert np.array_equal(r.conv_pool, expect)
    # the conv outputs use that history: y of token t is SiLU(bias + sum_i w_i H[t+i])
    w = act_to_f64(_raw(b.conv_w)).reshape(C, W)
    y = r.y["spec"]
    for n in range(len(rows)):
        L = qsl[n + 1] - qsl[n]
        src = ssi[n, na[n] - 1]
        hist = pre[src, :W - 1] if src > 0 else np.zeros((W - 1, C), dtype=pre.dtype)
        H = act_to_f64(np.concatenate([hist, x[tok[qsl[n]: qsl[n + 1]]]], axis=0))
        for t in range(L):
            z = (w * H[t: t + W].T).sum(axis=1)
            np.testing.assert_allclose(y[qsl[n] + t], z / (1 + np.exp(-z)), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("layer", [SMALL, SMALL_F32])
def test_per_slot_chain_matches_rolled_chain(layer):
    # two verify steps over the same slots: once the first history agrees, both layouts give
    # the same outputs and states at every step (no NULL slots, so every write is visible)
    k, n_rows, W = 4, 5, layer.conv_width
    acc1 = [1, 2, 3, 4, 2]
    acc2 = [4, 1, 2, 3, 3]
    b1 = build_batch(layer, [RowSpec("spec", k, acc1[i]) for i in range(n_rows)], num_slots=48, spec_cols=k, seed=5)
    b2 = build_batch(layer, [RowSpec("spec", k, acc2[i]) for i in range(n_rows)], num_slots=48, spec_cols=k, seed=6)
    b2.spec = copy.copy(b2.spec)
    b2.spec.spec_state_indices = b1.spec.spec_state_indices.clone()
    ssi = b1.spec.spec_state_indices.numpy()

    rolled_conv = _raw(b1.conv_pool)
    slot_conv = rolled_conv.copy()
    for n in range(n_rows):  # the per-slot history is the rolled ring read at num_accepted-1
        a = acc1[n] - 1
        slot_conv[ssi[n, a], :W - 1] = rolled_conv[ssi[n, 0], a: a + W - 1]
    ssm = _raw(b1.ssm_pool)

    rr1 = run_oracle(b1, conv_pool=rolled_conv.copy(), ssm_pool=ssm.copy())
    rs1 = run_oracle(with_layouts(b1, conv_layout=1), conv_pool=slot_conv.copy(), ssm_pool=ssm.copy())
    assert np.array_equal(rr1.out, rs1.out)
    assert np.array_equal(rr1.ssm_pool, rs1.ssm_pool)
    rr2 = run_oracle(b2, conv_pool=rr1.conv_pool, ssm_pool=rr1.ssm_pool)
    rs2 = run_oracle(with_layouts(b2, conv_layout=1), conv_pool=rs1.conv_pool, ssm_pool=rs1.ssm_pool)
    assert np.array_equal(rr2.out, rs2.out)
    assert np.array_equal(rr2.ssm_pool, rs2.ssm_pool)
    # and the per-slot pool holds, in every verify slot, the rolled ring's window at that token
    for n in range(n_rows):
        for t in range(k):
            assert np.array_equal(rs2.conv_pool[ssi[n, t], :W - 1], rr2.conv_pool[ssi[n, 0], t: t + W - 1])


def test_negative_control_scattered_snapshots_are_not_the_rolled_contract():
    # "[GDN] Spec-decoding-aware attention kernel", Problem: under the rolled contract only the
    # column-0 slot of a verify row is updated and columns 1..K-1 stay untouched; writing
    # per-token snapshots across the K slots and then reading the ring as rolled diverges.
    layer, k = SMALL, 4
    rows = [RowSpec("spec", k, 1 + i % k) for i in range(5)]
    b1 = build_batch(layer, rows, num_slots=48, spec_cols=k, seed=61)
    pre = _raw(b1.conv_pool)
    rolled = run_oracle(b1)
    scattered = run_oracle(with_layouts(b1, conv_layout=1))
    ssi = b1.spec.spec_state_indices.numpy()
    for n in range(len(rows)):
        for t in range(1, k):
            assert np.array_equal(rolled.conv_pool[ssi[n, t]], pre[ssi[n, t]])       # untouched
        assert not np.array_equal(scattered.conv_pool[ssi[n, k - 1]], pre[ssi[n, k - 1]])  # written
    # the next verify step reads the ring as rolled: from the scattered pool its outputs differ
    b2 = build_batch(layer, [RowSpec("spec", k, 3) for _ in range(5)], num_slots=48, spec_cols=k, seed=62)
    b2.spec = copy.copy(b2.spec)
    b2.spec.spec_state_indices = b1.spec.spec_state_indices.clone()
    good = run_oracle(b2, conv_pool=rolled.conv_pool.copy(), ssm_pool=rolled.ssm_pool.copy())
    bad = run_oracle(b2, conv_pool=scattered.conv_pool.copy(), ssm_pool=scattered.ssm_pool.copy())
    diff = np.abs(good.out_f64 - bad.out_f64).max()
    assert diff > 1e-3, diff

"""Test scenarios built from the seeded generators (shared by the oracle pins and GPU parity)."""
from __future__ import annotations

import copy
from typing import List

import torch

from gated_deltanet_linear_spec_gb300.workloads import Batch, LayerShape, RowSpec, Subset, build_batch


def relocate(batch: Batch, new_starts: List[int]) -> Batch:
    """The same rows with the same values, placed at other global token positions.

    Each subset keeps its local row order; x, a, b move with their tokens and token_indx is
    remapped, so a correct implementation gives every token the same output it had before
    (at its new position).  Returns the new batch; ``new_of_old`` maps old -> new positions.
    """
    T = batch.num_actual_tokens
    new_of_old = torch.empty(T, dtype=torch.long)
    for i, r in enumerate(batch.rows):
        o, n = batch.row_global_start[i], new_starts[i]
        new_of_old[o: o + r.length] = torch.arange(n, n + r.length)
    if sorted(new_of_old.tolist()) != list(range(T)):
        raise ValueError("new starts must tile the global tokens")
    nb = copy.copy(batch)
    for name in ("x", "a", "b"):
        src = getattr(batch, name)
        dst = torch.empty_like(src)
        dst[new_of_old] = src
        setattr(nb, name, dst)
    for name in ("spec", "non_spec"):
        s = getattr(batch, name)
        if s is None:
            continue
        tok = s.token_indx if s.token_indx is not None else torch.arange(s.num_tokens, dtype=torch.int32)
        ns = copy.copy(s)
        ns.token_indx = new_of_old[tok.long()].to(torch.int32)
        setattr(nb, name, ns)
    nb.row_global_start = list(new_starts)
    nb.new_of_old = new_of_old
    return nb


def with_subsets(batch: Batch, spec=None, non_spec=None, num_decodes=0, num_prefills=0) -> Batch:
    nb = copy.copy(batch)
    nb.spec, nb.non_spec = spec, non_spec
    nb.num_decodes, nb.num_prefills = num_decodes, num_prefills
    return nb


def p3_layout(layer: LayerShape, golden: dict, seed: int, spec_cols: int = 4) -> Batch:
    """The page-3 reachability composition: spec and non-spec rows at the printed token starts."""
    rows, starts = [], []
    for st, ln in zip(golden["spec_row_global_starts"], golden["spec_row_lengths"]):
        rows.append(RowSpec("spec", ln, 1 + (st // 4) % spec_cols)); starts.append(st)
    for st, ln in zip(golden["non_spec_row_global_starts"], golden["non_spec_row_lengths"]):
        rows.append(RowSpec("prefill" if ln > 1 else "decode", ln)); starts.append(st)
    return build_batch(layer, rows, num_slots=64, spec_cols=spec_cols, seed=seed, starts=starts,
                       force_token_indx=True)


def accepted_prefix_pair(layer: LayerShape, n_acc: int, seed: int, k_call: int = 4, prev_acc: int = 2):
    """Two ways to reach the same next step (the rollback contract of the spec path).

    Path A: a spec step over k_call verify tokens (history anchor prev_acc-1, SSM load from
    column prev_acc-1), then a spec step B with num_accepted = n_acc.
    Path A': a non-spec step over only the first n_acc of those tokens, starting from the same
    conv history and SSM state, then the same step B as a spec row with num_accepted = 1
    whose column 0 is the non-spec slot.
    Returns (stepA, stepB, stepA2, stepB2); every step is a Batch sharing one pool pair.
    """
    gen = torch.Generator().manual_seed(seed)
    base = build_batch(layer, [RowSpec("spec", k_call, prev_acc)], num_slots=16, spec_cols=k_call, seed=seed)
    ssi = base.spec.spec_state_indices.clone()               # [1, k_call], distinct, > 0
    used = set(ssi.view(-1).tolist())
    free = [p for p in range(1, 16) if p not in used]
    c_ns = free[0]                                           # slot of the non-spec path
    fresh = torch.tensor([[c_ns] + free[1: k_call]], dtype=torch.int32)
    W = layer.conv_width
    # Pools: the non-spec slot starts from what path A reads (conv anchor prev_acc-1, SSM column prev_acc-1)
    conv_pool = base.conv_pool.clone()
    ssm_pool = base.ssm_pool.clone()
    s0, sload = int(ssi[0, 0]), int(ssi[0, prev_acc - 1])
    conv_pool[c_ns, : W - 1] = conv_pool[s0, prev_acc - 1: prev_acc - 1 + W - 1]
    ssm_pool[c_ns] = ssm_pool[sload]
    C, Hv = layer.channels, layer.num_v_heads
    act = layer.act_dtype
    xB = torch.randn((k_call, C), generator=gen).to(act)
    aB = torch.randn((k_call, Hv), generator=gen).to(act)
    bB = torch.randn((k_call, Hv), generator=gen).to(act)
    q1 = lambda n: torch.tensor([0, n], dtype=torch.int32)  # noqa: E731

    stepA = copy.copy(base)
    stepA.conv_pool, stepA.ssm_pool = conv_pool, ssm_pool
    stepB = copy.copy(stepA)
    stepB.x, stepB.a, stepB.b = xB, aB, bB
    stepB.spec = Subset(q1(k_call), None, spec_state_indices=ssi,
                        num_accepted_tokens=torch.tensor([n_acc], dtype=torch.int32))
    stepA2 = copy.copy(stepA)
    stepA2.x, stepA2.a, stepA2.b = base.x[:n_acc].clone(), base.a[:n_acc].clone(), base.b[:n_acc].clone()
    stepA2.spec = None
    stepA2.non_spec = Subset(q1(n_acc), None, state_indices=torch.tensor([c_ns], dtype=torch.int32),
                             has_initial_state=torch.tensor([1], dtype=torch.int32))
    stepA2.num_decodes, stepA2.num_prefills = (1, 0) if n_acc == 1 else (0, 1)
    stepB2 = copy.copy(stepB)
    stepB2.spec = Subset(q1(k_call), None, spec_state_indices=fresh,
                         num_accepted_tokens=torch.tensor([1], dtype=torch.int32))
    return stepA, stepB, stepA2, stepB2

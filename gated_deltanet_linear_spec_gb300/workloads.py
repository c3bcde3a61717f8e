"""Seeded synthetic inputs for the GDN speculative-decoding path.

This module only draws random numbers and lays out index tensors; it holds none of the
method's arithmetic.  The tests, the smoke check and the bench build their inputs here and
hand the same bits to the CUDA library and to the CPU oracle.

Value distributions (all drawn with a seeded ``torch.Generator`` on the CPU):
  x (the packed q|k|v activations), a, b ~ N(0, 1) in the activation dtype;
  A_log = log U[1, 16]; dt_bias ~ N(0, 0.1); conv weights ~ N(0, 0.5);
  prior conv pool ~ N(0, 1) (activation dtype) and prior SSM pool ~ N(0, 1) (fp32), so that
  every slot holds data and "untouched" can be checked byte for byte.
Slots are distinct draws from 1..P-1 (slot 0 is reserved as NULL); NULL entries are set to 0
at seeded positions.

Row kinds follow the pages' vocabulary: ``spec`` rows verify drafts (their tokens are the
"verify tokens", K_call = drafts + 1 at most), ``decode`` rows are one-token non-spec rows,
``prefill`` rows are non-spec rows of any length.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import List, Optional

import torch


@dataclass
class LayerShape:
    num_k_heads: int
    num_v_heads: int
    head_k_dim: int
    head_v_dim: int
    conv_width: int = 4
    conv_state_len: int = 3
    act_dtype: torch.dtype = torch.bfloat16
    qkv_layout: int = 0   # 0: x packed q|k|v; 1: x per k-head groups
    conv_layout: int = 0  # 0: rolled spec conv history at column 0; 1: one snapshot per spec slot

    @property
    def channels(self) -> int:
        return 2 * self.num_k_heads * self.head_k_dim + self.num_v_heads * self.head_v_dim


def per_khead_order(layer: "LayerShape") -> torch.Tensor:
    """Index vector P with x_per_khead[:, P[c]] = x_packed[:, c]: for each k-head g the group
    q_g | k_g | v of the g-th block of Hv/Hk v-heads (the reorder_input=False projection order)."""
    Hk, Hv, dk, dv = layer.num_k_heads, layer.num_v_heads, layer.head_k_dim, layer.head_v_dim
    G = Hv // Hk
    group = 2 * dk + G * dv
    pos = []
    for kind in ("q", "k"):
        for g in range(Hk):
            base = g * group + (0 if kind == "q" else dk)
            pos += list(range(base, base + dk))
    for hv in range(Hv):
        base = (hv // G) * group + 2 * dk + (hv % G) * dv
        pos += list(range(base, base + dv))
    return torch.tensor(pos, dtype=torch.long)


def with_layouts(batch: "Batch", qkv_layout: int = 0, conv_layout: int = 0) -> "Batch":
    """The same packed-order batch seen through other layouts: with qkv_layout 1 the x columns
    are moved to the per-k-head order; conv_layout only changes how the conv pool is read and
    written, so the drawn pool stays as it is.  Every other tensor is shared."""
    import copy
    import dataclasses
    if batch.layer.qkv_layout != 0:
        raise ValueError("with_layouts expects a batch in the packed x order")
    nb = copy.copy(batch)
    nb.layer = dataclasses.replace(batch.layer, qkv_layout=qkv_layout, conv_layout=conv_layout)
    if qkv_layout == 1:
        x = torch.empty_like(batch.x)
        x[:, per_khead_order(batch.layer)] = batch.x
        nb.x = x
    return nb


# The layer the pages' production traffic runs (Qwen3-Next-style GDN): 16 k-heads, 32 v-heads,
# head dims 128, width-4 conv over 8192 packed channels.
def big_layer(state_len: int, act_dtype: torch.dtype = torch.bfloat16) -> LayerShape:
    return LayerShape(16, 32, 128, 128, 4, state_len, act_dtype)


@dataclass
class RowSpec:
    kind: str                      # "spec" | "decode" | "prefill"
    length: int
    num_accepted: int = 1          # spec and aware rows: accepted tokens of the previous step, 1..spec_cols
    has_initial_state: bool = True  # non-spec rows
    aware: bool = False            # non-spec rows: carries its previous verify step's acceptance


@dataclass
class Subset:
    """Index tensors of one subset (int32, CPU).  ``token_indx`` None means identity."""
    query_start_loc: torch.Tensor
    token_indx: Optional[torch.Tensor] = None
    state_indices: Optional[torch.Tensor] = None
    has_initial_state: Optional[torch.Tensor] = None
    spec_state_indices: Optional[torch.Tensor] = None
    num_accepted_tokens: Optional[torch.Tensor] = None

    @property
    def is_spec(self) -> bool:
        # a non-spec subset may carry spec_state_indices too (acceptance-aware rows)
        return self.spec_state_indices is not None and self.state_indices is None

    @property
    def num_seqs(self) -> int:
        return self.query_start_loc.numel() - 1

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def spec_cols(self) -> int:
        return 0 if self.spec_state_indices is None else int(self.spec_state_indices.shape[1])


@dataclass
class Batch:
    layer: LayerShape
    conv_w: torch.Tensor                 # [C, W] act
    conv_b: Optional[torch.Tensor]       # [C] act or None
    A_log: torch.Tensor                  # [Hv] fp32
    dt_bias: torch.Tensor                # [Hv] fp32
    conv_pool: torch.Tensor              # [P, state_len, C] act
    ssm_pool: torch.Tensor               # [P, Hv, dv, dk] fp32
    x: torch.Tensor                      # [T, C] act (pre-conv, global token order)
    a: torch.Tensor                      # [T, Hv] act
    b: torch.Tensor                      # [T, Hv] act
    spec: Optional[Subset]
    non_spec: Optional[Subset]
    num_decodes: int
    num_prefills: int
    rows: List[RowSpec] = field(default_factory=list)
    row_global_start: List[int] = field(default_factory=list)  # global first token of each RowSpec

    @property
    def num_actual_tokens(self) -> int:
        return self.x.shape[0]


def _randn(shape, gen, std=1.0, dtype=torch.float32):
    return (torch.randn(shape, generator=gen, dtype=torch.float32) * std).to(dtype)


_POOL_CHUNK = 8  # slots per independently seeded block


def _pool_randn(shape, seed: int, tag: int, dtype) -> torch.Tensor:
    """N(0, 1) pool [P, ...]: block j of _POOL_CHUNK slots comes from its own generator seeded
    by (seed, tag, j), so the values do not depend on how many threads fill them."""
    out = torch.empty(shape, dtype=dtype)
    P = shape[0]
    blocks = list(range(0, P, _POOL_CHUNK))

    def fill(j0):
        g = torch.Generator().manual_seed((int(seed) * 1_000_003 + int(tag) * 65_537 + j0 // _POOL_CHUNK) & 0x7FFFFFFFFFFF)
        n = min(_POOL_CHUNK, P - j0)
        out[j0:j0 + n] = torch.randn((n,) + tuple(shape[1:]), generator=g).to(dtype)

    if len(blocks) <= 2:
        for j0 in blocks:
            fill(j0)
    else:
        with ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1))) as ex:
            list(ex.map(fill, blocks))
    return out


def build_batch(layer: LayerShape, rows: List[RowSpec], *, num_slots: int, spec_cols: int = 0,
                seed: int = 0, null_frac: float = 0.0, spec_nulls: Optional[List[tuple]] = None,
                non_spec_nulls: Optional[List[int]] = None, shuffle_from: Optional[int] = None,
                force_token_indx: bool = False, conv_bias: bool = False,
                starts: Optional[List[int]] = None) -> Batch:
    """Lay ``rows`` out in global token order and draw every input.

    ``shuffle_from``: rows at positions >= this index are placed in a seeded random global
    order (the rows before it keep their place at the front).  The spec subset lists spec
    rows in global order; the non-spec subset lists decode rows first, then prefill rows.
    ``spec_nulls`` puts 0 at the given (spec row, column) entries; ``null_frac`` puts 0 at
    round(null_frac * entries) seeded entries of spec_state_indices.  ``starts`` gives each
    row's first global token explicitly (the rows must tile 0..T-1).
    """
    gen = torch.Generator().manual_seed(seed)
    C, W, SL = layer.channels, layer.conv_width, layer.conv_state_len
    Hv, dk, dv, act = layer.num_v_heads, layer.head_k_dim, layer.head_v_dim, layer.act_dtype

    order = list(range(len(rows)))
    if shuffle_from is not None and shuffle_from < len(rows):
        tail = order[shuffle_from:]
        perm = torch.randperm(len(tail), generator=gen).tolist()
        order = order[:shuffle_from] + [tail[i] for i in perm]
    row_start = [0] * len(rows)
    pos = 0
    for r in order:
        row_start[r] = pos
        pos += rows[r].length
    T = pos
    if starts is not None:
        covered = sorted(t for i, r in enumerate(rows) for t in range(starts[i], starts[i] + r.length))
        if covered != list(range(T)):
            raise ValueError("explicit row starts must tile the global tokens exactly")
        row_start = list(starts)

    spec_ids = sorted([i for i, r in enumerate(rows) if r.kind == "spec"], key=lambda i: row_start[i])
    dec_ids = sorted([i for i, r in enumerate(rows) if r.kind == "decode"], key=lambda i: row_start[i])
    pre_ids = sorted([i for i, r in enumerate(rows) if r.kind == "prefill"], key=lambda i: row_start[i])
    ns_ids = dec_ids + pre_ids

    aware = any(rows[i].aware for i in ns_ids)
    if aware and spec_cols < 1:
        raise ValueError("acceptance-aware rows need spec_cols >= 1")
    base_need = len(spec_ids) * spec_cols + len(ns_ids)
    need = base_need + (len(ns_ids) * (spec_cols - 1) if aware else 0)
    if need > num_slots - 1:
        raise ValueError(f"pool of {num_slots} slots cannot give {need} distinct non-NULL slots")
    slots = (torch.randperm(num_slots - 1, generator=gen)[:need] + 1).to(torch.int32)

    def subset(ids, is_spec):
        if not ids:
            return None
        lens = [rows[i].length for i in ids]
        qsl = torch.tensor([0] + list(torch.tensor(lens).cumsum(0).tolist()), dtype=torch.int32)
        tok = torch.cat([torch.arange(row_start[i], row_start[i] + rows[i].length) for i in ids]).to(torch.int32)
        return qsl, tok

    spec = non_spec = None
    if spec_ids:
        qsl, tok = subset(spec_ids, True)
        ssi = slots[: len(spec_ids) * spec_cols].reshape(len(spec_ids), spec_cols).clone()
        n_entries = ssi.numel()
        k = int(round(null_frac * n_entries))
        if k:
            flat = ssi.view(-1)
            flat[torch.randperm(n_entries, generator=gen)[:k]] = 0
        for (rr, cc) in (spec_nulls or []):
            ssi[rr, cc] = 0
        na = torch.tensor([rows[i].num_accepted for i in spec_ids], dtype=torch.int32)
        spec = Subset(qsl, tok, spec_state_indices=ssi, num_accepted_tokens=na)
    if ns_ids:
        qsl, tok = subset(ns_ids, False)
        si = slots[len(spec_ids) * spec_cols: base_need].clone()
        for rr in (non_spec_nulls or []):
            si[rr] = 0
        hi = torch.tensor([int(rows[i].has_initial_state) for i in ns_ids], dtype=torch.int32)
        non_spec = Subset(qsl, tok, state_indices=si, has_initial_state=hi)
        if aware:
            # the previous verify step's slots: column 0 is the row's own slot (a block table
            # row), the others fresh; rows that are not aware accepted exactly one token
            ssi = torch.cat([si[:, None], slots[base_need:need].reshape(len(ns_ids), spec_cols - 1)], 1)
            non_spec.spec_state_indices = ssi.contiguous()
            non_spec.num_accepted_tokens = torch.tensor(
                [rows[i].num_accepted if rows[i].aware else 1 for i in ns_ids], dtype=torch.int32)

    # token_indx is only passed when it is not the identity (or when asked for).
    for s in (spec, non_spec):
        if s is not None and not force_token_indx:
            if s.num_tokens == T and torch.equal(s.token_indx, torch.arange(T, dtype=torch.int32)):
                s.token_indx = None

    conv_w = _randn((C, W), gen, 0.5, act)
    conv_b = _randn((C,), gen, 0.5, act) if conv_bias else None
    A_log = torch.log(torch.empty(Hv).uniform_(1.0, 16.0, generator=gen)).to(torch.float32)
    dt_bias = _randn((Hv,), gen, 0.1)
    conv_pool = _pool_randn((num_slots, SL, C), seed, 1, act)
    ssm_pool = _pool_randn((num_slots, Hv, dv, dk), seed, 2, torch.float32)
    x = _randn((T, C), gen, 1.0, act)
    a = _randn((T, Hv), gen, 1.0, act)
    b = _randn((T, Hv), gen, 1.0, act)
    return Batch(layer, conv_w, conv_b, A_log, dt_bias, conv_pool, ssm_pool, x, a, b, spec, non_spec,
                 len(dec_ids), len(pre_ids), rows, row_start)


def uniform_accepts(n: int, k_call: int, gen_seed: int) -> List[int]:
    g = torch.Generator().manual_seed(gen_seed)
    return (torch.randint(1, k_call + 1, (n,), generator=g)).tolist()


# ------------------------------------------------------------------------------------------
# The named workloads.

def tiny(seed: int = 0) -> Batch:
    """1 layer, Hk=2, Hv=4, dk=dv=16, width 4, fp32; 3 spec rows of 3 verify tokens (2 drafts),
    num_accepted uniform in {1,2,3}, a 16-slot pool with 9 distinct slots of which one is NULL."""
    layer = LayerShape(2, 4, 16, 16, 4, 5, torch.float32)
    acc = uniform_accepts(3, 3, seed + 100)
    rows = [RowSpec("spec", 3, acc[i]) for i in range(3)]
    null = [(int(seed % 3), int((seed // 3) % 3))]
    return build_batch(layer, rows, num_slots=16, spec_cols=3, seed=seed, spec_nulls=null)


def non_spec_decode(seed: int = 1, batch: int = 64) -> Batch:
    """Big layer, bf16 activations, fp32 state; 64 one-token rows; 256-slot pool."""
    rows = [RowSpec("decode", 1) for _ in range(batch)]
    return build_batch(big_layer(3), rows, num_slots=256, seed=seed)


def spec_verify(seed: int = 2, batch: int = 64, drafts: int = 3, num_slots: int = 512,
                null_frac: float = 0.05) -> Batch:
    """Big layer; 64 spec rows of drafts+1 = 4 verify tokens; num_accepted uniform in [1, 4];
    distinct random slots in a 512-slot pool with 5% of the spec_state_indices entries NULL."""
    k_call = drafts + 1
    acc = uniform_accepts(batch, k_call, seed + 100)
    rows = [RowSpec("spec", k_call, acc[i]) for i in range(batch)]
    return build_batch(big_layer(2 + k_call), rows, num_slots=num_slots, spec_cols=k_call, seed=seed,
                       null_frac=null_frac)


def mixed(seed: int = 3) -> Batch:
    """Big layer; 8 one-token non-spec rows first, then 32 spec rows of 4 tokens and 2 prefill rows
    (512 tokens from a fresh state, 1024 tokens continuing a prior one) in seeded order; both
    token_indx tensors are non-identity."""
    acc = uniform_accepts(32, 4, seed + 100)
    rows = [RowSpec("decode", 1) for _ in range(8)]
    rows += [RowSpec("spec", 4, acc[i]) for i in range(32)]
    rows += [RowSpec("prefill", 512, has_initial_state=False), RowSpec("prefill", 1024)]
    return build_batch(big_layer(6), rows, num_slots=512, spec_cols=4, seed=seed, shuffle_from=8)


def mixed_small(seed: int = 7) -> Batch:
    """A small bf16 mixed batch (1 k-head, 2 v-heads of 128) that still spans several tiles,
    conv segments, chunks and ragged tails: 3 decode rows first, then (seeded order) 5 spec rows
    of up to 4 tokens -- one of them ragged -- and 2 prefill rows of 70 and 130 tokens (one
    fresh)."""
    layer = LayerShape(1, 2, 128, 128, 4, 6, torch.bfloat16)
    acc = uniform_accepts(5, 4, seed + 100)
    rows = [RowSpec("decode", 1) for _ in range(3)]
    rows += [RowSpec("spec", 4 if i != 2 else 2, acc[i]) for i in range(5)]
    rows += [RowSpec("prefill", 70, has_initial_state=False), RowSpec("prefill", 130)]
    return build_batch(layer, rows, num_slots=48, spec_cols=4, seed=seed, shuffle_from=3, spec_nulls=[(1, 3)])


def sweep_point(drafts: int, batch: int, seed: int) -> Batch:
    """Spec verify at K drafts and the given batch over a 2048-slot pool (or batch*(K+1)+1 slots
    when 2048 cannot hold distinct slots for every verify token); no NULLs."""
    k_call = drafts + 1
    slots = max(2048, batch * k_call + 1)
    acc = uniform_accepts(batch, k_call, seed + 100)
    rows = [RowSpec("spec", k_call, acc[i]) for i in range(batch)]
    return build_batch(big_layer(2 + k_call), rows, num_slots=slots, spec_cols=k_call, seed=seed)


def long_prefill(length: int = 8192, seed: int = 20) -> Batch:
    """One chunked-prefill row continuing a prior state (the long-sequence point of the sweep)."""
    rows = [RowSpec("prefill", length)]
    return build_batch(big_layer(3), rows, num_slots=4, seed=seed)


def bytes_of(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else t.numel() * t.element_size()


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = ["LayerShape", "RowSpec", "per_khead_order", "with_layouts", "Subset", "Batch", "build_batch", "big_layer", "tiny",
           "non_spec_decode", "spec_verify", "mixed", "mixed_small", "sweep_point", "long_prefill",
           "uniform_accepts", "bytes_of", "ceil_div"]

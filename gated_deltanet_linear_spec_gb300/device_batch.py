"""Moves a seeded ``workloads.Batch`` to the GPU and builds the binding's descriptors for it."""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import Layer, Params, Pools, Rows, gdn_mixed_batch, mixed_batch_workspace_bytes
from .workloads import Batch, Subset


@dataclass
class DeviceBatch:
    layer: Layer
    params: Params
    pools: Pools
    x: torch.Tensor
    a: torch.Tensor
    b: torch.Tensor
    spec: Optional[Rows]
    non_spec: Optional[Rows]
    num_decodes: int
    num_prefills: int
    out: torch.Tensor
    workspace: torch.Tensor
    status: torch.Tensor

    def run(self, stream=None) -> None:
        """One pass of the whole path (gdn_mixed_batch) over this batch."""
        gdn_mixed_batch(self.layer, self.params, self.pools, self.x, self.a, self.b, self.non_spec,
                        self.num_decodes, self.num_prefills, self.spec, self.out, self.workspace,
                        self.status, stream)


def rows_to_device(s: Optional[Subset], device) -> Optional[Rows]:
    if s is None:
        return None
    d = lambda t: None if t is None else t.to(device=device, dtype=torch.int32).contiguous()  # noqa: E731
    return Rows(d(s.query_start_loc), s.num_tokens, d(s.token_indx), d(s.state_indices), d(s.has_initial_state),
                d(s.spec_state_indices), d(s.num_accepted_tokens))


def to_device(batch: Batch, device="cuda", pools: Optional[Pools] = None) -> DeviceBatch:
    L = batch.layer
    layer = Layer(L.num_k_heads, L.num_v_heads, L.head_k_dim, L.head_v_dim, L.conv_width, L.conv_state_len,
                  L.act_dtype, qkv_layout=L.qkv_layout, conv_layout=L.conv_layout)
    dev = lambda t: None if t is None else t.to(device).contiguous()  # noqa: E731
    params = Params(dev(batch.conv_w), dev(batch.A_log), dev(batch.dt_bias), dev(batch.conv_b))
    if pools is None:
        pools = Pools(dev(batch.conv_pool), dev(batch.ssm_pool))
    spec, non_spec = rows_to_device(batch.spec, device), rows_to_device(batch.non_spec, device)
    T = batch.num_actual_tokens
    out = torch.zeros((T, L.num_v_heads, L.head_v_dim), dtype=L.act_dtype, device=device)
    ws = torch.empty(max(1, mixed_batch_workspace_bytes(layer, non_spec, batch.num_prefills, spec)),
                     dtype=torch.uint8, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    return DeviceBatch(layer, params, pools, dev(batch.x), dev(batch.a), dev(batch.b), spec, non_spec,
                       batch.num_decodes, batch.num_prefills, out, ws, status)

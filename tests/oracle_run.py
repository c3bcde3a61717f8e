"""Test-side glue: run the CPU oracle over a seeded ``Batch`` (numpy copies, never the device)."""
from __future__ import annotations

import os
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

import oracle
from gated_deltanet_linear_spec_gb300.workloads import Batch, Subset


def np_act(t: torch.Tensor) -> np.ndarray:
    """A CPU tensor as the oracle's array: bf16 -> uint16 bits, fp32 -> float32 (copied)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    if t.dtype == torch.float32:
        return t.numpy().copy()
    if t.dtype == torch.int32:
        return t.numpy().copy()
    raise TypeError(t.dtype)


def act_to_f64(a: np.ndarray) -> np.ndarray:
    """Oracle activation array (uint16 bf16 bits or float32) as float64 values."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def oracle_layer(batch: Batch, scale: Optional[float] = None) -> oracle.Layer:
    L = batch.layer
    return oracle.Layer(L.num_k_heads, L.num_v_heads, L.head_k_dim, L.head_v_dim, L.conv_width,
                        L.conv_state_len, L.act_dtype == torch.bfloat16, scale,
                        qkv_layout=L.qkv_layout, conv_layout=L.conv_layout)


def oracle_rows(s: Optional[Subset]) -> Optional[oracle.Rows]:
    if s is None:
        return None
    f = lambda t: None if t is None else np_act(t)  # noqa: E731
    return oracle.Rows(f(s.query_start_loc), s.is_spec, f(s.token_indx), f(s.state_indices),
                       f(s.has_initial_state), f(s.spec_state_indices), f(s.num_accepted_tokens))


@dataclass
class OracleResult:
    conv_pool: np.ndarray
    ssm_pool: np.ndarray
    out: np.ndarray       # act dtype bits [T, Hv, dv]
    out_f64: np.ndarray   # unrounded outputs
    y: dict               # subset name -> post-conv q|k|v (float64, local order)


def run_oracle(batch: Batch, heads: Optional[tuple] = None, nthreads: Optional[int] = None,
               subsets=("spec", "non_spec"), conv_pool: Optional[np.ndarray] = None,
               ssm_pool: Optional[np.ndarray] = None, precision: str = "f64") -> OracleResult:
    """The whole path (conv, then gated delta rule) over the batch's subsets, on pool copies.
    ``precision="f32"`` runs the oracle's float build instead (a rounding-noise measurement)."""
    L = oracle_layer(batch)
    T, Hv, dv = batch.num_actual_tokens, batch.layer.num_v_heads, batch.layer.head_v_dim
    cp = np_act(batch.conv_pool) if conv_pool is None else conv_pool
    sp = np_act(batch.ssm_pool) if ssm_pool is None else ssm_pool
    x, a, b = np_act(batch.x), np_act(batch.a), np_act(batch.b)
    w = np_act(batch.conv_w)
    cb = None if batch.conv_b is None else np_act(batch.conv_b)
    A_log, dt_bias = np_act(batch.A_log), np_act(batch.dt_bias)
    out = np.zeros((T, Hv, dv), dtype=x.dtype)
    out_f64 = np.full((T, Hv, dv), np.nan, dtype=np.float64 if precision == "f64" else np.float32)
    nthreads = nthreads or max(1, len(os.sched_getaffinity(0)))
    ys = {}
    for name in subsets:
        rows = oracle_rows(getattr(batch, name))
        if rows is None or rows.num_seqs == 0:
            continue
        y = oracle.conv_update(L, w, cb, cp, x, T, rows, precision)
        ys[name] = y
        oracle.recurrent(L, A_log, dt_bias, sp, y, a, b, T, rows, out, out_f64, heads, nthreads, precision)
    return OracleResult(cp, sp, out, out_f64, ys)

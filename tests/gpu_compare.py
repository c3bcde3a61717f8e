"""GPU-vs-oracle comparison helpers for the parity tests (the oracle side never sees GPU data).

Tolerances (the target's, written out here):
  outputs, bf16 activations:  |gpu - ref| <= 2e-2 + 2e-2 |ref|   (ref = the oracle's fp64 value)
  outputs, fp32 activations:  |gpu - ref| <= 1e-4 + 1e-4 |ref|   (derived: the state bound below
                              applied to o = S q^ with |q^| <= 1/sqrt(dk))
  fp32 state per (slot, head):  ||gpu - ref||_F <= 1e-4 ||ref||_F
  conv ring, set of written slots, untouched slots: bit-exact.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from gated_deltanet_linear_spec_gb300.device_batch import to_device
from gated_deltanet_linear_spec_gb300.workloads import Batch
from tests.oracle_run import OracleResult, act_to_f64, np_act

BF16_TOL = 2e-2
F32_TOL = 1e-4
STATE_REL = 1e-4


@dataclass
class GpuResult:
    out: np.ndarray        # act bits / fp32 [T, Hv, dv]
    conv_pool: np.ndarray  # act bits
    ssm_pool: np.ndarray   # fp32
    status: int


def run_gpu(batch: Batch, runs: int = 1) -> GpuResult:
    db = to_device(batch)
    for _ in range(runs):
        db.run()
    torch.cuda.synchronize()
    res = GpuResult(np_act(db.out.cpu()), np_act(db.pools.conv_pool.cpu()), db.pools.ssm_pool.cpu().numpy(),
                    int(db.status.item()))
    del db
    return res


def changed_slots(pre: np.ndarray, post: np.ndarray, heads: Optional[tuple] = None) -> set:
    if heads is not None:
        pre, post = pre[:, heads[0]:heads[1]], post[:, heads[0]:heads[1]]
    flat_pre = pre.reshape(pre.shape[0], -1).view(np.uint32) if pre.dtype == np.float32 else pre.reshape(pre.shape[0], -1)
    flat_post = post.reshape(post.shape[0], -1).view(np.uint32) if post.dtype == np.float32 else post.reshape(post.shape[0], -1)
    return set(np.nonzero((flat_pre != flat_post).any(axis=1))[0].tolist())


def assert_outputs_close(gpu_out: np.ndarray, ref: OracleResult, bf16: bool, heads: Optional[tuple] = None,
                         rows_mask: Optional[np.ndarray] = None):
    mask = ~np.isnan(ref.out_f64)
    if rows_mask is not None:
        mask &= rows_mask[:, None, None]
    g = act_to_f64(gpu_out)[mask]
    r = ref.out_f64[mask]
    tol = BF16_TOL if bf16 else F32_TOL
    bad = np.abs(g - r) > tol + tol * np.abs(r)
    assert mask.any(), "no outputs were compared"
    assert not bad.any(), (f"{int(bad.sum())} of {bad.size} outputs off; worst |d|="
                           f"{float(np.abs(g - r).max()):.3e}")


def assert_states_close(pre_ssm: np.ndarray, gpu_ssm: np.ndarray, ref_ssm: np.ndarray, heads: Optional[tuple] = None):
    """Written slots agree exactly as a set; each written (slot, head) within STATE_REL; every
    other slot is bit-identical to its prior value on the GPU."""
    exp = changed_slots(pre_ssm, ref_ssm, heads)
    got_all = changed_slots(pre_ssm, gpu_ssm)
    assert got_all == exp, f"written SSM slots differ: only gpu {sorted(got_all - exp)[:8]}, only ref {sorted(exp - got_all)[:8]}"
    h0, h1 = heads if heads is not None else (0, pre_ssm.shape[1])
    worst = 0.0
    for s in exp:
        for h in range(h0, h1):
            r = ref_ssm[s, h].astype(np.float64)
            d = gpu_ssm[s, h].astype(np.float64) - r
            nr = np.linalg.norm(r)
            rel = np.linalg.norm(d) / (nr if nr > 0 else 1.0)
            worst = max(worst, rel)
    assert worst <= STATE_REL, f"state rel error {worst:.3e} > {STATE_REL}"
    return worst


def assert_parity(batch: Batch, gpu: GpuResult, ref: OracleResult, heads: Optional[tuple] = None):
    bf16 = batch.layer.act_dtype == torch.bfloat16
    assert gpu.status == 0, f"device status {gpu.status:#x}"
    assert_outputs_close(gpu.out, ref, bf16, heads)
    assert np.array_equal(gpu.conv_pool, ref.conv_pool), "conv ring differs"
    return assert_states_close(batch.ssm_pool.numpy(), gpu.ssm_pool, ref.ssm_pool, heads)

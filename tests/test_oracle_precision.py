"""The rounding noise of the definition in fp32, against the tolerances (CPU only).

The oracle works in double.  Its float build takes exactly the same steps in float, so the gap
between the two is the rounding noise that any fp32 token-by-token implementation of the
definition carries.  These tests bound that gap far below the parity tolerances of
``tests/gpu_compare.py`` (fp32 state: 1e-4 relative per (slot, head); fp32 outputs: 1e-4 +
1e-4 |ref|), so a parity failure cannot come from fp32 rounding alone; and they check that the
float build really rounds (it must not reproduce the double results bit for bit).
"""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_spec_gb300 import workloads as W
from gated_deltanet_linear_spec_gb300.workloads import LayerShape, RowSpec, build_batch
from tests.oracle_run import run_oracle

STATE_NOISE = 1e-6   # observed <= 3e-7
OUT_NOISE = 1e-6     # absolute; observed <= 1e-7 with |o| <= 0.25


def _cases():
    return {
        "spec_verify": (W.spec_verify(), (0, 2)),
        "mixed_small": (W.mixed_small(), None),
        "prefill_512": (build_batch(LayerShape(1, 2, 128, 128, 4, 6, torch.bfloat16), [RowSpec("prefill", 512)],
                                    num_slots=8, seed=5), None),
        "tiny_fp32": (W.tiny(0), None),
    }


@pytest.mark.parametrize("name", list(_cases()))
def test_fp32_rounding_noise_is_far_below_the_tolerances(name):
    batch, heads = _cases()[name]
    r64 = run_oracle(batch, heads=heads)
    r32 = run_oracle(batch, heads=heads, precision="f32")
    pre = batch.ssm_pool.numpy()
    P = pre.shape[0]
    written = np.nonzero((r64.ssm_pool.reshape(P, -1) != pre.reshape(P, -1)).any(axis=1))[0]
    assert len(written) > 0
    h0, h1 = heads if heads else (0, batch.layer.num_v_heads)
    worst = 0.0
    for s in written:
        for h in range(h0, h1):
            a64 = r64.ssm_pool[s, h].astype(np.float64)
            a32 = r32.ssm_pool[s, h].astype(np.float64)
            worst = max(worst, float(np.linalg.norm(a32 - a64) / np.linalg.norm(a64)))
    assert 0.0 < worst <= STATE_NOISE
    m = ~np.isnan(r64.out_f64)
    gap = np.abs(r32.out_f64[m].astype(np.float64) - r64.out_f64[m])
    assert gap.max() <= OUT_NOISE
    # the float build rounds: some stored state differs from the double build's
    assert not np.array_equal(r32.ssm_pool, r64.ssm_pool)

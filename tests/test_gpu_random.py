"""GPU parity on seeded random configurations of everything the library accepts at once.

Each case draws a layer (k-heads, GQA ratio, dk in {16, 32, 64, 128}, dv a multiple of 16, bf16 or
fp32 activations, conv width 2-4, both x layouts and both conv layouts, a conv slot of the
smallest legal length or a little more, optional conv bias) and a mixed batch of spec rows
(ragged lengths up to the verify width, any acceptance, NULL entries), decode rows and prefill
rows (lengths that end inside a chunk, span several 64-token chunks, or are two tokens),
acceptance-aware and fresh rows, NULL non-spec slots, in a shuffled global order; the GPU
result is compared with the oracle's on the same inputs with the tolerances of
``tests/gpu_compare.py``.  The spec contract and its edge cases come from "[GDN]
Spec-decoding-aware attention kernel" (Changes), the mixed split from "[Bugfix] Align Qwen GDN
gates with speculative tokens" (Purpose) and the layouts from "[XE2] Support MTP of QWEN model".
"""
import random

import pytest
import torch

from gated_deltanet_linear_spec_gb300.workloads import LayerShape, RowSpec, build_batch, with_layouts
from tests.gpu_compare import assert_parity, run_gpu
from tests.oracle_run import run_oracle

pytestmark = pytest.mark.gpu


def random_case(seed: int, chunked: bool = False):
    """One random layer and batch; ``chunked`` fixes the layer the tensor-core prefill takes
    (dk = dv = 128, bf16) and adds a prefill row of several chunks."""
    rng = random.Random(seed)
    hk = rng.choice([1, 2, 4])
    hv = hk * rng.choice([1, 2, 4])
    dk = rng.choice([16, 32, 64, 128, 128])
    dv = rng.choice([16, 32, 48, 64, 128, 128]) if dk != 128 else rng.choice([32, 64, 128, 128])
    act = rng.choice([torch.bfloat16, torch.bfloat16, torch.float32])
    if chunked:
        dk, dv, act = 128, 128, torch.bfloat16
    width = rng.choice([2, 3, 4, 4])
    k = rng.randint(1, 6)
    conv_layout, qkv_layout = rng.randint(0, 1), rng.randint(0, 1)
    state_len = (width - 2 + k if conv_layout == 0 else width - 1) + rng.choice([0, 0, 1, 3])
    state_len = max(state_len, width - 1)
    layer = LayerShape(hk, hv, dk, dv, width, state_len, act)

    rows = []
    for _ in range(rng.randint(0, 6)):
        rows.append(RowSpec("spec", rng.randint(1, k), rng.randint(1, k)))
    for _ in range(rng.randint(0, 4)):
        aware = rng.random() < 0.4
        rows.append(RowSpec("decode", 1, rng.randint(1, k) if aware else 1, rng.random() > 0.2, aware))
    for _ in range(rng.randint(0, 3)):
        aware = rng.random() < 0.3
        length = rng.choice([2, rng.randint(3, 63), rng.randint(65, 150), 64, 128])
        rows.append(RowSpec("prefill", length, rng.randint(1, k) if aware else 1, rng.random() > 0.25, aware))
    if chunked:
        rows.append(RowSpec("prefill", rng.randint(129, 300), rng.randint(1, k), rng.random() > 0.2, rng.random() < 0.5))
    if not rows:
        rows.append(RowSpec("spec", k, rng.randint(1, k)))

    n_spec = sum(r.kind == "spec" for r in rows)
    n_ns = len(rows) - n_spec
    spec_nulls = [(rng.randrange(n_spec), rng.randrange(k)) for _ in range(rng.randint(0, 2))] if n_spec else None
    ns_nulls = [rng.randrange(n_ns)] if n_ns and rng.random() < 0.3 else None
    need = n_spec * k + n_ns * k
    b = build_batch(layer, rows, num_slots=need + 1 + rng.randint(0, 8), spec_cols=k, seed=1000 + seed,
                    spec_nulls=spec_nulls, non_spec_nulls=ns_nulls, shuffle_from=0,
                    conv_bias=rng.random() < 0.5)
    return with_layouts(b, qkv_layout=qkv_layout, conv_layout=conv_layout)


@pytest.mark.parametrize("seed", range(64))
def test_random_configuration(seed):
    b = random_case(seed)
    assert_parity(b, run_gpu(b), run_oracle(b))


@pytest.mark.parametrize("seed", range(100, 116))
def test_random_configuration_on_the_chunked_prefill_layer(seed):
    b = random_case(seed, chunked=True)
    assert_parity(b, run_gpu(b), run_oracle(b))

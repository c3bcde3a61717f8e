"""GPU parity at the edges of the accepted shapes: the largest verify width (64 tokens per spec
row, the limit of one conv work unit) in both conv layouts, conv widths 2 and 3, fp32
activations with a token-recurrence prefill, and head sizes the chunked path does not take."""
import pytest
import torch

from gated_deltanet_linear_spec_gb300.workloads import LayerShape, RowSpec, build_batch, with_layouts
from tests.gpu_compare import assert_parity, run_gpu
from tests.oracle_run import run_oracle

pytestmark = pytest.mark.gpu


def _parity(batch):
    assert_parity(batch, run_gpu(batch), run_oracle(batch))


@pytest.mark.parametrize("conv_layout", [0, 1])
def test_widest_verify_rows(conv_layout):
    k = 64
    layer = LayerShape(2, 4, 32, 32, 4, k + 2 if conv_layout == 0 else 3, torch.bfloat16)
    rows = [RowSpec("spec", 64, 64), RowSpec("spec", 33, 17), RowSpec("spec", 1, 1), RowSpec("spec", 64, 1),
            RowSpec("decode", 1), RowSpec("prefill", 100)]
    b = build_batch(layer, rows, num_slots=4 * k + 8, spec_cols=k, seed=91, shuffle_from=0,
                    spec_nulls=[(0, 5), (1, 16), (3, 63)])
    _parity(with_layouts(b, conv_layout=conv_layout))


@pytest.mark.parametrize("width", [2, 3])
def test_narrow_convs(width):
    layer = LayerShape(2, 4, 64, 64, width, width - 2 + 4, torch.bfloat16)
    rows = [RowSpec("spec", 4, 1 + i % 4) for i in range(6)] + [RowSpec("decode", 1), RowSpec("prefill", 70)]
    _parity(build_batch(layer, rows, num_slots=48, spec_cols=4, seed=90 + width, shuffle_from=0, conv_bias=True))


def test_fp32_activations_with_prefill_rows():
    layer = LayerShape(2, 4, 128, 128, 4, 6, torch.float32)
    rows = [RowSpec("spec", 4, 3), RowSpec("spec", 2, 1), RowSpec("decode", 1),
            RowSpec("prefill", 130), RowSpec("prefill", 9, has_initial_state=False)]
    _parity(build_batch(layer, rows, num_slots=32, spec_cols=4, seed=93, shuffle_from=0))


@pytest.mark.parametrize("dims", [(16, 16), (64, 128), (128, 64), (128, 256), (32, 48)])
def test_head_sizes(dims):
    dk, dv = dims
    layer = LayerShape(1, 2, dk, dv, 4, 6, torch.bfloat16)
    rows = [RowSpec("spec", 4, 2), RowSpec("spec", 3, 3), RowSpec("decode", 1), RowSpec("prefill", 66)]
    _parity(build_batch(layer, rows, num_slots=24, spec_cols=4, seed=94 + dk + dv, shuffle_from=0))

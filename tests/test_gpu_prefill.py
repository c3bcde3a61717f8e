"""GPU tests of the tensor-core chunked prefill (gdn_chunk_prefill and the prefill rows of
gdn_mixed_batch): it equals the token recurrence of the same rows (the invariant "chunked prefill
equals the per-token recurrence") and the oracle, on ragged lengths around the 64-token chunk,
fresh and continued states, NULL slots, and fp32 or bf16 post-conv inputs."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_spec_gb300 as gdn
from gated_deltanet_linear_spec_gb300.device_batch import to_device
from gated_deltanet_linear_spec_gb300.workloads import LayerShape, RowSpec, build_batch
from tests.gpu_compare import assert_outputs_close, assert_parity, assert_states_close, run_gpu
from tests.oracle_run import np_act, run_oracle

pytestmark = pytest.mark.gpu
LAYER = LayerShape(2, 4, 128, 128, 4, 3, torch.bfloat16)


def _prefill_batch(lengths, seed, fresh=(), nulls=()):
    rows = [RowSpec("prefill", L, has_initial_state=(i not in fresh)) for i, L in enumerate(lengths)]
    return build_batch(LAYER, rows, num_slots=4 * len(lengths) + 4, seed=seed, non_spec_nulls=list(nulls))


@pytest.mark.parametrize("lengths", [[1], [63], [64], [65], [200, 5, 128, 64]])
def test_chunked_prefill_matches_oracle(lengths):
    batch = _prefill_batch(lengths, seed=sum(lengths), fresh=(0,))
    assert_parity(batch, run_gpu(batch), run_oracle(batch))


def test_chunked_prefill_null_slot_and_fresh_rows():
    batch = _prefill_batch([90, 33, 150], seed=5, fresh=(1,), nulls=(2,))
    assert_parity(batch, run_gpu(batch), run_oracle(batch))


@pytest.mark.parametrize("qkv_dtype", [torch.float32, torch.bfloat16])
def test_chunked_prefill_equals_token_recurrence(qkv_dtype):
    batch = _prefill_batch([300, 77, 129], seed=7, fresh=(1,))
    ref = run_oracle(batch)
    y = torch.from_numpy(ref.y["non_spec"]).to(qkv_dtype).cuda()
    outs, pools = [], []
    for chunked in (True, False):
        d = to_device(batch)
        if chunked:
            gdn.gdn_chunk_prefill(d.layer, d.params, d.pools, y, d.a, d.b, d.non_spec, d.out, status=d.status)
        else:
            gdn.gdn_recurrent_step(d.layer, d.params, d.pools, y, d.a, d.b, d.non_spec, d.out, d.status)
        torch.cuda.synchronize()
        assert int(d.status.item()) == 0
        outs.append(np_act(d.out.cpu()))
        pools.append(d.pools.ssm_pool.cpu().numpy())
    tok = type("R", (), {"out_f64": np.where(np.isnan(ref.out_f64), np.nan,
                                               (outs[1].astype(np.uint32) << 16).view(np.float32).astype(np.float64))})
    assert_outputs_close(outs[0], tok, bf16=True)
    assert_states_close(batch.ssm_pool.numpy(), pools[0], pools[1])


def test_prefill_workspace_is_required():
    batch = _prefill_batch([100], seed=9)
    d = to_device(batch)
    y = torch.zeros((100, LAYER.channels), device="cuda")
    need = gdn.gdn_prefill_workspace_bytes(d.layer, d.non_spec, 1)
    assert need > 0
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_chunk_prefill(d.layer, d.params, d.pools, y, d.a, d.b, d.non_spec, d.out, workspace=small)
    assert e.value.name == "WORKSPACE"

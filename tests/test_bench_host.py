"""The bench's host arithmetic behind the roofline numbers (CPU only): the algorithmic bytes of
the recurrence and the FLOPs of the chunked prefill, recounted here from the batch's own index
tensors and the chunk-form operation counts, independently of the bench's loops."""
import torch

import bench
from gated_deltanet_linear_spec_gb300 import workloads as W

MIB2 = 2 * 1024 * 1024  # one SSM slot of the big layer: Hv * dv * dk * 4 bytes


def test_spec_verify_recurrence_bytes():
    b = W.spec_verify()
    ssi, na = b.spec.spec_state_indices, b.spec.num_accepted_tokens.long()
    assert b.spec.num_tokens == ssi.numel()              # every row has all spec_cols tokens
    loads = int((ssi.gather(1, (na - 1)[:, None]) > 0).sum())
    stores = int((ssi > 0).sum())
    assert (loads, stores) == (61, 243)                  # 5% of 256 entries NULL, seeded
    T, Hv, dv = b.num_actual_tokens, b.layer.num_v_heads, b.layer.head_v_dim
    expected = (loads + stores) * MIB2 + T * (2 * Hv * 2 + Hv * dv * 2)  # states; a, b and out in bf16
    alg = bench.algorithmic_bytes(b)
    assert alg["recurrence"] == expected == 639_664_128
    assert (alg["state_loads"], alg["state_stores"]) == (loads, stores)


def test_non_spec_decode_bytes_count_one_load_and_one_store_per_row():
    b = W.non_spec_decode()
    si = b.non_spec.state_indices
    rows = int((si > 0).sum())
    alg = bench.algorithmic_bytes(b)
    assert alg["state_loads"] == alg["state_stores"] == rows
    assert alg["ssm"] == 2 * rows * MIB2


def test_prefill_flops_of_the_chunk_form():
    b = W.long_prefill(8192)
    c, d, Hv = 64, 128, b.layer.num_v_heads
    chunks = 8192 // c
    # per (chunk, v-head): 5 c^2 d + 3 c d^2 + c^3 / 6 multiply-adds, two FLOPs each
    per_chunk = 2 * (5 * c * c * d + 3 * c * d * d + c ** 3 / 6)
    assert abs(per_chunk - 11.6e6) < 0.05e6
    assert bench.prefill_flops(b) == chunks * Hv * per_chunk
    assert abs(bench.prefill_flops(b) - 47.6e9) < 0.1e9


def test_ragged_prefill_rows_round_up_to_whole_chunks():
    layer = W.LayerShape(1, 2, 128, 128, 4, 6, torch.bfloat16)
    b = W.build_batch(layer, [W.RowSpec("decode", 1), W.RowSpec("prefill", 65), W.RowSpec("prefill", 64)],
                      num_slots=16, seed=1)
    c, d = 64, 128
    per_chunk = 2 * (5 * c * c * d + 3 * c * d * d + c ** 3 / 6)
    assert bench.prefill_flops(b) == (2 + 1) * 2 * per_chunk   # 65 tokens -> 2 chunks, 64 -> 1; 2 v-heads


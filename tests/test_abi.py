"""The C ABI on the host (no GPU needed): the library loads, exports every function that
include/gdn.h declares, and rejects malformed calls with the documented code before it
enqueues anything ("[XE2] Support MTP of QWEN model": every optional tensor is checked before
use, the conservation check replaces the rectangular one; "[GDN] Spec-decoding-aware attention
kernel": the spec pair comes together).

Every call below is built to fail validation, so no kernel is ever launched with the fake
pointers used here (on a GPU machine as well as without one).
"""
import ctypes
import os
import re

import pytest

import gated_deltanet_linear_spec_gb300 as gdn
from gated_deltanet_linear_spec_gb300 import _LayerDesc, _LayerParams, _Pools, _Rows

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADER = os.path.join(INCLUDE, "gdn.h")
TESTING_HEADER = os.path.join(INCLUDE, "gdn_testing.h")
FAKE = 0x100000  # an aligned non-NULL address; never dereferenced because validation fails first


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(gdn.LIB_PATH):
        from gated_deltanet_linear_spec_gb300 import build
        build.build()
    return gdn.library()


def declared_functions(header=HEADER):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_\w+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert {"gdn_conv_update", "gdn_recurrent_step", "gdn_chunk_prefill", "gdn_mixed_batch"} <= set(names)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(gdn.EXPORTS) == set(names)


def test_every_header_is_covered_and_exported(lib):
    headers = sorted(f for f in os.listdir(INCLUDE) if f.endswith(".h"))
    assert headers == ["gdn.h", "gdn_testing.h"]
    testing = declared_functions(TESTING_HEADER)
    assert set(testing) == set(gdn.TESTING_EXPORTS)
    assert not [n for n in testing if not hasattr(lib, n)]


def test_testing_hook_sets_and_resets_without_a_gpu(lib):
    # host-only: the hook stores settings that later prefill launches read
    assert lib.gdn_testing_set_prefill_faults(ctypes.c_uint64(10_000_000), 0) == 0
    assert lib.gdn_testing_set_prefill_faults(ctypes.c_uint64(0), -1) == 0


def big_layer(**kw):
    d = dict(num_k_heads=16, num_v_heads=32, head_k_dim=128, head_v_dim=128, conv_width=4, conv_state_len=6,
             act_dtype=gdn.GDN_BF16, scale=0.0, qkv_layout=0, conv_layout=0)
    d.update(kw)
    return _LayerDesc(**d)


def params():
    return _LayerParams(FAKE, None, FAKE, FAKE)


def pools():
    return _Pools(FAKE, FAKE, 512)


def spec_rows(n=64, k=4, **kw):
    d = dict(num_seqs=n, num_tokens=n * k, query_start_loc=FAKE, token_indx=None, state_indices=None,
             has_initial_state=None, spec_state_indices=FAKE, num_accepted_tokens=FAKE, spec_cols=k)
    d.update(kw)
    return _Rows(**d)


def ns_rows(n=8, t=8, **kw):
    d = dict(num_seqs=n, num_tokens=t, query_start_loc=FAKE, token_indx=FAKE, state_indices=FAKE,
             has_initial_state=None, spec_state_indices=None, num_accepted_tokens=None, spec_cols=0)
    d.update(kw)
    return _Rows(**d)


def mixed(lib, layer=None, prm=None, pl=None, non_spec=None, spec=None, n_tokens=None, decodes=8, prefills=0,
          x=FAKE, ws=FAKE, ws_bytes=1 << 40, a=FAKE, out=FAKE):
    layer = layer or big_layer()
    prm = prm or params()
    pl = pl or pools()
    spec = spec if spec is not None else spec_rows(token_indx=FAKE)
    non_spec = non_spec if non_spec is not None else ns_rows()
    if n_tokens is None:
        n_tokens = spec.num_tokens + non_spec.num_tokens
    return lib.gdn_mixed_batch(ctypes.byref(layer), ctypes.byref(prm), ctypes.byref(pl), x, a, FAKE, n_tokens,
                               ctypes.byref(non_spec), decodes, prefills, ctypes.byref(spec), out, ws, ws_bytes,
                               None, None)


ERR = {v: k for k, v in gdn.ERRORS.items()}


def test_status_strings(lib):
    for code in list(gdn.ERRORS) + [0, -99]:
        s = lib.gdn_status_string(code)
        assert isinstance(s, bytes) and s


def test_null_and_dtype_checks(lib):
    assert lib.gdn_mixed_batch(None, None, None, None, None, None, 0, None, 0, 0, None, None, None, 0, None,
                               None) == ERR["NULL_ARG"]
    assert mixed(lib, layer=big_layer(act_dtype=7)) == ERR["DTYPE"]
    assert mixed(lib, prm=_LayerParams(FAKE, None, None, FAKE)) == ERR["NULL_ARG"]
    assert mixed(lib, pl=_Pools(FAKE, None, 512)) == ERR["NULL_ARG"]
    # num_spec > 0 with no query_start_loc (an unchecked optional on the pages)
    assert mixed(lib, spec=spec_rows(query_start_loc=None, token_indx=FAKE)) == ERR["NULL_ARG"]
    # mixed mode needs both token_indx
    assert mixed(lib, spec=spec_rows(token_indx=None)) == ERR["NULL_ARG"]
    # a non-spec subset needs its state indices
    assert mixed(lib, non_spec=ns_rows(state_indices=None)) == ERR["NULL_ARG"]
    assert mixed(lib, x=None) == ERR["NULL_ARG"]


def test_spec_pair_is_required(lib):
    assert mixed(lib, spec=spec_rows(token_indx=FAKE, num_accepted_tokens=None)) == ERR["SPEC_PAIR"]
    assert mixed(lib, spec=spec_rows(token_indx=FAKE, spec_state_indices=None)) == ERR["SPEC_PAIR"]
    # the non-spec slot of a mixed call cannot hold spec rows, nor the spec slot non-spec rows
    assert mixed(lib, non_spec=spec_rows(token_indx=FAKE), decodes=64) == ERR["SPEC_PAIR"]
    assert mixed(lib, spec=ns_rows()) == ERR["SPEC_PAIR"]


@pytest.mark.parametrize("kw", [dict(num_v_heads=24), dict(head_k_dim=48), dict(head_v_dim=72),
                                dict(conv_width=5), dict(conv_state_len=2), dict(num_k_heads=0),
                                dict(qkv_layout=2), dict(conv_layout=3)])
def test_shape_checks(lib, kw):
    assert mixed(lib, layer=big_layer(**kw)) == ERR["SHAPE"]


def test_acceptance_aware_non_spec_rows(lib):
    # a non-spec subset may carry the spec pair (the previous verify step's slots and acceptance)
    aware = ns_rows(spec_state_indices=FAKE, num_accepted_tokens=FAKE, spec_cols=4)
    assert mixed(lib, non_spec=aware, ws_bytes=16) == ERR["WORKSPACE"]
    # ... still as a pair, with a valid column count that fits the rolled ring
    assert mixed(lib, non_spec=ns_rows(spec_state_indices=FAKE, spec_cols=4)) == ERR["SPEC_PAIR"]
    assert mixed(lib, non_spec=ns_rows(spec_state_indices=FAKE, num_accepted_tokens=FAKE, spec_cols=0)) == ERR["SHAPE"]
    assert mixed(lib, non_spec=ns_rows(spec_state_indices=FAKE, num_accepted_tokens=FAKE, spec_cols=5)) == ERR["SHAPE"]
    # the spec slot takes only spec rows, so aware rows there are refused
    assert mixed(lib, spec=spec_rows(state_indices=FAKE, token_indx=FAKE)) == ERR["SPEC_PAIR"]


def test_spec_cols_must_fit_the_conv_ring(lib):
    # state_len 6 with W = 4 holds at most 4 verify tokens per row in the rolled layout
    assert mixed(lib, spec=spec_rows(k=5, token_indx=FAKE)) == ERR["SHAPE"]
    # the per-slot layout keeps W-1 columns per slot, so the same row only reaches the workspace check
    assert mixed(lib, spec=spec_rows(k=5, token_indx=FAKE), layer=big_layer(conv_layout=1),
                 ws_bytes=16) == ERR["WORKSPACE"]
    assert mixed(lib, spec=spec_rows(k=65, token_indx=FAKE), layer=big_layer(conv_state_len=80)) == ERR["SHAPE"]


def test_row_counts(lib):
    assert mixed(lib, decodes=5, prefills=1) == ERR["SHAPE"]       # 6 != 8 non-spec rows
    assert mixed(lib, decodes=-1, prefills=9) == ERR["SHAPE"]
    assert mixed(lib, non_spec=ns_rows(n=0, t=3)) == ERR["SHAPE"]  # tokens without rows


def test_conservation_not_rectangularity(lib):
    base = spec_rows(token_indx=FAKE).num_tokens + ns_rows().num_tokens
    assert mixed(lib, n_tokens=base + 1) == ERR["CONSERVATION"]
    assert mixed(lib, n_tokens=base - 1) == ERR["CONSERVATION"]
    # a ragged spec subset (fewer tokens than rows x spec_cols) is not rejected for its shape:
    # with a workspace that is too small the call gets as far as the workspace check
    ragged = spec_rows(token_indx=FAKE, num_tokens=64 * 4 - 7)
    assert mixed(lib, spec=ragged, ws_bytes=16) == ERR["WORKSPACE"]


def test_workspace_checks(lib):
    layer, s, n = big_layer(), spec_rows(token_indx=FAKE), ns_rows()
    need = lib.gdn_workspace_bytes(ctypes.byref(layer), ctypes.byref(n), ctypes.byref(s))
    C = 2 * 16 * 128 + 32 * 128
    r256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    assert need == r256(s.num_tokens * C * 4) + r256(n.num_tokens * C * 4)
    assert mixed(lib, ws_bytes=need - 1) == ERR["WORKSPACE"]
    assert mixed(lib, ws=None) == ERR["WORKSPACE"]
    # prefill rows add the chunk records (one per 64-token chunk and v-head, bounded from the tokens)
    pre = ns_rows(n=2, t=1536)
    extra = lib.gdn_prefill_workspace_bytes(ctypes.byref(layer), ctypes.byref(pre), 2)
    assert extra == ((1536 + 63) // 64 + 2) * 32 * 123904
    assert lib.gdn_prefill_workspace_bytes(ctypes.byref(layer), ctypes.byref(pre), 0) == 0
    small_layer = big_layer(head_k_dim=64, head_v_dim=64)  # token-recurrence prefill: no records
    assert lib.gdn_prefill_workspace_bytes(ctypes.byref(small_layer), ctypes.byref(pre), 2) == 0
    need_base = lib.gdn_workspace_bytes(ctypes.byref(layer), ctypes.byref(pre), ctypes.byref(s))
    assert mixed(lib, non_spec=pre, decodes=0, prefills=2, ws_bytes=need_base + extra - 256) == ERR["WORKSPACE"]


def test_alignment_checks(lib):
    assert mixed(lib, x=FAKE + 2) == ERR["ALIGN"]
    assert mixed(lib, ws=FAKE + 64) == ERR["ALIGN"]
    assert mixed(lib, pl=_Pools(FAKE + 8, FAKE, 512)) == ERR["ALIGN"]


def test_entry_points_validate_before_launch(lib):
    layer, prm, pl = big_layer(), params(), pools()
    rows = spec_rows(num_accepted_tokens=None)
    assert lib.gdn_conv_update(ctypes.byref(layer), ctypes.byref(prm), ctypes.byref(pl), FAKE, 256,
                               ctypes.byref(rows), FAKE, gdn.GDN_F32, None, None) == ERR["SPEC_PAIR"]
    assert lib.gdn_conv_update(ctypes.byref(layer), ctypes.byref(prm), ctypes.byref(pl), FAKE, 256,
                               ctypes.byref(spec_rows()), FAKE, 9, None, None) == ERR["DTYPE"]
    assert lib.gdn_recurrent_step(ctypes.byref(layer), ctypes.byref(prm), ctypes.byref(pl), FAKE, gdn.GDN_F32,
                                  FAKE, FAKE, 256, ctypes.byref(rows), FAKE, None, None) == ERR["SPEC_PAIR"]
    assert lib.gdn_recurrent_step(ctypes.byref(layer), ctypes.byref(prm), ctypes.byref(pl), FAKE + 4,
                                  gdn.GDN_F32, FAKE, FAKE, 256, ctypes.byref(spec_rows()), FAKE, None,
                                  None) == ERR["ALIGN"]
    # chunked prefill: spec rows are refused, so are other chunk sizes and a missing workspace
    assert lib.gdn_chunk_prefill(ctypes.byref(layer), ctypes.byref(prm), ctypes.byref(pl), FAKE, gdn.GDN_F32,
                                 FAKE, FAKE, 256, ctypes.byref(spec_rows()), 64, FAKE, FAKE, 1 << 40, None,
                                 None) == ERR["SPEC_PAIR"]
    pre = ns_rows(n=1, t=100, token_indx=None)
    assert lib.gdn_chunk_prefill(ctypes.byref(layer), ctypes.byref(prm), ctypes.byref(pl), FAKE, gdn.GDN_F32,
                                 FAKE, FAKE, 100, ctypes.byref(pre), 32, FAKE, FAKE, 1 << 40, None,
                                 None) == ERR["SHAPE"]
    assert lib.gdn_chunk_prefill(ctypes.byref(layer), ctypes.byref(prm), ctypes.byref(pl), FAKE, gdn.GDN_F32,
                                 FAKE, FAKE, 100, ctypes.byref(pre), 64, FAKE, None, 0, None,
                                 None) == ERR["WORKSPACE"]


def test_static_workspace_rejects_large_batches_before_touching_the_gpu(lib):
    layer, prm, pl = big_layer(), params(), pools()
    s = spec_rows(n=512, k=4, token_indx=None)  # 2048 tokens x 32 KiB of scratch > 16 MiB
    rc = lib.gdn_mixed_batch_static_workspace(ctypes.byref(layer), ctypes.byref(prm), ctypes.byref(pl), FAKE,
                                              FAKE, FAKE, s.num_tokens, None, 0, 0, ctypes.byref(s), FAKE, None,
                                              None)
    assert rc == ERR["WORKSPACE"]


def test_output_alignment_on_the_chunked_path(lib):
    # the tensor-core prefill writes 16-byte output vectors: a misaligned out is refused there
    pre = ns_rows(n=8, t=300)
    assert mixed(lib, non_spec=pre, decodes=6, prefills=2, out=FAKE + 2) == ERR["ALIGN"]


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="relies on validation alone to stop a launch with fake pointers")
def test_conv_grid_limit_is_checked_before_launch(lib):
    # non-spec rows are cut into 16-token conv work units (grid.y); ~1.1 M tokens need more than
    # the 65535 units one launch can address, which must be refused before anything is enqueued
    layer, prm, pl = big_layer(), params(), pools()
    big = ns_rows(n=8, t=1_100_000, token_indx=FAKE)
    assert lib.gdn_conv_update(ctypes.byref(layer), ctypes.byref(prm), ctypes.byref(pl), FAKE, 1_100_000,
                               ctypes.byref(big), FAKE, gdn.GDN_F32, None, None) == ERR["SHAPE"]
    assert mixed(lib, non_spec=big, decodes=0, prefills=8) == ERR["SHAPE"]

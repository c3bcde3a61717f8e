"""The C ABI from plain C (CPU only): ``tests/c_client.c`` is compiled with the host C compiler
against ``include/gdn.h``, linked to the in-tree shared library and run.  Its workspace sizes
must match the Python binding's and the closed forms, and every refused call must return the
documented code ("[XE2] Support MTP of QWEN model": every optional tensor checked before use,
the conservation check; "[GDN] Spec-decoding-aware attention kernel": the spec pair)."""
import os
import shutil
import subprocess

import pytest
import torch

import gated_deltanet_linear_spec_gb300 as gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="relies on validation alone to stop launches with fake pointers")


@pytest.fixture(scope="module")
def client_output(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("no host C compiler")
    if not os.path.exists(gdn.LIB_PATH):
        from gated_deltanet_linear_spec_gb300 import build
        build.build()
    libdir = os.path.dirname(gdn.LIB_PATH)
    exe = str(tmp_path_factory.mktemp("c_client") / "c_client")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_client.c"), "-o", exe, gdn.LIB_PATH,
                    f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    return dict(line.split(" ", 1) for line in out.strip().splitlines())


def test_workspace_sizes(client_output):
    C = 2 * 16 * 128 + 32 * 128
    assert int(client_output["ws_spec"]) == 256 * C * 4          # fp32 post-conv q|k|v of 256 tokens
    assert int(client_output["ws_mixed"]) == (256 + 8) * C * 4
    # one 123904-byte record per (64-token chunk, v-head), bounded by ceil(T / 64) + rows chunks
    assert int(client_output["ws_prefill"]) == (8192 // 64 + 1) * 32 * 123904


def test_status_strings_name_every_code(client_output):
    names = {0: "OK", 1: "NULL_ARG", 2: "SPEC_PAIR", 3: "SHAPE", 4: "CONSERVATION", 5: "WORKSPACE",
             6: "DTYPE", 7: "CUDA", 8: "ALIGN"}
    texts = [client_output[f"status{i}"] for i in names]
    assert all(texts) and len(set(texts)) == len(texts)


def test_refused_calls_return_the_documented_codes(client_output):
    err = {v: k for k, v in gdn.ERRORS.items()}
    assert int(client_output["mixed_null"]) == err["NULL_ARG"]
    assert int(client_output["conv_spec_pair"]) == err["SPEC_PAIR"]
    assert int(client_output["conv_dtype"]) == err["DTYPE"]
    assert int(client_output["recurrent_align"]) == err["ALIGN"]
    assert int(client_output["prefill_chunk"]) == err["SHAPE"]
    assert int(client_output["mixed_shape"]) == err["SHAPE"]
    assert int(client_output["mixed_conservation"]) == err["CONSERVATION"]
    assert int(client_output["mixed_workspace"]) == err["WORKSPACE"]

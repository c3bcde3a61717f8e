"""GB300-native Gated DeltaNet speculative-decoding hot path: Python binding of ``libgdn.so``.

The functions here mirror the C entry points in ``include/gdn.h`` one for one
(``gdn_conv_update``, ``gdn_recurrent_step``, ``gdn_chunk_prefill``, ``gdn_mixed_batch``,
``gdn_workspace_bytes``) and only marshal arguments: torch CUDA tensors become device
pointers, the current torch stream becomes the ``cudaStream_t``, and a negative return code
becomes a ``GdnError``.  Every step of the path runs in the library's CUDA kernels; there is
no fallback, and a missing library raises at the first call.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn.so")

GDN_F32, GDN_BF16 = 0, 1
GDN_QKV_PACKED, GDN_QKV_PER_KHEAD = 0, 1
GDN_CONV_ROLLED, GDN_CONV_PER_SLOT = 0, 1
STATUS_SLOT_RANGE, STATUS_NUM_ACCEPTED, STATUS_TOKEN_RANGE, STATUS_ROW_RANGE = 0x1, 0x2, 0x4, 0x8
STATUS_WAIT_TIMEOUT = 0x10
ERRORS = {-1: "NULL_ARG", -2: "SPEC_PAIR", -3: "SHAPE", -4: "CONSERVATION", -5: "WORKSPACE",
          -6: "DTYPE", -7: "CUDA", -8: "ALIGN"}


class GdnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code
        self.name = ERRORS.get(code, str(code))


class _LayerDesc(ctypes.Structure):
    _fields_ = [("num_k_heads", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
                ("head_k_dim", ctypes.c_int32), ("head_v_dim", ctypes.c_int32),
                ("conv_width", ctypes.c_int32), ("conv_state_len", ctypes.c_int32),
                ("act_dtype", ctypes.c_int32), ("scale", ctypes.c_float),
                ("qkv_layout", ctypes.c_int32), ("conv_layout", ctypes.c_int32)]


class _LayerParams(ctypes.Structure):
    _fields_ = [("conv_weight", ctypes.c_void_p), ("conv_bias", ctypes.c_void_p),
                ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p)]


class _Pools(ctypes.Structure):
    _fields_ = [("conv_pool", ctypes.c_void_p), ("ssm_pool", ctypes.c_void_p), ("num_slots", ctypes.c_int64)]


class _Rows(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_tokens", ctypes.c_int32),
                ("query_start_loc", ctypes.c_void_p), ("token_indx", ctypes.c_void_p),
                ("state_indices", ctypes.c_void_p), ("has_initial_state", ctypes.c_void_p),
                ("spec_state_indices", ctypes.c_void_p), ("num_accepted_tokens", ctypes.c_void_p),
                ("spec_cols", ctypes.c_int32)]


EXPORTS = ("gdn_workspace_bytes", "gdn_prefill_workspace_bytes", "gdn_conv_update", "gdn_recurrent_step", "gdn_chunk_prefill",
           "gdn_mixed_batch", "gdn_mixed_batch_static_workspace", "gdn_status_string")
# include/gdn_testing.h: hooks that let tests drive the kernels' failure paths
TESTING_EXPORTS = ("gdn_testing_set_prefill_faults",)
STATIC_WORKSPACE_BYTES = 16 << 20

_lib = None
_lock = threading.Lock()


def library() -> ctypes.CDLL:
    """Loads ``libgdn.so`` (built by ``build.py``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: run gated_deltanet_linear_spec_gb300.build first")
            lib = ctypes.CDLL(LIB_PATH)
            P, I32, VP = ctypes.POINTER, ctypes.c_int32, ctypes.c_void_p
            lib.gdn_status_string.restype = ctypes.c_char_p
            lib.gdn_status_string.argtypes = [ctypes.c_int]
            lib.gdn_workspace_bytes.restype = ctypes.c_size_t
            lib.gdn_workspace_bytes.argtypes = [P(_LayerDesc), P(_Rows), P(_Rows)]
            lib.gdn_prefill_workspace_bytes.restype = ctypes.c_size_t
            lib.gdn_prefill_workspace_bytes.argtypes = [P(_LayerDesc), P(_Rows), I32]
            lib.gdn_conv_update.restype = ctypes.c_int
            lib.gdn_conv_update.argtypes = [P(_LayerDesc), P(_LayerParams), P(_Pools), VP, I32, P(_Rows), VP,
                                            ctypes.c_int, VP, VP]
            lib.gdn_recurrent_step.restype = ctypes.c_int
            lib.gdn_recurrent_step.argtypes = [P(_LayerDesc), P(_LayerParams), P(_Pools), VP, ctypes.c_int, VP,
                                               VP, I32, P(_Rows), VP, VP, VP]
            lib.gdn_chunk_prefill.restype = ctypes.c_int
            lib.gdn_chunk_prefill.argtypes = [P(_LayerDesc), P(_LayerParams), P(_Pools), VP, ctypes.c_int, VP,
                                              VP, I32, P(_Rows), I32, VP, VP, ctypes.c_size_t, VP, VP]
            lib.gdn_mixed_batch.restype = ctypes.c_int
            lib.gdn_mixed_batch.argtypes = [P(_LayerDesc), P(_LayerParams), P(_Pools), VP, VP, VP, I32, P(_Rows),
                                            I32, I32, P(_Rows), VP, VP, ctypes.c_size_t, VP, VP]
            lib.gdn_mixed_batch_static_workspace.restype = ctypes.c_int
            lib.gdn_mixed_batch_static_workspace.argtypes = [P(_LayerDesc), P(_LayerParams), P(_Pools), VP, VP, VP,
                                                             I32, P(_Rows), I32, I32, P(_Rows), VP, VP, VP]
            lib.gdn_testing_set_prefill_faults.restype = ctypes.c_int
            lib.gdn_testing_set_prefill_faults.argtypes = [ctypes.c_uint64, I32]
            _lib = lib
    return _lib


# ------------------------------------------------------------------------------------------
# Descriptors (Python views of the C structs)

def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return GDN_BF16
    if dt == torch.float32:
        return GDN_F32
    raise TypeError(f"unsupported dtype {dt}")


def _ptr(t: Optional[torch.Tensor], dtype: Optional[torch.dtype] = None, name: str = "") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise TypeError(f"{name}: expected a contiguous tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    return t.data_ptr()


@dataclass
class Layer:
    num_k_heads: int
    num_v_heads: int
    head_k_dim: int
    head_v_dim: int
    conv_width: int
    conv_state_len: int
    act_dtype: torch.dtype = torch.bfloat16
    scale: float = 0.0  # <= 0: 1/sqrt(head_k_dim)
    qkv_layout: int = 0   # GDN_QKV_PACKED / GDN_QKV_PER_KHEAD (channel order of x)
    conv_layout: int = 0  # GDN_CONV_ROLLED / GDN_CONV_PER_SLOT (spec conv history)

    @property
    def channels(self) -> int:
        return 2 * self.num_k_heads * self.head_k_dim + self.num_v_heads * self.head_v_dim

    def c(self) -> _LayerDesc:
        return _LayerDesc(self.num_k_heads, self.num_v_heads, self.head_k_dim, self.head_v_dim, self.conv_width,
                          self.conv_state_len, _dtype_code(self.act_dtype), float(self.scale), int(self.qkv_layout),
                          int(self.conv_layout))


@dataclass
class Params:
    conv_weight: torch.Tensor
    A_log: torch.Tensor
    dt_bias: torch.Tensor
    conv_bias: Optional[torch.Tensor] = None

    def c(self, act: torch.dtype) -> _LayerParams:
        return _LayerParams(_ptr(self.conv_weight, act, "conv_weight"), _ptr(self.conv_bias, act, "conv_bias"),
                            _ptr(self.A_log, torch.float32, "A_log"), _ptr(self.dt_bias, torch.float32, "dt_bias"))


@dataclass
class Pools:
    conv_pool: Optional[torch.Tensor]
    ssm_pool: torch.Tensor

    def c(self, act: torch.dtype) -> _Pools:
        return _Pools(_ptr(self.conv_pool, act, "conv_pool"), _ptr(self.ssm_pool, torch.float32, "ssm_pool"),
                      int(self.ssm_pool.shape[0]))


@dataclass
class Rows:
    """One subset of rows (int32 CUDA tensors).  Speculative when spec_state_indices is set."""
    query_start_loc: torch.Tensor
    num_tokens: int
    token_indx: Optional[torch.Tensor] = None
    state_indices: Optional[torch.Tensor] = None
    has_initial_state: Optional[torch.Tensor] = None
    spec_state_indices: Optional[torch.Tensor] = None
    num_accepted_tokens: Optional[torch.Tensor] = None

    @property
    def num_seqs(self) -> int:
        return self.query_start_loc.numel() - 1

    def c(self) -> _Rows:
        i32 = torch.int32
        cols = 0 if self.spec_state_indices is None else int(self.spec_state_indices.shape[-1])
        return _Rows(self.num_seqs, int(self.num_tokens), _ptr(self.query_start_loc, i32, "query_start_loc"),
                     _ptr(self.token_indx, i32, "token_indx"), _ptr(self.state_indices, i32, "state_indices"),
                     _ptr(self.has_initial_state, i32, "has_initial_state"),
                     _ptr(self.spec_state_indices, i32, "spec_state_indices"),
                     _ptr(self.num_accepted_tokens, i32, "num_accepted_tokens"), cols)


def _rows_ref(r: Optional[Rows]):
    return None if r is None else ctypes.byref(r.c())


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(rc: int) -> None:
    if rc != 0:
        raise GdnError(rc, library().gdn_status_string(rc).decode())


# ------------------------------------------------------------------------------------------
# The entry points

def gdn_workspace_bytes(layer: Layer, non_spec: Optional[Rows], spec: Optional[Rows]) -> int:
    return int(library().gdn_workspace_bytes(ctypes.byref(layer.c()), _rows_ref(non_spec), _rows_ref(spec)))


def gdn_prefill_workspace_bytes(layer: Layer, rows: Optional[Rows], num_prefills: int) -> int:
    return int(library().gdn_prefill_workspace_bytes(ctypes.byref(layer.c()), _rows_ref(rows), int(num_prefills)))


def mixed_batch_workspace_bytes(layer: Layer, non_spec: Optional[Rows], num_prefills: int,
                                spec: Optional[Rows]) -> int:
    """Total workspace gdn_mixed_batch needs for this batch."""
    return gdn_workspace_bytes(layer, non_spec, spec) + gdn_prefill_workspace_bytes(layer, non_spec, num_prefills)


def gdn_conv_update(layer: Layer, params: Params, pools: Pools, x: torch.Tensor, rows: Rows, y: torch.Tensor,
                    status: Optional[torch.Tensor] = None, stream=None) -> None:
    act = layer.act_dtype
    rc = library().gdn_conv_update(ctypes.byref(layer.c()), ctypes.byref(params.c(act)), ctypes.byref(pools.c(act)),
                                   _ptr(x, act, "x"), int(x.shape[0]), ctypes.byref(rows.c()), _ptr(y, None, "y"),
                                   _dtype_code(y.dtype), _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc)


def gdn_recurrent_step(layer: Layer, params: Params, pools: Pools, qkv: torch.Tensor, a: torch.Tensor,
                       b: torch.Tensor, rows: Rows, out: torch.Tensor, status: Optional[torch.Tensor] = None,
                       stream=None) -> None:
    act = layer.act_dtype
    rc = library().gdn_recurrent_step(ctypes.byref(layer.c()), ctypes.byref(params.c(act)),
                                      ctypes.byref(pools.c(act)), _ptr(qkv, None, "qkv"), _dtype_code(qkv.dtype), _ptr(a, act, "a"),
                                      _ptr(b, act, "b"), int(a.shape[0]), ctypes.byref(rows.c()),
                                      _ptr(out, act, "out"), _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc)


def gdn_chunk_prefill(layer: Layer, params: Params, pools: Pools, qkv: torch.Tensor, a: torch.Tensor,
                      b: torch.Tensor, rows: Rows, out: torch.Tensor, workspace: Optional[torch.Tensor] = None,
                      chunk_size: int = 64, status: Optional[torch.Tensor] = None, stream=None) -> None:
    act = layer.act_dtype
    need = gdn_prefill_workspace_bytes(layer, rows, rows.num_seqs)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=qkv.device)
    ws_ptr = _ptr(workspace, torch.uint8, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel()
    rc = library().gdn_chunk_prefill(ctypes.byref(layer.c()), ctypes.byref(params.c(act)), ctypes.byref(pools.c(act)),
                                     _ptr(qkv, None, "qkv"), _dtype_code(qkv.dtype), _ptr(a, act, "a"),
                                     _ptr(b, act, "b"), int(a.shape[0]), ctypes.byref(rows.c()), int(chunk_size),
                                     _ptr(out, act, "out"), ws_ptr, ws_bytes, _ptr(status, torch.int32, "status"),
                                     _stream(stream))
    _check(rc)


def gdn_mixed_batch(layer: Layer, params: Params, pools: Pools, x: torch.Tensor, a: torch.Tensor,
                    b: torch.Tensor, non_spec: Optional[Rows], num_decodes: int, num_prefills: int,
                    spec: Optional[Rows], out: torch.Tensor, workspace: Optional[torch.Tensor] = None,
                    status: Optional[torch.Tensor] = None, stream=None,
                    num_actual_tokens: Optional[int] = None) -> None:
    """``num_actual_tokens`` (default x.shape[0]) may be smaller than the row count of x, a, b
    and out, e.g. for inputs padded to a CUDA-graph bucket; rows past it are never touched."""
    act = layer.act_dtype
    if num_actual_tokens is None:
        num_actual_tokens = int(x.shape[0])
    if workspace is None:
        need = mixed_batch_workspace_bytes(layer, non_spec, num_prefills, spec)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    rc = library().gdn_mixed_batch(ctypes.byref(layer.c()), ctypes.byref(params.c(act)), ctypes.byref(pools.c(act)),
                                   _ptr(x, act, "x"), _ptr(a, act, "a"), _ptr(b, act, "b"), int(num_actual_tokens),
                                   _rows_ref(non_spec), int(num_decodes), int(num_prefills), _rows_ref(spec),
                                   _ptr(out, act, "out"), _ptr(workspace, torch.uint8, "workspace"),
                                   workspace.numel(), _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc)


def gdn_mixed_batch_static_workspace(layer: Layer, params: Params, pools: Pools, x: torch.Tensor, a: torch.Tensor,
                                     b: torch.Tensor, non_spec: Optional[Rows], num_decodes: int, num_prefills: int,
                                     spec: Optional[Rows], out: torch.Tensor, status: Optional[torch.Tensor] = None,
                                     stream=None) -> None:
    """gdn_mixed_batch with the library's fixed device scratch, for callers that cannot
    allocate device memory (see include/gdn.h); allocates nothing itself."""
    act = layer.act_dtype
    rc = library().gdn_mixed_batch_static_workspace(
        ctypes.byref(layer.c()), ctypes.byref(params.c(act)), ctypes.byref(pools.c(act)), _ptr(x, act, "x"),
        _ptr(a, act, "a"), _ptr(b, act, "b"), int(x.shape[0]), _rows_ref(non_spec), int(num_decodes),
        int(num_prefills), _rows_ref(spec), _ptr(out, act, "out"), _ptr(status, torch.int32, "status"),
        _stream(stream))
    _check(rc)


def gdn_testing_set_prefill_faults(wait_ns: int = 0, drop_copy_chunk: int = -1) -> None:
    """Test hook (include/gdn_testing.h): the wall-clock limit of the chunked prefill's bounded
    waits (0 = the default, one second) and a chunk whose record copy the scan leaves out on
    purpose (< 0 = none), for every later prefill launch in this process."""
    _check(library().gdn_testing_set_prefill_faults(int(wait_ns), int(drop_copy_chunk)))


__all__ = ["Layer", "Params", "Pools", "Rows", "GdnError", "library", "LIB_PATH", "EXPORTS",
           "gdn_workspace_bytes", "gdn_prefill_workspace_bytes", "mixed_batch_workspace_bytes", "STATUS_WAIT_TIMEOUT", "gdn_conv_update", "gdn_recurrent_step", "gdn_chunk_prefill",
           "gdn_mixed_batch", "gdn_mixed_batch_static_workspace", "STATIC_WORKSPACE_BYTES",
           "TESTING_EXPORTS", "gdn_testing_set_prefill_faults", "GDN_F32", "GDN_BF16", "STATUS_SLOT_RANGE", "STATUS_NUM_ACCEPTED",
           "STATUS_TOKEN_RANGE", "STATUS_ROW_RANGE"]

"""Python face of the CPU oracle in ``gdn_ref.c`` (ctypes over numpy arrays).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, ``__graft_entry__.smoke()``
and the bench's CPU-baseline leg may import this module.  It shares nothing with the CUDA
library: it builds its own shared object from ``gdn_ref.c`` with the host C compiler and
never receives a value that the CUDA library computed.

Everything here is argument marshalling; the arithmetic is in ``gdn_ref.c``.  bf16 arrays
travel as ``uint16`` bit patterns.  The functions mutate the pools they are given, exactly
like the library does on the device.  ``precision="f64"`` (the oracle) works in double;
``precision="f32"`` loads the float build of the same source, used only to measure the
rounding noise of an fp32 implementation of the definition.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_ref.c")
_LIB_PATHS = {"f64": os.path.join(_HERE, "libgdn_ref.so"), "f32": os.path.join(_HERE, "libgdn_ref_f32.so")}
_REAL = {"f64": np.float64, "f32": np.float32}
_libs: dict = {}
_lock = threading.Lock()


def build(force: bool = False, precision: str = "f64") -> str:
    """Compile ``gdn_ref.c`` into ``libgdn_ref.so`` (or, for ``precision="f32"``, the float
    build ``libgdn_ref_f32.so``) beside it (portable C11, no -march)."""
    path = _LIB_PATHS[precision]
    if force or not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
        tmp = path + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
               *(["-DGDN_REF_FLOAT"] if precision == "f32" else []), _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, path)
    return path


def build_all(force: bool = False) -> None:
    """Both builds (the oracle and its float twin)."""
    for precision in _LIB_PATHS:
        build(force, precision)


class _Layer(ctypes.Structure):
    _fields_ = [("num_k_heads", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
                ("head_k_dim", ctypes.c_int32), ("head_v_dim", ctypes.c_int32),
                ("conv_width", ctypes.c_int32), ("conv_state_len", ctypes.c_int32),
                ("act_is_bf16", ctypes.c_int32), ("scale", ctypes.c_double),
                ("norm_eps", ctypes.c_double), ("qkv_layout", ctypes.c_int32), ("conv_layout", ctypes.c_int32)]


class _Rows(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_tokens", ctypes.c_int32),
                ("query_start_loc", ctypes.c_void_p), ("token_indx", ctypes.c_void_p),
                ("state_indices", ctypes.c_void_p), ("has_initial_state", ctypes.c_void_p),
                ("spec_state_indices", ctypes.c_void_p), ("num_accepted_tokens", ctypes.c_void_p),
                ("spec_cols", ctypes.c_int32), ("is_spec", ctypes.c_int32)]


def _load(precision: str = "f64"):
    with _lock:
        if precision not in _libs:
            lib = ctypes.CDLL(build(precision=precision))
            lib.gdn_ref_conv.restype = ctypes.c_int
            lib.gdn_ref_conv.argtypes = [ctypes.POINTER(_Layer), ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                         ctypes.c_int32, ctypes.POINTER(_Rows), ctypes.c_void_p]
            lib.gdn_ref_recurrent.restype = ctypes.c_int
            lib.gdn_ref_recurrent.argtypes = [ctypes.POINTER(_Layer), ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                              ctypes.POINTER(_Rows), ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
            _libs[precision] = lib
    return _libs[precision]


@dataclass
class Layer:
    num_k_heads: int
    num_v_heads: int
    head_k_dim: int
    head_v_dim: int
    conv_width: int = 4
    conv_state_len: int = 3
    act_bf16: bool = True
    scale: Optional[float] = None  # None -> 1/sqrt(head_k_dim)
    norm_eps: float = 1e-6
    qkv_layout: int = 0   # 0 packed q|k|v; 1 per k-head groups (x only)
    conv_layout: int = 0  # 0 rolled history at column 0; 1 one snapshot per spec slot

    @property
    def channels(self) -> int:
        return 2 * self.num_k_heads * self.head_k_dim + self.num_v_heads * self.head_v_dim

    def _c(self) -> _Layer:
        scale = self.scale if self.scale is not None else 1.0 / np.sqrt(self.head_k_dim)
        return _Layer(self.num_k_heads, self.num_v_heads, self.head_k_dim, self.head_v_dim,
                      self.conv_width, self.conv_state_len, int(self.act_bf16), float(scale),
                      float(self.norm_eps), int(self.qkv_layout), int(self.conv_layout))


@dataclass
class Rows:
    """One subset of rows.  Integer arrays are int32; None where the subset has no such tensor."""
    query_start_loc: np.ndarray
    is_spec: bool
    token_indx: Optional[np.ndarray] = None
    state_indices: Optional[np.ndarray] = None
    has_initial_state: Optional[np.ndarray] = None
    spec_state_indices: Optional[np.ndarray] = None
    num_accepted_tokens: Optional[np.ndarray] = None

    @property
    def num_seqs(self) -> int:
        return int(len(self.query_start_loc) - 1)

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1]) if len(self.query_start_loc) else 0

    def _c(self, keep: list) -> _Rows:
        def ptr(a):
            if a is None:
                return None
            a = np.ascontiguousarray(a, dtype=np.int32)
            keep.append(a)
            return a.ctypes.data
        cols = 0 if self.spec_state_indices is None else int(np.asarray(self.spec_state_indices).shape[-1])
        return _Rows(self.num_seqs, self.num_tokens, ptr(self.query_start_loc), ptr(self.token_indx),
                     ptr(self.state_indices), ptr(self.has_initial_state),
                     ptr(self.spec_state_indices), ptr(self.num_accepted_tokens), cols,
                     int(self.is_spec))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _need(a: np.ndarray, dtype, name: str) -> np.ndarray:
    if a.dtype != dtype or not a.flags.c_contiguous:
        raise TypeError(f"{name}: expected a C-contiguous {np.dtype(dtype).name} array")
    return a


def conv_update(layer: Layer, conv_w: np.ndarray, conv_b: Optional[np.ndarray], conv_pool: np.ndarray,
                x: np.ndarray, num_global: int, rows: Rows, precision: str = "f64") -> np.ndarray:
    """Conv update of one subset; mutates ``conv_pool``; returns y [T_sub, C] (float64, or
    float32 for the float build; local order)."""
    act = np.uint16 if layer.act_bf16 else np.float32
    _need(conv_w, act, "conv_w"); _need(conv_pool, act, "conv_pool"); _need(x, act, "x")
    if conv_b is not None:
        _need(conv_b, act, "conv_b")
    y = np.zeros((rows.num_tokens, layer.channels), dtype=_REAL[precision])
    keep: list = []
    L, R = layer._c(), rows._c(keep)
    rc = _load(precision).gdn_ref_conv(ctypes.byref(L), _ptr(conv_w), _ptr(conv_b), _ptr(conv_pool),
                              int(conv_pool.shape[0]), _ptr(x), int(num_global), ctypes.byref(R), _ptr(y))
    if rc:
        raise ValueError(f"oracle conv rejected its inputs (rc={rc})")
    return y


def recurrent(layer: Layer, A_log: np.ndarray, dt_bias: np.ndarray, ssm_pool: np.ndarray,
              qkv: np.ndarray, a: np.ndarray, b: np.ndarray, num_global: int, rows: Rows,
              out: np.ndarray, out_f64: Optional[np.ndarray] = None, heads: Optional[tuple] = None,
              nthreads: int = 1, precision: str = "f64") -> None:
    """Gated delta rule over one subset; mutates ``ssm_pool`` and ``out`` (and ``out_f64``,
    which like ``qkv`` is float64, or float32 for the float build)."""
    act = np.uint16 if layer.act_bf16 else np.float32
    _need(A_log, np.float32, "A_log"); _need(dt_bias, np.float32, "dt_bias")
    _need(ssm_pool, np.float32, "ssm_pool"); _need(qkv, _REAL[precision], "qkv")
    _need(a, act, "a"); _need(b, act, "b"); _need(out, act, "out")
    if out_f64 is not None:
        _need(out_f64, _REAL[precision], "out_f64")
    h0, h1 = heads if heads is not None else (0, 0)
    keep: list = []
    L, R = layer._c(), rows._c(keep)
    rc = _load(precision).gdn_ref_recurrent(ctypes.byref(L), _ptr(A_log), _ptr(dt_bias), _ptr(ssm_pool),
                                   int(ssm_pool.shape[0]), _ptr(qkv), _ptr(a), _ptr(b), int(num_global),
                                   ctypes.byref(R), _ptr(out), _ptr(out_f64), int(h0), int(h1),
                                   int(nthreads))
    if rc:
        raise ValueError(f"oracle recurrence rejected its inputs (rc={rc})")


def mixed_batch(layer: Layer, conv_w, conv_b, A_log, dt_bias, conv_pool, ssm_pool, x, a, b,
                num_global: int, subsets: list, out: np.ndarray, out_f64: Optional[np.ndarray] = None,
                heads: Optional[tuple] = None, nthreads: int = 1, precision: str = "f64") -> None:
    """The whole path over a batch split into subsets (each a ``Rows``): conv, then recurrence.

    Each subset gathers x, a and b through its own token_indx and scatters its outputs back
    through it; rows of different subsets must use different slots.
    """
    for rows in subsets:
        if rows.num_seqs == 0:
            continue
        y = conv_update(layer, conv_w, conv_b, conv_pool, x, num_global, rows, precision)
        recurrent(layer, A_log, dt_bias, ssm_pool, y, a, b, num_global, rows, out, out_f64, heads, nthreads,
                  precision)

"""fp64 CPU oracle of the GPT-OSS decode sampling tail.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library and never imports it.

The arithmetic lives in ``tail_oracle.c`` (plain C, double precision, one
function per step of the tail as defined on the "GPT-OSS Tail Chunked
Megakernel Kernel API Reference" page).  This module only compiles that file
with gcc and marshals numpy arrays into it.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
against closed forms, exhaustive decodes, brute force and hand-worked cases.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tail_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}


def build(force: bool = False) -> str:
    """Compile ``tail_oracle.c`` into ``liboracle.so`` next to it (gcc -O2)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
                           "-lpthread", "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def use_library(path: str | None) -> None:
    """Point the wrappers at another build of ``tail_oracle.c`` (None: the default one).

    Used by the planted-mistake tests, which compile mutated copies of the
    source in a temporary directory and check that the pins reject them."""
    global _lib, _override
    with _lock:
        _override = path
        _lib = None


_override = None


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = _override or build()
            L = ctypes.CDLL(path)
            P = ctypes.c_void_p
            i32, i64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_float
            L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_double.restype = ctypes.c_double
            L.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_f16_to_double.restype = ctypes.c_double
            L.oracle_widen.argtypes = [P, i32, i64, P]
            L.oracle_widen.restype = None
            L.oracle_rstd.argtypes = [P, i32, i32, i32, i32, f32, i32, P]
            L.oracle_logits.argtypes = [P, i32, P, P, i32, i32, i32, i32, f32, i32, i32, P]
            L.oracle_topk.argtypes = [P, i32, i32, i32, i32, P, P]
            L.oracle_sample_row.argtypes = [P, P, i32, P, i32, P, P, P, P, P]
            L.oracle_tail.argtypes = [P, i32, P, P, i32, i32, i32, i32, i32, f32, i32, P, i32,
                                      i32, P, P, P, P]
            L.oracle_f32_to_bf16_rne.argtypes = [f32]
            L.oracle_f32_to_bf16_rne.restype = ctypes.c_uint16
            L.oracle_moe_combine.argtypes = [P, P, i32, i32, i32, P, i32, i32, P]
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _hidden_bits(hidden: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(hidden, dtype=np.float32)
    return np.ascontiguousarray(hidden.view(np.uint16) if hidden.dtype != np.uint16 else hidden)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def widen(bits: np.ndarray, dtype: str) -> np.ndarray:
    src = _hidden_bits(bits, dtype)
    out = np.empty(src.size, dtype=np.float64)
    lib().oracle_widen(_ptr(src), DTYPE_CODES[dtype], src.size, _ptr(out))
    return out.reshape(src.shape)


def rstd(hidden, dtype, H, Hu, eps, zero_pad) -> np.ndarray:
    x = _hidden_bits(hidden, dtype)
    B = x.size // H
    out = np.empty(B, dtype=np.float64)
    rc = lib().oracle_rstd(_ptr(x), DTYPE_CODES[dtype], B, H, Hu, eps, int(zero_pad), _ptr(out))
    if rc:
        raise ValueError(f"oracle_rstd failed: {rc}")
    return out


def logits(hidden, dtype, gamma, w_t, Hu, eps, zero_pad, nthreads=None) -> np.ndarray:
    x = _hidden_bits(hidden, dtype)
    H, V = w_t.shape
    B = x.size // H
    g = np.ascontiguousarray(gamma, dtype=np.float32).reshape(-1)
    w = np.ascontiguousarray(w_t, dtype=np.uint16)
    out = np.empty((B, V), dtype=np.float64)
    rc = lib().oracle_logits(_ptr(x), DTYPE_CODES[dtype], _ptr(g), _ptr(w), B, H, Hu, V, eps,
                             int(zero_pad), nthreads or default_threads(), _ptr(out))
    if rc:
        raise ValueError(f"oracle_logits failed: {rc}")
    return out


def topk(logit_rows: np.ndarray, k: int, nthreads=None):
    L = np.ascontiguousarray(logit_rows, dtype=np.float64)
    B, V = L.shape
    vals = np.empty((B, k), dtype=np.float64)
    idx = np.empty((B, k), dtype=np.int32)
    rc = lib().oracle_topk(_ptr(L), B, V, k, nthreads or default_threads(), _ptr(vals), _ptr(idx))
    if rc:
        raise ValueError(f"oracle_topk failed: {rc}")
    return vals, idx


class SampleReport:
    """One row's draw with the data needed to judge boundary cases."""

    def __init__(self, token, kk, m, cdf, pcum):
        self.token = token   # sampled vocabulary index
        self.kk = kk         # candidates after the top_k cut
        self.m = m           # candidates after the top_p cut
        self.cdf = cdf       # C_j / C_{m-1} for j < m
        self.pcum = pcum     # sum_{i<=j} p_i for j < kk

    def __repr__(self):
        return f"SampleReport(token={self.token}, kk={self.kk}, m={self.m})"


def sample_row(vals: np.ndarray, idx: np.ndarray, p: np.ndarray) -> SampleReport:
    v = np.ascontiguousarray(vals, dtype=np.float64).reshape(-1)
    i = np.ascontiguousarray(idx, dtype=np.int32).reshape(-1)
    pp = np.ascontiguousarray(p, dtype=np.float32).reshape(-1)
    n = v.size
    tok = np.zeros(1, np.int32)
    kk = np.zeros(1, np.int32)
    m = np.zeros(1, np.int32)
    cdf = np.zeros(n, np.float64)
    pcum = np.zeros(n, np.float64)
    rc = lib().oracle_sample_row(_ptr(v), _ptr(i), n, _ptr(pp), pp.size, _ptr(tok), _ptr(kk),
                                 _ptr(m), _ptr(cdf), _ptr(pcum))
    if rc:
        raise ValueError(f"oracle_sample_row failed: {rc}")
    return SampleReport(int(tok[0]), int(kk[0]), int(m[0]), cdf[: int(m[0])], pcum[: int(kk[0])])


def tail(hidden, dtype, gamma, w_t, Hu, k, eps, zero_pad, params=None, nthreads=None):
    """Whole tail: returns (logits fp64 [B,V], topk vals [B,k], topk idx [B,k], tokens [B] or None)."""
    x = _hidden_bits(hidden, dtype)
    H, V = w_t.shape
    B = x.size // H
    g = np.ascontiguousarray(gamma, dtype=np.float32).reshape(-1)
    w = np.ascontiguousarray(w_t, dtype=np.uint16)
    L = np.empty((B, V), np.float64)
    tv = np.empty((B, k), np.float64)
    ti = np.empty((B, k), np.int32)
    toks = np.zeros(B, np.int32)
    if params is not None:
        P = np.ascontiguousarray(params, dtype=np.float32)
        ncols = P.shape[1]
        pptr = _ptr(P)
    else:
        ncols, pptr = 4, None
    rc = lib().oracle_tail(_ptr(x), DTYPE_CODES[dtype], _ptr(g), _ptr(w), B, H, Hu, V, k, eps,
                           int(zero_pad), pptr, ncols, nthreads or default_threads(), _ptr(L),
                           _ptr(tv), _ptr(ti), _ptr(toks))
    if rc:
        raise ValueError(f"oracle_tail failed: {rc}")
    return L, tv, ti, (toks if params is not None else None)


def f32_to_bf16(v: float) -> int:
    """bf16 bits of an fp32 value, rounded to nearest, ties to even."""
    return int(lib().oracle_f32_to_bf16_rne(ctypes.c_float(v)))


def moe_combine(x_bits: np.ndarray, slots: np.ndarray, w: np.ndarray, n_routed: int | None = None) -> np.ndarray:
    """The tail's producer step: per lane, r = the fp32 fma chain of w[s] * slots[s] over the routed
    slots s < n_routed (in order from 0), sh = the same chain over the shared slots s >= n_routed,
    and h = bf16(x + bf16(r + sh)).

    x_bits [B, H] bf16 bits; slots [B, S, H] float32, or uint16 bf16 bits; w [B, S] float32;
    n_routed: routed slots (None: all S, no shared slot).  Returns h [B, H] as bf16 bits."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    B, H = x.shape
    y = np.ascontiguousarray(slots)
    S = y.shape[1] if y.ndim == 3 else 0
    nr = S if n_routed is None else int(n_routed)
    sd = DTYPE_CODES["f32"] if y.dtype == np.float32 else DTYPE_CODES["bf16"]
    wt = np.ascontiguousarray(w, dtype=np.float32).reshape(B, S)
    h = np.empty((B, H), np.uint16)
    rc = lib().oracle_moe_combine(_ptr(x), _ptr(y) if S else None, sd, S, nr, _ptr(wt) if S else None, B, H,
                                  _ptr(h))
    if rc:
        raise ValueError(f"oracle_moe_combine failed: {rc}")
    return h

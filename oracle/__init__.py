"""fp64 CPU oracle for the PASA attention forward pass.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package. The product path (the CUDA library and its
Python binding) never touches it, and it shares no code with them.

* :func:`attention` / :func:`attention_recovered` / :func:`row_max_abs_score` /
  :func:`row_max_abs_recovered` / :func:`block_max_abs_score` wrap the plain C
  implementation in ``attention_ref.c`` (compiled with gcc by :func:`build`).
* ``pseudo_average`` holds the numpy reference for the key-block pseudo-average and the
  shifted keys.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import pseudo_average  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_ref.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attention_ref.c into oracle/_build/liboracle.so (gcc, OpenMP, -O2, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_attention.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, i64,
                                             ctypes.c_int, ctypes.c_double, p, i64]
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_attention_recovered.argtypes = [p, p, p, i64, p, p, p, i64, i64, i64, i64,
                                                       i64, i64, ctypes.c_int, ctypes.c_double, p, i64]
            lib.oracle_attention_recovered.restype = ctypes.c_int
            lib.oracle_row_max_abs_score.argtypes = [p, p, p, i64, i64, i64, i64, i64, i64,
                                                     ctypes.c_int, p, i64]
            lib.oracle_row_max_abs_score.restype = ctypes.c_int
            lib.oracle_row_max_abs_recovered.argtypes = [p, p, p, i64, p, i64, i64, i64, i64, i64, i64,
                                                         ctypes.c_int, p, i64]
            lib.oracle_row_max_abs_recovered.restype = ctypes.c_int
            lib.oracle_block_max_abs_score.argtypes = [p, p, p, i64, p, i64, i64, i64, i64, i64, i64, ctypes.c_int]
            lib.oracle_block_max_abs_score.restype = ctypes.c_int
            lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_half_to_double.restype = ctypes.c_double
            _lib = lib
    return _lib


def _bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.float16:
        raise TypeError("oracle inputs are fp16 arrays")
    return x.view(np.uint16)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def attention(q, k, v, causal: bool, scale: float | None = None, rows=None):
    """Plain fp64 attention of fp16 inputs q [B,Hq,Sq,D], k/v [B,Hkv,Sk,D].

    Returns (o, lse) in float64: o [B,Hq,Sq,D] and lse [B,Hq,Sq] when ``rows`` is None,
    else o [len(rows), D] and lse [len(rows)] for the flat row indices in ``rows``.
    """
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = B * Hq * Sq if r is None else len(r)
    o = np.empty((n, D), np.float64)
    lse = np.empty((n,), np.float64)
    rc = _load().oracle_attention(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq,
                                  Sk, D, int(bool(causal)), scale, _ptr(r), n)
    if rc != 0:
        raise ValueError("oracle_attention: bad shape")
    if r is None:
        return o.reshape(B, Hq, Sq, D), lse.reshape(B, Hq, Sq)
    return o, lse


def attention_recovered(q, kshift, means, block_rows: int, v, causal: bool,
                        scale: float | None = None, rows=None):
    """fp64 attention from shifted keys plus per-block offsets q . m_j (global recovering)."""
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = kshift.shape
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    qb, kb, mb, vb = _bits(q), _bits(kshift), _bits(means), _bits(v)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = B * Hq * Sq if r is None else len(r)
    o = np.empty((n, D), np.float64)
    lse = np.empty((n,), np.float64)
    rc = _load().oracle_attention_recovered(_ptr(qb), _ptr(kb), _ptr(mb), block_rows, _ptr(vb),
                                            _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Sk, D,
                                            int(bool(causal)), scale, _ptr(r), n)
    if rc != 0:
        raise ValueError("oracle_attention_recovered: bad shape")
    if r is None:
        return o.reshape(B, Hq, Sq, D), lse.reshape(B, Hq, Sq)
    return o, lse


def row_max_abs_score(q, k, causal: bool, rows=None) -> np.ndarray:
    """max_j |q_i . k_j| (unscaled) over the visible keys of each row, in fp64."""
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    qb, kb = _bits(q), _bits(k)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = B * Hq * Sq if r is None else len(r)
    out = np.empty((n,), np.float64)
    rc = _load().oracle_row_max_abs_score(_ptr(qb), _ptr(kb), _ptr(out), B, Hq, Hkv, Sq, Sk, D,
                                          int(bool(causal)), _ptr(r), n)
    if rc != 0:
        raise ValueError("oracle_row_max_abs_score: bad shape")
    return out if r is not None else out.reshape(B, Hq, Sq)


def row_max_abs_recovered(q, kshift, means, block_rows: int, causal: bool, rows=None) -> np.ndarray:
    """max_j |q_i . (k'_j + m_(j / block_rows))| (unscaled) over the visible keys of each row, in fp64."""
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = kshift.shape
    qb, kb, mb = _bits(q), _bits(kshift), _bits(means)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = B * Hq * Sq if r is None else len(r)
    out = np.empty((n,), np.float64)
    rc = _load().oracle_row_max_abs_recovered(_ptr(qb), _ptr(kb), _ptr(mb), block_rows, _ptr(out), B, Hq, Hkv,
                                              Sq, Sk, D, int(bool(causal)), _ptr(r), n)
    if rc != 0:
        raise ValueError("oracle_row_max_abs_recovered: bad shape")
    return out if r is not None else out.reshape(B, Hq, Sq)


def block_max_abs_score(q, k, block_rows: int, causal: bool, means=None) -> np.ndarray:
    """Per key block, max |q_i . k_j| (or |q_i . (k_j + m_block)| with means) over the rows
    that see the block's keys, in fp64: [B, Hq, ceil(Sk / block_rows)]."""
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    nb = -(-Sk // block_rows)
    qb, kb = _bits(q), _bits(k)
    mb = None if means is None else _bits(means)
    out = np.empty((B, Hq, nb), np.float64)
    rc = _load().oracle_block_max_abs_score(_ptr(qb), _ptr(kb), _ptr(mb), block_rows, _ptr(out), B, Hq, Hkv, Sq,
                                            Sk, D, int(bool(causal)))
    if rc != 0:
        raise ValueError("oracle_block_max_abs_score: bad shape")
    return out


def half_to_double(bits: int) -> float:
    """The oracle's own binary16 decoder (exposed so tests can pin it)."""
    return _load().oracle_half_to_double(bits)

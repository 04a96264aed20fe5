"""Plain FP64 CPU oracle for the fixed-order row softmax -- TEST INFRASTRUCTURE ONLY.

The product library (``deterministic_attention_softmax_gb300``) never imports this package.
Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference legs
use it.  It wraps ``fos_oracle.c`` (plain C, double precision, one row at a time) with ctypes
and numpy; see that file's header for the definitions it follows and where the pages state
them:

* forward  -- "[WS1][kernels] Add fixed-order joint-attention softmax for Qwen-Image",
  Summary (softmax along the key dimension); LSE and masked rows from "Batch-invariant
  attention (standard softmax--cuda version)", Implementation / Path Status; the sink from
  "[ROCm] Jax Add softmax sink (learnable off-by-one) support", Description.
* backward -- the first page's "Fixed-order backward" (the softmax VJP).
* d_sink   -- the derivative of the rows' losses with respect to the per-head sink logit.

``oracle/gemm.py`` holds the FP64 oracle of the two contractions around the softmax (QK and
PV, with their backward products), pinned by ``tests/test_oracle_gemm.py``.

All inputs are numpy arrays holding the exact stored values (bf16/fp32 widened to float64).
Parity for every function here is pinned by ``tests/test_oracle.py`` and
``tests/test_golden.py`` (closed forms, invariants, finite differences, brute force).
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fos_oracle.c")
_LIB = os.path.join(_HERE, "libfos_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile ``fos_oracle.c`` into ``libfos_oracle.so`` with gcc (OpenMP when available).

    ``-ffp-contract=off`` keeps the arithmetic the same on x86-64 and aarch64 hosts.
    """
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
    tmp = _LIB + f".tmp{os.getpid()}"
    try:
        subprocess.run(base + ["-fopenmp", "-o", tmp, _SRC, "-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-o", tmp, _SRC, "-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    lib.fos_oracle_fwd.argtypes = [i64, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, i32]
    lib.fos_oracle_fwd.restype = ctypes.c_int
    lib.fos_oracle_bwd.argtypes = [i64, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, i32]
    lib.fos_oracle_bwd.restype = ctypes.c_int
    lib.fos_oracle_sink_grad.argtypes = [i32, i32, i32, vp, vp, vp, vp]
    lib.fos_oracle_sink_grad.restype = ctypes.c_int
    lib.fos_oracle_max_threads.argtypes = []
    lib.fos_oracle_max_threads.restype = ctypes.c_int
    _lib = lib
    return lib


def max_threads() -> int:
    """Threads the oracle's parallel row loop uses by default."""
    return int(_load().fos_oracle_max_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _masks(kv_valid_len, key_mask, sink):
    kv = None if kv_valid_len is None else np.ascontiguousarray(kv_valid_len, dtype=np.int32)
    km = None if key_mask is None else np.ascontiguousarray(key_mask, dtype=np.uint8)
    sk = None if sink is None else _f64(sink)
    return kv, km, sk


def _row_ids(row_ids, n):
    if row_ids is None:
        return None
    ids = np.ascontiguousarray(row_ids, dtype=np.int64)
    if ids.shape != (n,):
        raise ValueError("row_ids must have one entry per given row")
    return ids


def softmax_fwd(scores, *, batch, heads, q_len, causal=False, kv_valid_len=None,
                key_mask=None, sink=None, row_ids=None, nthreads=0):
    """P and LSE of the given rows (``scores`` is n x L).  Returns (P [n, L], lse [n])."""
    x = _f64(scores)
    n, L = x.shape
    kv, km, sk = _masks(kv_valid_len, key_mask, sink)
    ids = _row_ids(row_ids, n)
    if ids is None and n != batch * heads * q_len:
        raise ValueError("without row_ids the rows must be batch*heads*q_len")
    p = np.empty_like(x)
    lse = np.empty(n, dtype=np.float64)
    rc = _load().fos_oracle_fwd(n, _ptr(ids), L, batch, heads, q_len, int(causal), _ptr(kv),
                                _ptr(km), _ptr(sk), _ptr(x), _ptr(p), _ptr(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle forward rejected its arguments")
    return p, lse


def softmax_bwd(probs, dprobs, *, batch, heads, q_len, causal=False, kv_valid_len=None,
                key_mask=None, row_ids=None, nthreads=0):
    """dScores and delta for the given P and dP (n x L each).  Returns (dS [n, L], delta [n])."""
    p = _f64(probs)
    dp = _f64(dprobs)
    if p.shape != dp.shape:
        raise ValueError("P and dP differ in shape")
    n, L = p.shape
    kv, km, _ = _masks(kv_valid_len, key_mask, None)
    ids = _row_ids(row_ids, n)
    if ids is None and n != batch * heads * q_len:
        raise ValueError("without row_ids the rows must be batch*heads*q_len")
    ds = np.empty_like(p)
    delta = np.empty(n, dtype=np.float64)
    rc = _load().fos_oracle_bwd(n, _ptr(ids), L, batch, heads, q_len, int(causal), _ptr(kv),
                                _ptr(km), _ptr(p), _ptr(dp), _ptr(ds), _ptr(delta),
                                int(nthreads))
    if rc != 0:
        raise ValueError("oracle backward rejected its arguments")
    return ds, delta


def sink_grad(lse, delta, sink, *, batch, heads, q_len):
    """d_sink [heads] from the LSE and delta of all batch*heads*q_len rows."""
    lse = _f64(lse)
    delta = _f64(delta)
    sk = _f64(sink)
    if lse.shape != (batch * heads * q_len,) or delta.shape != lse.shape or sk.shape != (heads,):
        raise ValueError("sink_grad wants lse/delta of all rows and one sink per head")
    out = np.empty(heads, dtype=np.float64)
    rc = _load().fos_oracle_sink_grad(batch, heads, q_len, _ptr(sk), _ptr(lse), _ptr(delta),
                                      _ptr(out))
    if rc != 0:
        raise ValueError("oracle sink_grad rejected its arguments")
    return out

"""Helpers shared by the GPU tests: dtype names, exact host copies, oracle calls."""

import numpy as np
import torch

import oracle
from oracle import tolerance as tol

DTYPES = {"float32": torch.float32, "bfloat16": torch.bfloat16, "float16": torch.float16}


def np64(t):
    """Exact float64 host copy (bf16/fp16/fp32 widen exactly)."""
    return t.detach().to(torch.float64).cpu().numpy()


def dev():
    return torch.device("cuda", 0)


def masks_np(kv=None, km=None, sink=None):
    return (None if kv is None else kv.cpu().numpy(),
            None if km is None else km.to(torch.uint8).cpu().numpy(),
            None if sink is None else np64(sink))


def assert_check(result, what):
    ok, worst, idx = result
    assert ok, f"{what}: tolerance exceeded (worst err/bound = {worst:.3g} at flat index {idx})"


def check_fwd(p, lse, p_ref, lse_ref, dtype_name, what=""):
    assert_check(tol.check_probs(np64(p), p_ref, dtype_name), f"P {what}")
    assert_check(tol.check_lse(np64(lse), lse_ref), f"LSE {what}")


def check_bwd(ds, delta, ds_ref, delta_ref, p_in, dp, dtype_name, valid=None, what=""):
    assert_check(tol.check_dscores(np64(ds), ds_ref, p_in, dp, dtype_name, valid), f"dS {what}")
    if delta is not None:
        assert_check(tol.check_delta(np64(delta), delta_ref, p_in, dp, valid), f"delta {what}")


_INT = {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64}


def bits_equal(a, b):
    """Bitwise equality (tells +0 from -0 and compares NaN payloads)."""
    if a.shape != b.shape or a.dtype != b.dtype:
        return False
    it = _INT[a.element_size()]
    return bool(torch.equal(a.contiguous().view(it), b.contiguous().view(it)))


def valid_matrix(rows_ids, L, batch, heads, q_len, causal, kv, km):
    """Boolean [n, L] of the mask definition (without the -inf rule), for tolerance scales."""
    rows_ids = np.asarray(rows_ids)
    b = rows_ids // (heads * q_len)
    i = rows_ids % q_len
    j = np.arange(L)[None, :]
    v = np.ones((len(rows_ids), L), dtype=bool)
    if causal:
        v &= j <= (L - q_len + i)[:, None]
    if kv is not None:
        v &= j < np.asarray(kv)[b][:, None]
    if km is not None:
        v &= np.asarray(km).reshape(-1, L)[b] != 0
    return v


__all__ = ["DTYPES", "bits_equal", "np64", "dev", "masks_np", "assert_check", "check_fwd", "check_bwd",
           "valid_matrix", "oracle", "tol"]

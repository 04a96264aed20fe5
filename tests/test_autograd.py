"""The differentiable op: ``fixed_order_softmax`` routes its forward and backward through the
library's kernels.  It gives the bits of direct calls of fos_softmax_fwd / fos_softmax_bwd /
fos_sink_grad, its sink gradient matches the FP64 oracle, and it refuses CPU tensors (the CPU
check runs without a GPU)."""

import pytest
import torch

import deterministic_attention_softmax_gb300 as fos
from gpu_util import assert_check, bits_equal, masks_np, np64, oracle, tol
from test_parity_small import make_case


def test_refuses_cpu_tensors():
    x = torch.zeros(4, 8, requires_grad=True)
    with pytest.raises(ValueError):
        fos.fixed_order_softmax(x)


def geo(c):
    return dict(batch=c["B"], heads=c["H"], q_len=c["Sq"], causal=c["causal"],
                kv_valid_len=c["kv"], key_mask=c["km"])


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.float16])
@pytest.mark.parametrize("mask", ["none", "all"])
def test_gradients_are_the_direct_calls_bits(dtype, mask):
    c = make_case(dtype, 1000, mask if mask != "none" else "sink", B=2, H=3, Sq=9, seed=5)
    x = c["x"].clone().requires_grad_(True)
    sink = c["sink"].clone().requires_grad_(True)
    p, lse = fos.fixed_order_softmax(x, sink=sink, **geo(c))
    assert not lse.requires_grad
    p.backward(c["dp"])
    p_ref, lse_ref = fos.fos_softmax_fwd(c["x"], sink=c["sink"], **geo(c))
    ds_ref, delta_ref = fos.fos_softmax_bwd(p_ref, c["dp"], **geo(c))
    ds_sink = fos.fos_sink_grad(lse_ref, delta_ref, c["sink"], batch=c["B"], heads=c["H"],
                                q_len=c["Sq"])
    torch.cuda.synchronize()
    assert bits_equal(p.detach(), p_ref) and bits_equal(lse, lse_ref)
    assert bits_equal(x.grad, ds_ref)
    assert bits_equal(sink.grad, ds_sink)


@pytest.mark.gpu
def test_sink_gradient_matches_the_oracle_through_autograd():
    # The FP64 oracle's d_sink from its own LSE and delta (on the GPU's P, which the backward
    # contract takes as given); bound: 1e-5 of the sum of |exp(sink - LSE) * delta| per head.
    c = make_case(torch.float32, 700, "all", B=3, H=4, Sq=11, seed=9)
    x = c["x"].clone().requires_grad_(True)
    sink = c["sink"].clone().requires_grad_(True)
    p, _ = fos.fixed_order_softmax(x, sink=sink, **geo(c))
    (p * c["dp"]).sum().backward()  # dP = c["dp"]
    kv, km, sk = masks_np(c["kv"], c["km"], c["sink"])
    kw = dict(batch=c["B"], heads=c["H"], q_len=c["Sq"], causal=c["causal"], kv_valid_len=kv,
              key_mask=km)
    _, lse64 = oracle.softmax_fwd(np64(c["x"]), sink=sk, **kw)
    _, delta64 = oracle.softmax_bwd(np64(p.detach()), np64(c["dp"]), **kw)
    dsink64 = oracle.sink_grad(lse64, delta64, sk, batch=c["B"], heads=c["H"], q_len=c["Sq"])
    assert_check(tol.check_dsink(np64(sink.grad), dsink64, lse64, delta64, sk, c["B"], c["H"],
                                 c["Sq"]), "d_sink through autograd")


@pytest.mark.gpu
def test_only_what_is_asked_for():
    c = make_case(torch.bfloat16, 512, "sink", B=1, H=2, Sq=4, seed=2)
    sink = c["sink"].clone().requires_grad_(True)
    p, _ = fos.fixed_order_softmax(c["x"], sink=sink, batch=1, heads=2, q_len=4)
    p.backward(c["dp"])  # scores need no gradient: only the sink's is formed
    assert sink.grad is not None and sink.grad.shape == (2,)
    x = c["x"].clone().requires_grad_(True)
    p, _ = fos.fixed_order_softmax(x, sink=c["sink"], batch=1, heads=2, q_len=4)
    p.backward(c["dp"].float().to(torch.bfloat16))
    assert x.grad is not None and x.grad.dtype == torch.bfloat16


def test_attention_refuses_cpu_tensors():
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16, requires_grad=True)
    k = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fos.fixed_order_attention(q, k, k)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("Hkv", [1, 2])
def test_attention_gradients_are_the_direct_calls_bits(dtype, Hkv):
    # fixed_order_attention's output and its dQ, dK, dV against the same library calls made
    # directly (QK, softmax in place, PV; dP by QK, dS in place, dQ by PV with the scale, dK and
    # dV by the key / value gradient kernel), bit for bit
    B, Hq, Sq, Skv, D = 2, 4, 130, 200, 64
    g = torch.Generator(device="cuda").manual_seed(Hkv + 90)
    q = torch.randn(B, Hq, Sq, D, generator=g, device="cuda").to(dtype)
    k = torch.randn(B, Hkv, Skv, D, generator=g, device="cuda").to(dtype)
    v = torch.randn(B, Hkv, Skv, D, generator=g, device="cuda").to(dtype)
    dout = torch.randn(B, Hq, Sq, D, generator=g, device="cuda").to(dtype)
    qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = fos.fixed_order_attention(qa, ka, va)
    out.backward(dout)
    scale = D ** -0.5
    s = fos.fos_qk_scores(q, k, scale, out_dtype=dtype)
    fos.fos_softmax_fwd(s, s, batch=B, heads=Hq, q_len=Sq)
    o_ref = fos.fos_pv_out(s, v, out_dtype=dtype)
    dp = fos.fos_qk_scores(dout, v, 1.0, out_dtype=dtype)
    fos.fos_softmax_bwd(s, dp, dp, batch=B, heads=Hq, q_len=Sq, want_delta=False)
    dq = fos.fos_pv_out(dp, k, scale=scale, out_dtype=dtype)
    dk = fos.fos_grad_kv(dp, q, Hkv, scale, out_dtype=dtype)
    dv = fos.fos_grad_kv(s, dout, Hkv, out_dtype=dtype)
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
    assert bits_equal(out.detach(), o_ref)
    for got, ref in ((qa.grad, dq), (ka.grad, dk), (va.grad, dv)):
        assert got.dtype == dtype and bits_equal(got, ref)


CHILD_BACKWARD = """
import torch
import deterministic_attention_softmax_gb300 as fos
g = torch.Generator(device="cuda").manual_seed(7)
q = torch.randn(1, 2, 70, 64, generator=g, device="cuda").to(torch.bfloat16).requires_grad_()
k = torch.randn(1, 1, 90, 64, generator=g, device="cuda").to(torch.bfloat16).requires_grad_()
v = torch.randn(1, 1, 90, 64, generator=g, device="cuda").to(torch.bfloat16).requires_grad_()
out = fos.fixed_order_attention(q, k, v, causal=True)
out.backward(torch.ones_like(out))
torch.cuda.synchronize()
assert fos.fos_device_error() == 0
print("ok", float(q.grad.float().abs().sum()), float(v.grad.float().abs().sum()))
"""


@pytest.mark.gpu
def test_attention_backward_first_on_a_fresh_autograd_thread():
    # In a fresh process the attention backward is the first library call on PyTorch's autograd
    # worker thread, which has no CUDA context bound yet; the contractions' tensor maps need one
    # (they are bound before encoding).  This failed with FOS_ERR_UNSUPPORTED before the fix.
    import os
    import subprocess
    import sys

    from conftest import ROOT

    r = subprocess.run([sys.executable, "-c", CHILD_BACKWARD], cwd=ROOT, capture_output=True,
                       text=True, timeout=600, env=dict(os.environ))
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout + r.stderr[-3000:]

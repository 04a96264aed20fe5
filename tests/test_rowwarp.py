"""Rows of at most 8 tiles go to the one-warp-per-row kernels by default (forward and
backward); ``generic=1`` keeps them on the CTA kernels.  Both must give the same bits (P, LSE,
dScores, delta) for every mask, a sink, every dtype, and any geometry of the one-warp kernels
(warps per CTA, buffers per warp, CTAs).  Parity against the oracle for short rows is covered by
the small parity grid."""

import pytest
import torch

import deterministic_attention_softmax_gb300 as fos
from gpu_util import bits_equal
from test_parity_small import make_case

pytestmark = pytest.mark.gpu

CTA = fos.Launch(generic=1)


def fwd(c, launch=None):
    kw = dict(batch=c["B"], heads=c["H"], q_len=c["Sq"], causal=c["causal"],
              kv_valid_len=c["kv"], key_mask=c["km"])
    return fos.fos_softmax_fwd(c["x"], sink=c["sink"], launch=launch, **kw)


def bwd(c, p, launch=None):
    kw = dict(batch=c["B"], heads=c["H"], q_len=c["Sq"], causal=c["causal"],
              kv_valid_len=c["kv"], key_mask=c["km"])
    return fos.fos_softmax_bwd(p, c["dp"], launch=launch, **kw)


@pytest.mark.parametrize("dtype,L", [(torch.bfloat16, 8), (torch.bfloat16, 200),
                                     (torch.bfloat16, 256), (torch.bfloat16, 264),
                                     (torch.bfloat16, 1000), (torch.bfloat16, 2048),
                                     (torch.float32, 1020), (torch.float16, 2048),
                                     (torch.float32, 4)])
@pytest.mark.parametrize("mask", ["none", "causal", "kvlen", "keymask", "sink", "all"])
def test_one_warp_rows_match_the_cta_kernel(dtype, L, mask):
    c = make_case(dtype, L, mask, B=3, H=4, Sq=37, seed=7)
    p, lse = fwd(c)
    p2, lse2 = fwd(c, CTA)
    ds, delta = bwd(c, p)
    ds2, delta2 = bwd(c, p, CTA)
    torch.cuda.synchronize()
    assert bits_equal(p, p2) and bits_equal(lse, lse2)
    assert bits_equal(ds, ds2) and bits_equal(delta, delta2)
    assert fos.fos_device_error() == 0


@pytest.mark.parametrize("opts", [dict(warps_per_cta=1), dict(warps_per_cta=2),
                                  dict(warps_per_cta=3), dict(warps_per_cta=8),
                                  dict(warps_per_cta=16), dict(stages=1), dict(stages=4),
                                  dict(warps_per_cta=2, stages=8), dict(ctas=1), dict(ctas=7),
                                  dict(load_path=1)],
                         ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()))
def test_one_warp_geometry_does_not_change_bits(opts):
    c = make_case(torch.bfloat16, 2048, "all", B=2, H=3, Sq=129, seed=3)
    ref = fwd(c, CTA)
    out = fwd(c, fos.Launch(**opts))
    gref = bwd(c, ref[0], CTA)
    gout = bwd(c, ref[0], fos.Launch(**opts))
    torch.cuda.synchronize()
    assert bits_equal(ref[0], out[0]) and bits_equal(ref[1], out[1])
    assert bits_equal(gref[0], gout[0]) and bits_equal(gref[1], gout[1])


def test_unaligned_short_rows_fall_back_to_plain_loads():
    # 2-byte offset: no bulk copies; the default launch still works (CTA kernel, plain loads),
    # a forced bulk path is refused
    buf = torch.randn(40 * 512 + 1, device="cuda").to(torch.bfloat16)
    x = buf[1:].view(40, 512)
    p, lse = fos.fos_softmax_fwd(x)
    p2, lse2 = fos.fos_softmax_fwd(x.clone())  # aligned copy: the one-warp kernel
    assert bits_equal(p, p2) and bits_equal(lse, lse2)
    with pytest.raises(fos.FosError) as e:
        fos.fos_softmax_fwd(x, launch=fos.Launch(load_path=1))
    assert e.value.status == 2
    dp = torch.randn(40 * 512 + 1, device="cuda").to(torch.bfloat16)[1:].view(40, 512)
    ds, delta = fos.fos_softmax_bwd(p, dp)  # unaligned dP: the CTA kernel, plain loads
    ds2, delta2 = fos.fos_softmax_bwd(p, dp.clone())
    assert bits_equal(ds, ds2) and bits_equal(delta, delta2)

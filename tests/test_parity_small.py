"""GPU vs FP64 oracle, element by element, on small problems that span several tiles and a
ragged tail, for every I/O dtype and mask kind, plus the edge cases (one key, fully masked
rows, -inf sinks, long rows past the register path, the longest staged rows, unaligned
rows, in-place calls).  All calls go through the C ABI."""

import math

import numpy as np
import pytest
import torch

import deterministic_attention_softmax_gb300 as fos
from gpu_util import (DTYPES, assert_check, bits_equal, check_bwd, check_fwd, dev, masks_np,
                      np64, oracle, tol)

pytestmark = pytest.mark.gpu

# tiny rows, a lane's 8 keys, the tile (256), the one-warp kernel's 2 / 4 / 8-tile instances on
# both sides of each boundary (512, 1024, 2048 keys; 2049 goes to the row groups), Qwen-Image's
# 4352
LENGTHS = [1, 2, 3, 7, 8, 255, 256, 257, 511, 512, 513, 1000, 1024, 1025, 2048, 2049, 4352]
MASKS = ["none", "causal", "kvlen", "keymask", "sink", "all"]


def make_case(dtype, L, mask, B=2, H=3, Sq=5, seed=0, sigma=3.0):
    g = torch.Generator(device="cuda").manual_seed(1000 * L + 17 * seed + MASKS.index(mask)
                                                   if mask in MASKS else seed)
    d = dev()
    Sq = min(Sq, L) if mask in ("causal", "all") else Sq
    rows = B * H * Sq
    x = (torch.randn(rows, L, generator=g, device=d) * sigma).to(dtype)
    dp = torch.randn(rows, L, generator=g, device=d).to(dtype)
    kv = km = sink = None
    causal = mask in ("causal", "all")
    if mask in ("kvlen", "all"):
        kv = torch.randint(0, L + 1, (B,), generator=g, device=d, dtype=torch.int32)
        kv[0] = L  # one full, one random
    if mask in ("keymask", "all"):
        km = (torch.rand(B, L, generator=g, device=d) < 0.7).to(torch.uint8)
    if mask in ("sink", "all"):
        sink = torch.randn(H, generator=g, device=d)
    return dict(x=x, dp=dp, kv=kv, km=km, sink=sink, B=B, H=H, Sq=Sq, causal=causal)


def run_and_check(dtype_name, c, launch=None, check_sink=True):
    dt = DTYPES[dtype_name]
    B, H, Sq = c["B"], c["H"], c["Sq"]
    kw = dict(batch=B, heads=H, q_len=Sq, causal=c["causal"], kv_valid_len=c["kv"],
              key_mask=c["km"])
    p, lse = fos.fos_softmax_fwd(c["x"], sink=c["sink"], launch=launch, **kw)
    kvn, kmn, skn = masks_np(c["kv"], c["km"], c["sink"])
    okw = dict(batch=B, heads=H, q_len=Sq, causal=c["causal"], kv_valid_len=kvn, key_mask=kmn)
    p_ref, lse_ref = oracle.softmax_fwd(np64(c["x"]), sink=skn, **okw)
    check_fwd(p, lse, p_ref, lse_ref, dtype_name)

    # backward on the oracle's P rounded to the dtype (independent of the CUDA forward)
    p_in = torch.from_numpy(p_ref).to(dt).to(dev())
    ds, delta = fos.fos_softmax_bwd(p_in, c["dp"], launch=launch, **kw)
    pin, dpn = np64(p_in), np64(c["dp"])
    ds_ref, delta_ref = oracle.softmax_bwd(pin, dpn, **okw)
    check_bwd(ds, delta, ds_ref, delta_ref, pin, dpn, dtype_name)

    if c["sink"] is not None and check_sink:
        d_sink = fos.fos_sink_grad(lse, delta, c["sink"], batch=B, heads=H, q_len=Sq,
                                   launch=launch)
        ref = oracle.sink_grad(lse_ref, delta_ref, skn, batch=B, heads=H, q_len=Sq)
        assert_check(tol.check_dsink(np64(d_sink), ref, lse_ref, delta_ref, skn, B, H, Sq),
                     "d_sink")
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
    return p, lse


@pytest.mark.parametrize("dtype_name", list(DTYPES))
@pytest.mark.parametrize("L", LENGTHS)
@pytest.mark.parametrize("mask", MASKS)
def test_small_grid(dtype_name, L, mask):
    run_and_check(dtype_name, make_case(DTYPES[dtype_name], L, mask))


@pytest.mark.parametrize("dtype_name", list(DTYPES))
def test_fully_masked_rows_and_minus_inf_sink(dtype_name):
    dt = DTYPES[dtype_name]
    c = make_case(dt, 300, "all", B=3, H=2, Sq=4)
    c["kv"] = torch.tensor([0, 300, 5], dtype=torch.int32, device=dev())
    c["sink"] = torch.tensor([-math.inf, 0.5], device=dev())
    c["x"][13, :] = float("-inf")  # a row (b=1, h=1) that is all -inf on its own
    p, lse = run_and_check(dtype_name, c)
    lse_h = lse.cpu().numpy()
    # batch 0 has no valid key: head 0 (sink -inf) gives -inf, head 1 gives its sink
    assert np.all(np.isneginf(lse_h[0:4])) and np.all(lse_h[4:8] == np.float32(0.5))
    assert torch.all(p[0:8] == 0)


@pytest.mark.parametrize("dtype_name", list(DTYPES))
@pytest.mark.parametrize("L", [8193, 16384])
def test_rows_past_the_register_path(dtype_name, L):
    # 33 and 64 tiles: the forward parks e_j in tensor memory with 5 and 8 warps (two warps share
    # a lane quarter, side by side in its columns); the backward re-reads P and dP from shared
    # memory
    run_and_check(dtype_name, make_case(DTYPES[dtype_name], L, "all", B=1, H=2, Sq=3))


@pytest.mark.parametrize("dtype_name", list(DTYPES))
@pytest.mark.parametrize("L", [16385, 24576, 32768])
def test_widest_parked_forward_layout(dtype_name, L):
    # 65, 96 and 128 tiles on the default launch: the CTA forward takes 9, 12 and 16 compute
    # warps with 8 tiles each parked in tensor memory, so up to four warps share a lane quarter
    # side by side in its columns (256 columns per CTA).  Every mask kind and a sink; 18 rows.
    run_and_check(dtype_name, make_case(DTYPES[dtype_name], L, "all", B=2, H=3, Sq=3))


@pytest.mark.parametrize("dtype_name", list(DTYPES))
@pytest.mark.parametrize("L", [18432, 32768])
@pytest.mark.parametrize("mask", ["none", "all"])
def test_wide_layouts_match_the_recompute_path(dtype_name, L, mask):
    # 72 and 128 tiles over 9, 12 and 16 warps: at 72 tiles every count parks e_j (8, 6 and 6
    # tiles per warp: three, three and four warps per lane quarter); at 128 tiles 16 warps park
    # 8 each while 9 and 12 warps recompute e_j in the second pass.  Eight warps (9 and 16
    # tiles per warp) recompute in both.  All must give the same bits, for the instance
    # specialised for unmasked rows and for the general one.
    c = make_case(DTYPES[dtype_name], L, mask, B=2, H=2, Sq=4)
    kw = dict(batch=c["B"], heads=c["H"], q_len=c["Sq"], causal=c["causal"],
              kv_valid_len=c["kv"], key_mask=c["km"], sink=c["sink"])
    ref = fos.fos_softmax_fwd(c["x"], launch=fos.Launch(warps_per_cta=8), **kw)
    for warps in (9, 12, 16):
        out = fos.fos_softmax_fwd(c["x"], launch=fos.Launch(warps_per_cta=warps), **kw)
        assert bits_equal(ref[0], out[0]) and bits_equal(ref[1], out[1]), warps
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0


@pytest.mark.parametrize("dtype_name,L_fwd,L_bwd", [("float32", 57000, 28672),
                                                    ("bfloat16", 100000, 57344),
                                                    ("float16", 100000, 57344)])
def test_longest_rows(dtype_name, L_fwd, L_bwd):
    dt = DTYPES[dtype_name]
    c = make_case(dt, L_fwd, "sink", B=1, H=1, Sq=2)
    p, lse = fos.fos_softmax_fwd(c["x"], sink=c["sink"], batch=1, heads=1, q_len=2)
    p_ref, lse_ref = oracle.softmax_fwd(np64(c["x"]), sink=np64(c["sink"]), batch=1, heads=1,
                                        q_len=2)
    check_fwd(p, lse, p_ref, lse_ref, dtype_name)
    c = make_case(dt, L_bwd, "none", B=1, H=1, Sq=2)
    p_ref, _ = oracle.softmax_fwd(np64(c["x"]), batch=1, heads=1, q_len=2)
    p_in = torch.from_numpy(p_ref).to(dt).to(dev())
    ds, delta = fos.fos_softmax_bwd(p_in, c["dp"], batch=1, heads=1, q_len=2)
    ds_ref, delta_ref = oracle.softmax_bwd(np64(p_in), np64(c["dp"]), batch=1, heads=1, q_len=2)
    check_bwd(ds, delta, ds_ref, delta_ref, np64(p_in), np64(c["dp"]), dtype_name)


@pytest.mark.parametrize("dtype_name", list(DTYPES))
def test_unaligned_rows_and_row_stride(dtype_name):
    # odd row stride and a base pointer one element past an aligned address: plain loads and
    # element stores must still match the oracle
    dt = DTYPES[dtype_name]
    g = torch.Generator(device="cuda").manual_seed(5)
    rows, L, ld = 12, 777, 781
    buf = (torch.randn(rows * ld + 1, generator=g, device=dev()) * 3).to(dt)
    x = buf[1:].view(rows, ld)[:, :L]
    p, lse = fos.fos_softmax_fwd(x, batch=1, heads=1, q_len=rows)
    p_ref, lse_ref = oracle.softmax_fwd(np64(x), batch=1, heads=1, q_len=rows)
    check_fwd(p, lse, p_ref, lse_ref, dtype_name, "unaligned")
    dpb = torch.randn(rows * ld + 1, generator=g, device=dev()).to(dt)
    dp = dpb[1:].view(rows, ld)[:, :L]
    pb = torch.empty(rows * ld + 1, dtype=dt, device=dev())
    p_in = pb[1:].view(rows, ld)[:, :L]
    p_in.copy_(torch.from_numpy(p_ref).to(dt))
    ds, delta = fos.fos_softmax_bwd(p_in, dp, batch=1, heads=1, q_len=rows)
    ds_ref, delta_ref = oracle.softmax_bwd(np64(p_in), np64(dp), batch=1, heads=1, q_len=rows)
    check_bwd(ds, delta, ds_ref, delta_ref, np64(p_in), np64(dp), dtype_name, what="unaligned")


@pytest.mark.parametrize("dtype_name", list(DTYPES))
def test_in_place(dtype_name):
    dt = DTYPES[dtype_name]
    c = make_case(dt, 1000, "all")
    kw = dict(batch=c["B"], heads=c["H"], q_len=c["Sq"], causal=True, kv_valid_len=c["kv"],
              key_mask=c["km"])
    p_out, lse_out = fos.fos_softmax_fwd(c["x"], sink=c["sink"], **kw)
    x2 = c["x"].clone()
    p_in, lse_in = fos.fos_softmax_fwd(x2, probs=x2, sink=c["sink"], **kw)
    assert p_in.data_ptr() == x2.data_ptr()
    assert bits_equal(p_in, p_out) and bits_equal(lse_in, lse_out)
    ds_out, d_out = fos.fos_softmax_bwd(p_out, c["dp"], **kw)
    dp2 = c["dp"].clone()
    ds_in, d_in = fos.fos_softmax_bwd(p_out, dp2, dscores=dp2, **kw)
    assert bits_equal(ds_in, ds_out) and bits_equal(d_in, d_out)


def test_zero_rows():
    x = torch.empty(0, 64, dtype=torch.bfloat16, device=dev())
    p, lse = fos.fos_softmax_fwd(x, batch=0, heads=1, q_len=1)
    assert p.shape == (0, 64) and lse.shape == (0,)


def test_exp_accuracy_on_two_key_rows():
    # The library's exp is 2^(x*log2 e) on the hardware base-2 approximation.  Its error over
    # the arguments the kernels use (x - max in [-80, 0]) is observed through two-key rows,
    # P_1 = exp(x1) / (1 + exp(x1)), against the exact value: a few float32 ulp near 0 and far
    # inside the 1e-6 float32 P tolerance everywhere.
    x1 = torch.linspace(-80, 0, 4001, device=dev())
    rows = torch.stack([torch.zeros_like(x1), x1], dim=1).contiguous()
    p, lse = fos.fos_softmax_fwd(rows)
    e = np.exp(np64(x1))
    p1_ref = e / (1 + e)
    err = np.abs(np64(p)[:, 1] - p1_ref)
    assert err.max() < 2e-7, err.max()


@pytest.mark.parametrize("dtype_name", list(DTYPES))
def test_deep_tiles_keep_subnormal_results(dtype_name):
    # One dominant key per row (x = 0) and every other key 88..94 below it: the normaliser is
    # about 1, so those probabilities are about e^-88..e^-94, below 2^-126 (subnormal in float32
    # and bf16, where 1 ULP of the FP64 value is 2^-133).  The dominant key's tile holds keys
    # more than 87 below its maximum and must keep subnormal exponentials; the other tiles
    # reach the subnormal range through their per-tile scale.
    dt = DTYPES[dtype_name]
    g = torch.Generator(device="cuda").manual_seed(77)
    rows, L = 40, 2048
    x = -88.0 - 6.0 * torch.rand(rows, L, generator=g, device=dev())
    x[:, 0] = 0.0
    x = x.to(dt)
    p, lse = fos.fos_softmax_fwd(x, q_len=rows)
    p_ref, lse_ref = oracle.softmax_fwd(np64(x), batch=1, heads=1, q_len=rows)
    check_fwd(p, lse, p_ref, lse_ref, dtype_name, "deep tiles")
    if dtype_name != "float16":  # fp16 has no range down there
        tiny = (p_ref > 2.0 ** -133) & (p_ref < 2.0 ** -126)
        assert tiny.sum() > 1000 and (np64(p)[tiny] > 0).all()
        first_tile = np.zeros_like(tiny)
        first_tile[:, 1:256] = True
        assert (tiny & first_tile).any()  # the exact path of the dominant key's tile

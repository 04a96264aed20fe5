"""Bitwise invariance on the GPU: a row gives the same bits whatever its batch size, its
position in the batch, its row offset, the launch geometry (CTAs, warps per CTA, pipeline
stages), the load path (bulk copy or plain loads, aligned or not), whether padding is given
as -inf scores or as valid lengths or a key mask, whether a -inf sink or no sink is given, and
whether the rows are processed in one launch or several.  ("[WS1][kernels] Add fixed-order
joint-attention softmax for Qwen-Image", Summary: the same row must not produce different
results because of its batch, launch geometry or backend; "Batch-invariant attention",
Acceptance Criteria: batch-size, batch-position and chunking invariance, bitwise.)"""

import math

import pytest
import torch

import deterministic_attention_softmax_gb300 as fos
from deterministic_attention_softmax_gb300 import workloads as W
from gpu_util import DTYPES, bits_equal, dev

pytestmark = pytest.mark.gpu


def fwd_bwd(x, dp, **kw):
    sink = kw.pop("sink", None)
    launch = kw.pop("launch", None)
    p, lse = fos.fos_softmax_fwd(x, sink=sink, launch=launch, **kw)
    ds, delta = fos.fos_softmax_bwd(p, dp, launch=launch, **kw)
    return p, lse, ds, delta


# ------------------------------------------------------------------ batch size and position


@pytest.mark.parametrize("dtype_name", ["bfloat16", "float32"])
def test_large_workload_sample_reembedded_at_batch_1_7_64(dtype_name):
    # The large workload's sample: 24 heads x 512 query rows x 8192 keys (sigma 5), placed at
    # several positions of batches of 1, 7 and 64 samples; the other samples are other noise.
    dt = DTYPES[dtype_name]
    H, Sq, L, sigma, seed = 24, 512, 8192, 5.0, 4
    n = H * Sq
    d = dev()
    xs = W.sample_rows(H, Sq, L, sigma, seed, 0, dt, d)
    dps = W.sample_rows(H, Sq, L, 1.0, seed + 1, 0, dt, d)
    ref = fwd_bwd(xs, dps, batch=1, heads=H, q_len=Sq)
    for B, positions in ((7, (0, 3, 6)), (64, (0, 37, 63))):
        x = W.normal((B * n, L), sigma, seed * 7 + B, dt, d)
        dp = W.normal((B * n, L), 1.0, seed * 11 + B, dt, d)
        for k in positions:
            x[k * n:(k + 1) * n] = xs
            dp[k * n:(k + 1) * n] = dps
        out = fwd_bwd(x, dp, batch=B, heads=H, q_len=Sq)
        for k in positions:
            sl = slice(k * n, (k + 1) * n)
            for a, b_ in zip(ref, out):
                assert bits_equal(a, b_[sl]), f"batch {B} position {k} differs"
        del x, dp, out
        torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype_name", ["bfloat16", "float32", "float16"])
@pytest.mark.parametrize("offset", [1, 3, 17, 4097])
def test_row_offsets(dtype_name, offset):
    dt = DTYPES[dtype_name]
    d = dev()
    n, L = 3000, 4608
    xs = W.normal((n, L), 4.0, 21, dt, d)
    dps = W.normal((n, L), 1.0, 22, dt, d)
    ref = fwd_bwd(xs, dps)
    x = W.normal((offset + n + 5, L), 4.0, 23, dt, d)
    dp = W.normal((offset + n + 5, L), 1.0, 24, dt, d)
    x[offset:offset + n] = xs
    dp[offset:offset + n] = dps
    out = fwd_bwd(x, dp)
    for a, b_ in zip(ref, out):
        assert bits_equal(a, b_[offset:offset + n])


# ------------------------------------------------------------------ launch geometry


def masked_case(dt, L=4400, B=2, H=4, Sq=64, seed=31):
    d = dev()
    g = torch.Generator(device="cuda").manual_seed(seed)
    rows = B * H * Sq
    x = (torch.randn(rows, L, generator=g, device=d) * 4).to(dt)
    dp = torch.randn(rows, L, generator=g, device=d).to(dt)
    kv = torch.tensor([L - 123, L], dtype=torch.int32, device=d)
    km = (torch.rand(B, L, generator=g, device=d) < 0.9).to(torch.uint8)
    sink = torch.randn(H, generator=g, device=d)
    kw = dict(batch=B, heads=H, q_len=Sq, causal=True, kv_valid_len=kv, key_mask=km, sink=sink)
    return x, dp, kw


LAUNCHES = [
    dict(warps_per_cta=1), dict(warps_per_cta=2), dict(warps_per_cta=3), dict(warps_per_cta=4),
    dict(warps_per_cta=16), dict(ctas=1), dict(ctas=3), dict(ctas=152), dict(ctas=1000),
    dict(stages=1), dict(stages=2), dict(stages=3), dict(stages=5), dict(load_path=1),
    dict(load_path=2), dict(load_path=2, warps_per_cta=5, ctas=77),
]


@pytest.mark.parametrize("dtype_name", ["bfloat16", "float32", "float16"])
@pytest.mark.parametrize("opts", LAUNCHES, ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()))
def test_launch_geometry(dtype_name, opts):
    x, dp, kw = masked_case(DTYPES[dtype_name])
    ref = fwd_bwd(x, dp, **kw)
    out = fwd_bwd(x, dp, launch=fos.Launch(**opts), **kw)
    for a, b_ in zip(ref, out):
        assert bits_equal(a, b_)


UNMASKED_LAUNCHES = [
    dict(generic=1), dict(warps_per_cta=1), dict(warps_per_cta=2), dict(warps_per_cta=3),
    dict(warps_per_cta=5), dict(warps_per_cta=9), dict(warps_per_cta=16), dict(ctas=7),
    dict(stages=1), dict(stages=2), dict(load_path=2), dict(generic=1, warps_per_cta=3),
]


@pytest.mark.parametrize("dtype_name", ["bfloat16", "float32", "float16"])
@pytest.mark.parametrize("L", [4352, 4400, 8192])
@pytest.mark.parametrize("opts", UNMASKED_LAUNCHES,
                         ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()))
def test_unmasked_rows_fast_and_generic_kernels_agree(dtype_name, L, opts):
    # Unmasked, sink-free, aligned rows take the kernel specialised for that case by default;
    # every other launch (generic kernel, plain loads, other register splits) gives its bits.
    dt = DTYPES[dtype_name]
    x = W.normal((300, L), 4.0, 41, dt, dev())
    dp = W.normal((300, L), 1.0, 42, dt, dev())
    ref = fwd_bwd(x, dp)
    out = fwd_bwd(x, dp, launch=fos.Launch(**opts))
    for a, b_ in zip(ref, out):
        assert bits_equal(a, b_)


@pytest.mark.parametrize("dtype_name", ["bfloat16", "float32", "float16"])
def test_unaligned_copy_matches_aligned(dtype_name):
    # same rows at a base pointer one element off 16-byte alignment (plain element loads and
    # element stores) and at an aligned one (bulk copies, 16-byte stores)
    dt = DTYPES[dtype_name]
    x, dp, kw = masked_case(dt)
    ref = fwd_bwd(x, dp, **kw)
    rows, L = x.shape
    bx = torch.empty(rows * L + 1, dtype=dt, device=dev())
    bd = torch.empty(rows * L + 1, dtype=dt, device=dev())
    xu = bx[1:].view(rows, L)
    dpu = bd[1:].view(rows, L)
    xu.copy_(x)
    dpu.copy_(dp)
    out = fwd_bwd(xu, dpu, **kw)
    for a, b_ in zip(ref, out):
        assert bits_equal(a, b_)


def test_repeat_runs_identical():
    x, dp, kw = masked_case(torch.bfloat16)
    a = fwd_bwd(x, dp, **kw)
    for _ in range(3):
        b_ = fwd_bwd(x, dp, **kw)
        for u, v in zip(a, b_):
            assert bits_equal(u, v)


def test_split_launches_match_one_launch():
    # rows processed in two launches (batch entries 0 and 1 separately) give the same bits
    x, dp, kw = masked_case(torch.bfloat16)
    ref = fwd_bwd(x, dp, **kw)
    half = x.shape[0] // 2
    for b in range(2):
        sl = slice(b * half, (b + 1) * half)
        kb = dict(kw, batch=1, kv_valid_len=kw["kv_valid_len"][b:b + 1].contiguous(),
                  key_mask=kw["key_mask"][b:b + 1].contiguous())
        out = fwd_bwd(x[sl], dp[sl], **kb)
        for a, b_ in zip(ref, out):
            assert bits_equal(a[sl], b_)


# ------------------------------------------------------------------ masks and sinks


@pytest.mark.parametrize("full", [False, True], ids=["small", "prompt_padding_full"])
def test_neg_inf_tail_equals_valid_lengths_and_key_mask(full):
    base = W.WORKLOADS["prompt_padding_bf16"]
    w = base if full else W.Workload("pad_small", base.dtype, 4, 3, 32, base.key_len,
                                     base.score_sigma, seed=base.seed, pad=base.pad)
    d = dev()
    x_inf = W.scores(w, d)                     # tail = -inf
    x_raw = W.scores(w, d, neg_inf_tail=False)  # tail = ordinary noise
    dp = W.dprobs(w, d)
    kv = W.valid_lengths(w).to(d)
    km = (torch.arange(w.key_len, device=d)[None, :] < kv[:, None]).to(torch.uint8)
    geo = dict(batch=w.batch, heads=w.heads, q_len=w.q_len)
    p_a, lse_a = fos.fos_softmax_fwd(x_inf, **geo)
    p_b, lse_b = fos.fos_softmax_fwd(x_raw, kv_valid_len=kv, **geo)
    p_c, lse_c = fos.fos_softmax_fwd(x_raw, key_mask=km, **geo)
    assert bits_equal(p_a, p_b) and bits_equal(lse_a, lse_b)
    assert bits_equal(p_a, p_c) and bits_equal(lse_a, lse_c)
    ds_a, de_a = fos.fos_softmax_bwd(p_a, dp, **geo)                   # no mask: P is 0 there
    ds_b, de_b = fos.fos_softmax_bwd(p_b, dp, kv_valid_len=kv, **geo)  # tail skipped
    ds_c, de_c = fos.fos_softmax_bwd(p_c, dp, key_mask=km, **geo)
    assert bits_equal(ds_a, ds_b) and bits_equal(de_a, de_b)
    assert bits_equal(ds_a, ds_c) and bits_equal(de_a, de_c)


@pytest.mark.parametrize("dtype_name", ["bfloat16", "float32"])
def test_minus_inf_sink_equals_no_sink(dtype_name):
    x, dp, kw = masked_case(DTYPES[dtype_name])
    kw.pop("sink")
    p0, l0 = fos.fos_softmax_fwd(x, **kw)
    H = kw["heads"]
    p1, l1 = fos.fos_softmax_fwd(x, sink=torch.full((H,), -math.inf, device=dev()), **kw)
    assert bits_equal(p0, p1) and bits_equal(l0, l1)


def test_sink_grad_geometry_invariant():
    w = W.WORKLOADS["sink_causal_bf16"]
    d = dev()
    g = torch.Generator(device="cpu").manual_seed(7)
    sink = W.sink_logits(w).to(d)
    lse = (torch.randn(w.rows, generator=g).abs() + 2).to(d)
    delta = (torch.randn(w.rows, generator=g) * 0.3).to(d)
    geo = dict(batch=w.batch, heads=w.heads, q_len=w.q_len)
    ref = fos.fos_sink_grad(lse, delta, sink, **geo)
    for warps in (1, 2, 3, 8, 16):
        out = fos.fos_sink_grad(lse, delta, sink, launch=fos.Launch(warps_per_cta=warps), **geo)
        assert bits_equal(ref, out)


@pytest.mark.parametrize("warps", list(range(1, 17)))
def test_every_warp_count_gives_the_same_bits(warps):
    # The CTA forward parks e_j in tensor memory: warp w in lane quarter w % 4, warps that share
    # a quarter side by side in its columns.  Every split of a 17-tile row over 1..16 warps
    # (parked or, past 8 tiles per warp, recomputed) gives the default launch's bits.
    x = W.normal((600, 4352), 4.0, 43, torch.bfloat16, dev())
    ref = fos.fos_softmax_fwd(x)
    out = fos.fos_softmax_fwd(x, launch=fos.Launch(warps_per_cta=warps))
    torch.cuda.synchronize()
    assert bits_equal(ref[0], out[0]) and bits_equal(ref[1], out[1])
    assert fos.fos_device_error() == 0


@pytest.mark.parametrize("L,opts", [(4352, dict()), (4352, dict(generic=1)),
                                    (200, dict(generic=1)), (2048, dict(generic=1, warps_per_cta=1))])
def test_more_ctas_than_tensor_memory_serves(L, opts):
    # One CTA per row: at most 512 / (columns per CTA) CTAs can hold tensor memory on an SM at
    # once.  The launch pads shared memory so that no more are resident; the others start as
    # resident ones exit.  Same bits as the default grid.
    x = W.normal((4096, L), 4.0, 44, torch.bfloat16, dev())
    ref = fos.fos_softmax_fwd(x, launch=fos.Launch(**opts) if opts else None)
    out = fos.fos_softmax_fwd(x, launch=fos.Launch(ctas=4096, **opts))
    torch.cuda.synchronize()
    assert bits_equal(ref[0], out[0]) and bits_equal(ref[1], out[1])
    assert fos.fos_device_error() == 0


# ------------------------------------------------------------------ row groups per CTA


@pytest.mark.parametrize("dtype_name", ["bfloat16", "float32", "float16"])
@pytest.mark.parametrize("L", [2304, 4352, 8192, 16384])
@pytest.mark.parametrize("masked", [False, True], ids=["unmasked", "masked"])
def test_row_groups_per_cta_give_the_same_bits(dtype_name, L, masked):
    # Rows whose warps park all their tiles in tensor memory run as row groups, several per
    # CTA, each group with its own ring of row buffers and its last warp issuing the copies.
    # Every split (groups per CTA, ring depth, CTAs) gives the bits of the general
    # one-row-per-CTA kernel; a split that does not fit the SM is refused as unsupported.
    dt = DTYPES[dtype_name]
    if masked:
        x, _, kw = masked_case(dt, L=L, Sq=48)
    else:
        x, kw = W.normal((700, L), 4.0, 51, dt, dev()), {}
    ref = fos.fos_softmax_fwd(x, launch=fos.Launch(generic=1), **kw)
    ran = 0
    for ng in (1, 2, 3, 4, 5, 8, 10):
        for ns in (1, 2, 3):
            for ctas in (0, 7):
                try:
                    out = fos.fos_softmax_fwd(
                        x, launch=fos.Launch(groups_per_cta=ng, stages=ns, ctas=ctas), **kw)
                except fos.FosError as e:
                    assert e.status == 2, (ng, ns, ctas)  # FOS_ERR_UNSUPPORTED
                    continue
                assert bits_equal(ref[0], out[0]) and bits_equal(ref[1], out[1]), (ng, ns, ctas)
                ran += 1
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
    assert ran >= 6

"""Guard bands: the kernels write nothing outside their outputs.  Outputs are views into larger
buffers filled with a sentinel pattern -- guard rows before and after, and the gap columns
key_len..ld-1 of every row -- and every byte outside the written region must still hold the
sentinel afterwards.  Covers the bulk-copy and plain-load paths, masks, and the sink."""

import pytest
import torch

import deterministic_attention_softmax_gb300 as fos
from gpu_util import DTYPES, dev

pytestmark = pytest.mark.gpu

GUARD = 3  # guard rows on each side


def guarded(rows, L, ld, dt, fill):
    """A (rows + 2*GUARD, ld) buffer of `fill` bytes and the [rows, L] view inside it."""
    buf = torch.empty((rows + 2 * GUARD) * ld, dtype=dt, device=dev())
    buf.view(torch.uint8).fill_(fill)
    view = buf.view(rows + 2 * GUARD, ld)[GUARD:GUARD + rows, :L]
    return buf, view


def untouched(buf, rows, L, ld, fill):
    b = buf.view(rows + 2 * GUARD, ld)
    inside = torch.zeros_like(b, dtype=torch.bool)
    inside[GUARD:GUARD + rows, :L] = True
    bytes_ = b.contiguous().view(torch.uint8).view(rows + 2 * GUARD, -1)
    esz = b.element_size()
    mask = inside.repeat_interleave(esz, dim=1)
    return bool(torch.all(bytes_[~mask] == fill))


def guarded_vec(n, fill):
    v = torch.empty(n + 2 * GUARD, dtype=torch.float32, device=dev())
    v.view(torch.uint8).fill_(fill)
    return v, v[GUARD:GUARD + n]


def vec_untouched(v, n, fill):
    b = v.view(torch.uint8)
    return bool(torch.all(b[:GUARD * 4] == fill) and torch.all(b[(GUARD + n) * 4:] == fill))


@pytest.mark.parametrize("dtype_name", list(DTYPES))
# 4352 / 4608: CTA kernels with e_j parked in tensor memory; 2048 / 1024 (aligned): one warp per
# row, e_j parked; 777 / 257 (unaligned): CTA kernels with plain loads, e_j in registers
@pytest.mark.parametrize("L,ld", [(4352, 4360), (4608, 4608), (2048, 2056), (1024, 1024),
                                  (777, 781), (257, 264)])
@pytest.mark.parametrize("masked", [False, True])
def test_outputs_stay_inside_their_rows(dtype_name, L, ld, masked):
    dt = DTYPES[dtype_name]
    B, H, Sq = 2, 3, 8
    rows = B * H * Sq
    g = torch.Generator(device="cuda").manual_seed(L + ld)
    xb, x = guarded(rows, L, ld, dt, 0x11)
    x.copy_((torch.randn(rows, L, generator=g, device=dev()) * 3).to(dt))
    dpb, dp = guarded(rows, L, ld, dt, 0x22)
    dp.copy_(torch.randn(rows, L, generator=g, device=dev()).to(dt))
    kw = dict(batch=B, heads=H, q_len=Sq)
    sink = None
    if masked:
        kw.update(causal=True, kv_valid_len=torch.tensor([L - 5, L // 2], dtype=torch.int32,
                                                         device=dev()),
                  key_mask=(torch.rand(B, L, generator=g, device=dev()) < 0.8).to(torch.uint8))
        sink = torch.randn(H, generator=g, device=dev())
    pb, p = guarded(rows, L, ld, dt, 0xA5)
    lb, lse = guarded_vec(rows, 0xA5)
    fos.fos_softmax_fwd(x, p, lse, sink=sink, **kw)
    dsb, ds = guarded(rows, L, ld, dt, 0x5A)
    db, delta = guarded_vec(rows, 0x5A)
    fos.fos_softmax_bwd(p, dp, ds, delta, **kw)
    torch.cuda.synchronize()
    assert untouched(pb, rows, L, ld, 0xA5), "forward wrote outside P"
    assert vec_untouched(lb, rows, 0xA5), "forward wrote outside LSE"
    assert untouched(dsb, rows, L, ld, 0x5A), "backward wrote outside dScores"
    assert vec_untouched(db, rows, 0x5A), "backward wrote outside delta"
    assert untouched(xb, rows, L, ld, 0x11) and untouched(dpb, rows, L, ld, 0x22)
    assert torch.isfinite(lse).all() or masked
    if sink is not None:
        sb, d_sink = guarded_vec(H, 0x3C)
        fos.fos_sink_grad(lse, delta, sink, d_sink, batch=B, heads=H, q_len=Sq)
        torch.cuda.synchronize()
        assert vec_untouched(sb, H, 0x3C), "sink gradient wrote outside d_sink"

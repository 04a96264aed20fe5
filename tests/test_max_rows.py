"""Problems of more than 2^31 rows: row indices then no longer fit 32 bits, and the kernels take
their 64-bit row-geometry path (row -> batch entry, head, query position by 64-bit division) and
64-bit addressing.  A causal bf16 problem of 2,148,007,936 rows of 8 keys with valid lengths
(about 86 GB on the device): rows around 2^31 and at the end against the FP64 oracle, and their
bits against a small launch of the same rows (the same batch entry's valid length and query
positions), forward and backward."""

import numpy as np
import pytest
import torch

import deterministic_attention_softmax_gb300 as fos
import oracle
from gpu_util import bits_equal, check_bwd, check_fwd, dev, np64, valid_matrix

pytestmark = pytest.mark.gpu

B, H, SQ, L = 65536, 4097, 8, 8
ROWS = B * H * SQ  # 2,148,007,936 > 2^31 - 1


def values(r0, n, salt):
    """Deterministic bf16 values in [-5, 5) for rows r0 .. r0+n-1 (element index e of the whole
    problem gets (e * 7919 + salt) mod 1000, scaled; no product exceeds 2^47)."""
    e = torch.arange(r0 * L, (r0 + n) * L, dtype=torch.int64, device=dev())
    v = ((e * 7919 + salt) % 1000).to(torch.float32) / 100.0 - 5.0
    return v.to(torch.bfloat16).view(n, L)


def fill(buf, salt):
    rows_per_chunk = 1 << 26
    for r0 in range(0, ROWS, rows_per_chunk):
        n = min(rows_per_chunk, ROWS - r0)
        buf[r0:r0 + n].copy_(values(r0, n, salt))


def test_more_than_2_31_rows():
    free, _ = torch.cuda.mem_get_info()
    if free < 100 * (1 << 30):
        pytest.skip("needs about 100 GB of free device memory")
    g = torch.Generator(device="cpu").manual_seed(3)
    kv_h = torch.randint(0, L + 1, (B,), generator=g, dtype=torch.int32)
    kv_h[-1] = L
    kv_h[(1 << 31) // (H * SQ)] = L - 3
    kv = kv_h.to(dev())
    kvn = kv_h.numpy()
    geo = dict(batch=B, heads=H, q_len=SQ, causal=True, kv_valid_len=kv)

    # sampled rows: the 8-row blocks around 2^31 and the last block
    base = (1 << 31) // SQ * SQ
    ids = np.concatenate([np.arange(base - 2 * SQ, base + 2 * SQ), np.arange(ROWS - SQ, ROWS)])
    ids_t = torch.from_numpy(ids).to(dev())
    okw = dict(batch=B, heads=H, q_len=SQ, causal=True, kv_valid_len=kvn, row_ids=ids)

    x = torch.empty(ROWS, L, dtype=torch.bfloat16, device=dev())
    fill(x, 17)
    p = torch.empty_like(x)
    lse = torch.empty(ROWS, dtype=torch.float32, device=dev())
    fos.fos_softmax_fwd(x, p, lse, **geo)
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
    x_s = x.index_select(0, ids_t)
    p_s, lse_s = p.index_select(0, ids_t), lse.index_select(0, ids_t)
    p_ref, lse_ref = oracle.softmax_fwd(np64(x_s), **okw)
    check_fwd(p_s, lse_s, p_ref, lse_ref, "bfloat16", "rows past 2^31")

    # backward in place of the scores: the sampled rows' P replaced by the oracle's P rounded
    # to bf16, dP drawn like the scores, dScores written over dP
    p_in_s = torch.from_numpy(p_ref).to(torch.bfloat16).to(dev())
    p.index_copy_(0, ids_t, p_in_s)
    dp = x
    del x
    fill(dp, 91)
    dp_s = dp.index_select(0, ids_t)
    delta = torch.empty(ROWS, dtype=torch.float32, device=dev())
    fos.fos_softmax_bwd(p, dp, dp, delta, **geo)
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
    ds_s, delta_s = dp.index_select(0, ids_t), delta.index_select(0, ids_t)
    pin, dpn = np64(p_in_s), np64(dp_s)
    ds_ref, delta_ref = oracle.softmax_bwd(pin, dpn, **okw)
    valid = valid_matrix(ids, L, B, H, SQ, True, kvn, None)
    check_bwd(ds_s, delta_s, ds_ref, delta_ref, pin, dpn, "bfloat16", valid=valid,
              what="rows past 2^31")
    del p, dp, lse, delta
    torch.cuda.empty_cache()

    # the same blocks as small launches (one batch entry, one head): the same bits
    for blk in range(0, len(ids), SQ):
        r0 = int(ids[blk])
        b = r0 // (H * SQ)
        sl = slice(blk, blk + SQ)
        small = dict(batch=1, heads=1, q_len=SQ, causal=True, kv_valid_len=kv[b:b + 1])
        ps, ls = fos.fos_softmax_fwd(values(r0, SQ, 17), **small)
        dss, dls = fos.fos_softmax_bwd(p_in_s[sl], dp_s[sl], **small)
        torch.cuda.synchronize()
        assert bits_equal(ps, p_s[sl]) and bits_equal(ls, lse_s[sl]), f"forward block at {r0}"
        assert bits_equal(dss, ds_s[sl]) and bits_equal(dls, delta_s[sl]), \
            f"backward block at {r0}"
    assert bits_equal(x_s, torch.cat([values(int(ids[k]), SQ, 17)
                                      for k in range(0, len(ids), SQ)]))

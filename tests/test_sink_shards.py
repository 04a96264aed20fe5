"""The sink gradient with rows sharded by batch entry, as ranks that each hold some batch
entries would run it: every shard runs the forward and backward on its own rows, writes the
chunk partials of its entries (fos_sink_grad_partials), and the partials of all shards,
concatenated in shard order and merged on the host (fos_sink_grad_merge), must give the bits of
fos_sink_grad on the whole batch.  The shards run one after another on one GPU."""

import pytest
import torch

import deterministic_attention_softmax_gb300 as fos
from deterministic_attention_softmax_gb300.shard import batch_shards
from gpu_util import bits_equal, dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,Sq,L,parts", [
    (4, 3, 384, 512, 2),   # shards of 2 batch entries (768 positions each)
    (4, 3, 384, 512, 3),   # some shards empty
    (6, 5, 256, 300, 4),   # one chunk per batch entry
    (7, 2, 64, 200, 3),    # four entries per chunk; a partial last chunk
])
def test_shards_give_the_whole_batch_bits(B, H, Sq, L, parts):
    g = torch.Generator().manual_seed(B * 100 + Sq)
    rows = B * H * Sq
    x = (torch.randn(rows, L, generator=g) * 3).to(torch.bfloat16).to(dev())
    dp = torch.randn(rows, L, generator=g).to(torch.bfloat16).to(dev())
    kv = torch.randint(L // 2, L + 1, (B,), generator=g, dtype=torch.int32).to(dev())
    sink = torch.randn(H, generator=g)
    sink[H - 1] = float("-inf")  # a head without a sink gets 0
    sink = sink.to(dev())
    geo = dict(batch=B, heads=H, q_len=Sq, causal=Sq <= L)

    p, lse = fos.fos_softmax_fwd(x, sink=sink, kv_valid_len=kv, **geo)
    ds, delta = fos.fos_softmax_bwd(p, dp, kv_valid_len=kv, **geo)
    ref = fos.fos_sink_grad(lse, delta, sink, batch=B, heads=H, q_len=Sq)

    cols = []
    for b0, b1 in batch_shards(B, Sq, parts):
        if b0 == b1:
            continue
        r0, r1 = b0 * H * Sq, b1 * H * Sq
        sgeo = dict(geo, batch=b1 - b0)
        sp, slse = fos.fos_softmax_fwd(x[r0:r1], sink=sink, kv_valid_len=kv[b0:b1], **sgeo)
        sds, sdelta = fos.fos_softmax_bwd(sp, dp[r0:r1], kv_valid_len=kv[b0:b1], **sgeo)
        assert bits_equal(slse, lse[r0:r1]) and bits_equal(sdelta, delta[r0:r1])
        part = fos.fos_sink_grad_partials(slse, sdelta, sink, batch=B, heads=H, q_len=Sq,
                                          batch_begin=b0, batch_end=b1)
        c0, c1 = fos.sink_chunk_range(Sq, b0, b1)
        assert part.shape == (H, c1 - c0)
        cols.append(part.cpu())
    merged = fos.fos_sink_grad_merge(torch.cat(cols, dim=1))
    assert bits_equal(merged, ref.cpu())
    assert float(merged[H - 1]) == 0.0
    assert fos.fos_device_error() == 0


def test_a_shard_off_the_chunk_grid_is_refused():
    B, H, Sq = 4, 2, 384
    lse = torch.zeros(3 * H * Sq, device=dev())
    delta = torch.zeros_like(lse)
    sink = torch.zeros(H, device=dev())
    with pytest.raises(fos.FosError) as e:  # starts at position 384
        fos.fos_sink_grad_partials(lse, delta, sink, batch=B, heads=H, q_len=Sq,
                                   batch_begin=1, batch_end=4)
    assert e.value.status == 1

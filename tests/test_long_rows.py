"""Rows longer than a shared-memory stage: the streaming kernels read such a row twice, in
segments of max(16, 2 x compute warps) tiles.  Their rows are checked against the FP64 oracle
within the parity tolerances; on rows that also fit a stage, forcing the streaming kernels
(load_path 3) must give the bits of the staged kernels, masks and sink included; and what they
cannot take (unaligned rows, plain loads, tile statistics beyond shared memory) is refused before
any launch."""

import pytest
import torch

import deterministic_attention_softmax_gb300 as fos
from gpu_util import bits_equal, dev
from test_parity_small import make_case, run_and_check

pytestmark = pytest.mark.gpu

STREAM = fos.Launch(load_path=3)


@pytest.mark.parametrize("dtype_name,L", [("float32", 70000), ("bfloat16", 150000),
                                          ("float16", 150000), ("bfloat16", 300000)])
@pytest.mark.parametrize("mask", ["none", "all"])
def test_rows_longer_than_a_stage_match_the_oracle(dtype_name, L, mask):
    # past what one stage holds (about 57k fp32 / 113k bf16 keys forward, half that backward),
    # so the default launch takes the streaming kernels
    c = make_case({"float32": torch.float32, "bfloat16": torch.bfloat16,
                   "float16": torch.float16}[dtype_name], L, mask, B=2, H=1, Sq=2)
    run_and_check(dtype_name, c)


def both_paths(c, dtype, launch_a=None, launch_b=STREAM):
    kw = dict(batch=c["B"], heads=c["H"], q_len=c["Sq"], causal=c["causal"],
              kv_valid_len=c["kv"], key_mask=c["km"])
    outs = []
    for lc in (launch_a, launch_b):
        p, lse = fos.fos_softmax_fwd(c["x"], sink=c["sink"], launch=lc, **kw)
        ds, delta = fos.fos_softmax_bwd(p, c["dp"], launch=lc, **kw)
        outs.append((p, lse, ds, delta))
    torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("L", [8, 264, 4096, 4352, 9000, 40000])  # 16-byte rows (bulk copies)
@pytest.mark.parametrize("mask", ["none", "causal", "kvlen", "keymask", "sink", "all"])
def test_streaming_gives_the_staged_bits(L, mask):
    c = make_case(torch.bfloat16, L, mask, B=2, H=3, Sq=5, seed=4)
    (a, b) = both_paths(c, torch.bfloat16)
    for x, y, name in zip(a, b, ("P", "LSE", "dScores", "delta")):
        assert bits_equal(x, y), f"{name} L={L} mask={mask}"
    assert fos.fos_device_error() == 0


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16])
@pytest.mark.parametrize("warps,stages", [(0, 0), (3, 2), (8, 5), (16, 0)])
def test_streaming_bits_do_not_depend_on_its_geometry(dtype, warps, stages):
    c = make_case(dtype, 20000, "all", B=2, H=2, Sq=3, seed=9)
    (a, b) = both_paths(c, dtype, None, fos.Launch(load_path=3, warps_per_cta=warps, stages=stages))
    for x, y in zip(a, b):
        assert bits_equal(x, y)


@pytest.mark.parametrize("stages", [1, 2, 3, 4])
@pytest.mark.parametrize("extra", [-1, 0, 1, 5])
@pytest.mark.parametrize("warps", [8, 12])
def test_segments_through_the_ring_give_the_staged_bits(stages, extra, warps):
    # Rows of fewer, as many and more segments than the ring has stages (segments of 16 tiles
    # with 8 warps, 24 with 12; the last one ragged), with valid lengths that give the rows of
    # one launch different segment counts: the stage and phase of every segment, in both
    # passes, cycle through the ring across rows of different lengths
    nseg = max(1, stages + extra)
    seg_keys = 256 * max(16, 2 * warps)
    L = seg_keys * (nseg - 1) + 1000
    c = make_case(torch.bfloat16, L, "all", B=2, H=2, Sq=3, seed=nseg + 10 * warps)
    (a, b) = both_paths(c, torch.bfloat16, None,
                        fos.Launch(load_path=3, warps_per_cta=warps, stages=stages))
    for x, y, name in zip(a, b, ("P", "LSE", "dScores", "delta")):
        assert bits_equal(x, y), f"{name} L={L} stages={stages} warps={warps}"
    assert fos.fos_device_error() == 0


def test_what_streaming_cannot_take_is_refused():
    # unaligned rows: 300001 bf16 keys are not a multiple of 16 bytes
    x = torch.zeros(2, 300001, dtype=torch.bfloat16, device=dev())
    with pytest.raises(fos.FosError) as e:
        fos.fos_softmax_fwd(x)
    assert e.value.status == 2
    # plain loads cannot stream
    y = torch.zeros(2, 300000, dtype=torch.bfloat16, device=dev())
    with pytest.raises(fos.FosError) as e:
        fos.fos_softmax_fwd(y, launch=fos.Launch(load_path=2))
    assert e.value.status == 2
    # the tile statistics alone exceed shared memory: 6 M keys forward (12 bytes per tile),
    # 15 M keys backward (4 bytes per tile)
    z = torch.zeros(1, 6_000_000, dtype=torch.bfloat16, device=dev())
    with pytest.raises(fos.FosError) as e:
        fos.fos_softmax_fwd(z)
    assert e.value.status == 2
    z = torch.zeros(1, 15_000_000, dtype=torch.bfloat16, device=dev())
    with pytest.raises(fos.FosError) as e:
        fos.fos_softmax_bwd(z, z)
    assert e.value.status == 2
    assert fos.fos_device_error() == 0

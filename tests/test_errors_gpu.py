"""Error behaviour on the GPU: the bounded-wait path (a copy that is never issued, so the wait
runs out after a short limit and the kernel returns an error status instead of hanging), the
context staying usable afterwards, and host-side refusals with real tensors."""

import pytest
import torch

import deterministic_attention_softmax_gb300 as fos
from gpu_util import bits_equal, dev

pytestmark = pytest.mark.gpu

TIMEOUT = 4  # FOS_ERR_TIMEOUT


def inputs(dtype=torch.bfloat16, rows=600, L=2048):
    g = torch.Generator(device="cuda").manual_seed(3)
    x = (torch.randn(rows, L, generator=g, device=dev()) * 3).to(dtype)
    dp = torch.randn(rows, L, generator=g, device=dev()).to(dtype)
    return x, dp


# staged rows (one warp per row at 2048 keys), streamed segments, the CTA kernels that park
# e_j in tensor memory (generic at 2048 keys; specialised at 4352, where the forward takes the
# row-group kernel), and the forward's row groups several to a CTA (3072 keys)
PATHS = {"staged": (2048, dict(load_path=1)), "streamed": (2048, dict(load_path=3)),
         "cta": (2048, dict(load_path=1, generic=1)), "cta_fast": (4352, dict(load_path=1)),
         "groups": (3072, dict(load_path=1, groups_per_cta=4, stages=2))}


@pytest.mark.parametrize("which", ["fwd", "bwd"])
@pytest.mark.parametrize("path", list(PATHS))
def test_stalled_copy_times_out_and_context_survives(which, path):
    L, opts = PATHS[path]
    x, dp = inputs(L=L)
    ref_p, ref_lse = fos.fos_softmax_fwd(x)
    ref_ds, ref_delta = fos.fos_softmax_bwd(ref_p, dp)
    assert fos.fos_device_error() == 0
    if which == "bwd" and "groups_per_cta" in opts:
        opts = dict(load_path=1)  # the backward has no row groups
    stall = fos.Launch(test_stall=1, wait_timeout_ns=20_000_000, **opts)
    if which == "fwd":
        fos.fos_softmax_fwd(x, launch=stall)
    else:
        fos.fos_softmax_bwd(ref_p, dp, launch=stall)
    assert fos.fos_device_error() == TIMEOUT
    assert fos.fos_device_error() == 0  # the word is cleared once read
    # the context is still usable and gives the same bits as before
    p, lse = fos.fos_softmax_fwd(x)
    ds, delta = fos.fos_softmax_bwd(p, dp)
    assert fos.fos_device_error() == 0
    assert bits_equal(p, ref_p) and bits_equal(lse, ref_lse)
    assert bits_equal(ds, ref_ds) and bits_equal(delta, ref_delta)


def test_invalid_and_unsupported_through_the_binding():
    x, dp = inputs(rows=8, L=4)
    with pytest.raises(fos.FosError) as e:  # causal with more queries than keys
        fos.fos_softmax_fwd(x, batch=1, heads=1, q_len=8, causal=True)
    assert e.value.status == 1
    with pytest.raises(fos.FosError) as e:  # rows != batch * heads * q_len
        fos.fos_softmax_fwd(x, batch=3, heads=1, q_len=3)
    assert e.value.status == 1
    buf = torch.zeros(8 * 64 + 1, dtype=torch.bfloat16, device=dev())
    xm = buf[1:].view(8, 64)  # 2-byte offset: bulk copies cannot be used
    with pytest.raises(fos.FosError) as e:
        fos.fos_softmax_fwd(xm, launch=fos.Launch(load_path=1))
    assert e.value.status == 2
    p, _ = fos.fos_softmax_fwd(xm, launch=fos.Launch(load_path=2))  # plain loads are fine
    assert torch.allclose(p.float(), torch.full_like(p.float(), 1 / 64))
    with pytest.raises(fos.FosError) as e:  # more stages than shared memory holds
        fos.fos_softmax_bwd(*inputs(rows=4, L=50000), launch=fos.Launch(stages=16))
    assert e.value.status == 2

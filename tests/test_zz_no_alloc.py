"""The host-buffer step for callers that may not allocate device memory
(fos_softmax_step_host_static: its scratch is a fixed 32 MB array inside the library).

Two calls in a row through the C ABI, on one stream and without a synchronisation between
them, must each give what the workspace-taking entry point (fos_softmax_step_host) gives for
the same inputs: the same bits, which is tighter than the oracle tolerance of the parity tests.
Between the two, a call of another dtype and row length fills the array with other bytes, so
the second call also shows that nothing in the array has to start at zero.
Problems whose scratch would not fit are refused with FOS_ERR_UNSUPPORTED before anything is
enqueued.  This file is collected last, and it builds the library itself so that it also runs
alone in a fresh process."""

import ctypes

import pytest
import torch

import deterministic_attention_softmax_gb300 as fos
from deterministic_attention_softmax_gb300 import _abi

pytestmark = pytest.mark.gpu

B, H, SQ, L = 2, 4, 1024, 1024  # 8192 rows of 2 KB: more than one chunk of the 32 MB array


@pytest.fixture(scope="module")
def lib():
    fos.build()
    return _abi.lib()


def host_inputs(seed):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(B * H * SQ, L, generator=g) * 3).to(torch.bfloat16).pin_memory()
    dp = torch.randn(B * H * SQ, L, generator=g).to(torch.bfloat16).pin_memory()
    return x, dp


def host_outputs():
    rows = B * H * SQ
    return dict(p=torch.empty(rows, L, dtype=torch.bfloat16).pin_memory(),
                lse=torch.empty(rows, dtype=torch.float32).pin_memory(),
                ds=torch.empty(rows, L, dtype=torch.bfloat16).pin_memory(),
                delta=torch.empty(rows, dtype=torch.float32).pin_memory(),
                d_sink=torch.empty(H, dtype=torch.float32).pin_memory())


def ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def bits(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32)


def test_two_calls_in_a_row_match_the_workspace_entry_point(lib):
    dev = torch.device("cuda", 0)
    kv = torch.tensor([1000, 777], dtype=torch.int32, device=dev)
    sink = torch.randn(H, generator=torch.Generator().manual_seed(9)).to(dev)
    desc = _abi.FosDesc(B * H * SQ, L, L, B, H, SQ, 1, 0, kv.data_ptr(), None, sink.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    ins = [host_inputs(seed) for seed in (1, 2)]
    outs = [host_outputs() for _ in ins]
    # the call in between: float32 rows of 3000 keys, another chunk layout in the array
    rows_f, L_f = 1536, 3000
    g = torch.Generator().manual_seed(4)
    xf = (torch.randn(rows_f, L_f, generator=g) * 4).pin_memory()
    dpf = torch.randn(rows_f, L_f, generator=g).pin_memory()
    of = dict(p=torch.empty_like(xf).pin_memory(), ds=torch.empty_like(xf).pin_memory(),
              lse=torch.empty(rows_f).pin_memory(), delta=torch.empty(rows_f).pin_memory())
    desc_f = _abi.FosDesc(rows_f, L_f, L_f, 1, 1, rows_f, 0, 0, None, None, None)
    calls = [(desc, _abi.FOS_BF16, ins[0], outs[0]), (desc_f, _abi.FOS_F32, (xf, dpf), of),
             (desc, _abi.FOS_BF16, ins[1], outs[1])]
    for d, dt, (x, dp), o in calls:  # back to back on one stream
        st = lib.fos_softmax_step_host_static(
            ctypes.byref(d), dt, ptr(x), ptr(dp), ptr(o["p"]), ptr(o["lse"]), ptr(o["ds"]),
            ptr(o["delta"]), ptr(o["d_sink"]) if "d_sink" in o else None, 0, stream, None)
        assert st == _abi.FOS_OK, lib.fos_status_string(st)
    torch.cuda.synchronize()
    ref_f = fos.fos_softmax_step_host(xf, dpf, batch=1, heads=1, q_len=rows_f)
    torch.cuda.synchronize()
    for got, want in zip((of["p"], of["lse"], of["ds"], of["delta"]), ref_f):
        assert torch.equal(bits(got), bits(want))
    geo = dict(batch=B, heads=H, q_len=SQ, causal=True, kv_valid_len=kv)
    for (x, dp), o in zip(ins, outs):
        ref = fos.fos_softmax_step_host(x, dp, sink=sink, **geo)
        torch.cuda.synchronize()
        for got, want in zip((o["p"], o["lse"], o["ds"], o["delta"], o["d_sink"]), ref):
            assert torch.equal(bits(got), bits(want))
    assert fos.fos_device_error() == 0


def test_a_given_chunk_and_refusals(lib):
    dev = torch.device("cuda", 0)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    x, dp = host_inputs(3)
    o = host_outputs()
    desc = _abi.FosDesc(B * H * SQ, L, L, 1, 1, B * H * SQ, 0, 0, None, None, None)

    def call(d, chunk, x=x, dp=dp):
        return lib.fos_softmax_step_host_static(
            ctypes.byref(d), _abi.FOS_BF16, ptr(x), ptr(dp), ptr(o["p"]), ptr(o["lse"]),
            ptr(o["ds"]), ptr(o["delta"]), None, chunk, stream, None)

    assert call(desc, 700) == _abi.FOS_OK
    torch.cuda.synchronize()
    ref = fos.fos_softmax_step_host(x, dp, batch=1, heads=1, q_len=B * H * SQ)
    torch.cuda.synchronize()
    assert torch.equal(bits(o["p"]), bits(ref[0])) and torch.equal(bits(o["ds"]), bits(ref[2]))
    # a chunk whose six tensors exceed the array
    assert call(desc, B * H * SQ) == _abi.FOS_ERR_UNSUPPORTED
    # one row of 3 M keys: six one-row tensors exceed the array
    one = _abi.FosDesc(1, 3_000_000, 3_000_000, 1, 1, 1, 0, 0, None, None, None)
    assert call(one, 0) == _abi.FOS_ERR_UNSUPPORTED
    # 5 M rows: LSE and delta alone exceed the array
    many = _abi.FosDesc(5_000_000, 8, 8, 1, 1, 5_000_000, 0, 0, None, None, None)
    assert call(many, 0) == _abi.FOS_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0

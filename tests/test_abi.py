"""The C-ABI library: it builds, loads, exports every symbol the header declares, and its host
argument checks reject bad calls before touching CUDA (no GPU needed, no kernel launched)."""

import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "fos_softmax.h")


@pytest.fixture(scope="module")
def abi():
    import deterministic_attention_softmax_gb300 as fos
    from deterministic_attention_softmax_gb300 import _abi

    fos.build()
    return _abi


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(fos_[a-z_]+)\s*\(", text))


def test_header_declares_the_binding_names(abi):
    assert declared_functions() == set(abi.EXPORTED)


def test_library_exports_every_declared_symbol(abi):
    lib = abi.lib()
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} is declared but not exported"


def test_struct_layout_matches_the_header(abi):
    # fos_desc: 2 x int64, 6 x int32, 3 pointers; fos_launch: 4 x int32, int64, 4 x int32
    assert ctypes.sizeof(abi.FosDesc) == 64
    assert abi.FosDesc.kv_valid_len.offset == 40
    assert ctypes.sizeof(abi.FosLaunch) == 40
    assert abi.FosLaunch.wait_timeout_ns.offset == 16
    assert abi.FosLaunch.groups_per_cta.offset == 32
    assert abi.FosLaunch.sink_fusion.offset == 36


def test_contraction_descriptors_match_the_header(abi):
    # fos_pv_desc: 6 x int32, int64, float (padded to 8 bytes)
    assert abi.FosPvDesc.ld_probs.offset == 24
    assert abi.FosPvDesc.scale.offset == 32
    assert ctypes.sizeof(abi.FosPvDesc) == 40


def _pv(abi, **kw):
    d = dict(batch=1, q_heads=2, kv_heads=1, q_len=8, kv_len=16, head_dim=64, ld_probs=16,
             scale=1.0)
    d.update(kw)
    return abi.FosPvDesc(**d)


@pytest.mark.parametrize("bad", [
    dict(scale=0.0), dict(scale=float("inf")), dict(scale=float("nan")),  # scale finite, nonzero
    dict(q_heads=3, kv_heads=2),                                         # not a multiple of kv_heads
    dict(kv_heads=0), dict(ld_probs=15), dict(batch=-1), dict(q_len=-1),
])
def test_contractions_reject_bad_descriptors(abi, bad):
    lib = abi.lib()
    d = _pv(abi, **bad)
    assert lib.fos_pv_out(ctypes.byref(d), abi.FOS_BF16, abi.FOS_F32, FAKE, FAKE, FAKE,
                          None) == abi.FOS_ERR_INVALID
    assert lib.fos_grad_kv(ctypes.byref(d), abi.FOS_BF16, abi.FOS_F32, FAKE, FAKE, FAKE,
                           None) == abi.FOS_ERR_INVALID


def test_contractions_reject_bad_dtypes_and_pointers(abi):
    lib = abi.lib()
    d = _pv(abi)
    # 16-bit inputs only; outputs float32, bf16 or fp16
    assert lib.fos_grad_kv(ctypes.byref(d), abi.FOS_F32, abi.FOS_F32, FAKE, FAKE, FAKE,
                           None) == abi.FOS_ERR_INVALID
    assert lib.fos_grad_kv(ctypes.byref(d), abi.FOS_BF16, 7, FAKE, FAKE, FAKE,
                           None) == abi.FOS_ERR_INVALID
    assert lib.fos_grad_kv(None, abi.FOS_BF16, abi.FOS_F32, FAKE, FAKE, FAKE,
                           None) == abi.FOS_ERR_INVALID
    assert lib.fos_grad_kv(ctypes.byref(d), abi.FOS_BF16, abi.FOS_F32, None, FAKE, FAKE,
                           None) == abi.FOS_ERR_INVALID
    assert lib.fos_grad_kv(ctypes.byref(d), abi.FOS_BF16, abi.FOS_F32, FAKE, FAKE, None,
                           None) == abi.FOS_ERR_INVALID
    # another head dimension is valid but unsupported
    d96 = _pv(abi, head_dim=96)
    assert lib.fos_grad_kv(ctypes.byref(d96), abi.FOS_BF16, abi.FOS_F32, FAKE, FAKE, FAKE,
                           None) == abi.FOS_ERR_UNSUPPORTED
    # no output: a no-op, even with null pointers
    d0 = _pv(abi, kv_len=0, ld_probs=0)
    assert lib.fos_grad_kv(ctypes.byref(d0), abi.FOS_BF16, abi.FOS_F32, None, None, None,
                           None) == abi.FOS_OK


def test_status_strings_and_fingerprint(abi):
    lib = abi.lib()
    for code, name in abi.STATUS_NAMES.items():
        assert lib.fos_status_string(code).decode().startswith(name)
    fp = lib.fos_contract_fingerprint().decode()
    for part in ("TILE_K=256", "xor tree 16,8,4,2,1", "sm_103a", "no atomics", "no fast-math"):
        assert part in fp


def _desc(abi, **kw):
    d = dict(rows=6, ld=8, key_len=8, batch=1, heads=2, q_len=3, causal=0, reserved=0,
             kv_valid_len=None, key_mask=None, sink=None)
    d.update(kw)
    return abi.FosDesc(**d)


FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: every case below fails validation first


@pytest.mark.parametrize("bad", [
    dict(rows=7),                    # rows != batch*heads*q_len
    dict(key_len=0, ld=0),           # no keys
    dict(ld=7),                      # ld < key_len
    dict(causal=2),
    dict(causal=1, q_len=9, rows=18, key_len=8),  # causal needs q_len <= key_len
    dict(reserved=1),
    dict(batch=-1, rows=-6),
])
def test_fwd_rejects_bad_descriptors(abi, bad):
    d = _desc(abi, **bad)
    st = abi.lib().fos_softmax_fwd(ctypes.byref(d), abi.FOS_BF16, FAKE, FAKE, FAKE, None, None)
    assert st == abi.FOS_ERR_INVALID


def test_rejects_null_pointers_and_bad_dtype(abi):
    lib = abi.lib()
    d = _desc(abi)
    assert lib.fos_softmax_fwd(None, abi.FOS_BF16, FAKE, FAKE, FAKE, None, None) == abi.FOS_ERR_INVALID
    assert lib.fos_softmax_fwd(ctypes.byref(d), 7, FAKE, FAKE, FAKE, None, None) == abi.FOS_ERR_INVALID
    assert lib.fos_softmax_fwd(ctypes.byref(d), abi.FOS_F32, None, FAKE, FAKE, None, None) == abi.FOS_ERR_INVALID
    assert lib.fos_softmax_fwd(ctypes.byref(d), abi.FOS_F32, FAKE, FAKE, None, None, None) == abi.FOS_ERR_INVALID
    assert lib.fos_softmax_bwd(ctypes.byref(d), abi.FOS_F32, FAKE, None, FAKE, None, None, None) == abi.FOS_ERR_INVALID
    # the sink gradient needs a sink (a null sink with a sink operation is an error, not a no-op)
    assert lib.fos_sink_grad(ctypes.byref(d), FAKE, FAKE, FAKE, None, None) == abi.FOS_ERR_INVALID


@pytest.mark.parametrize("bad", [
    dict(warps_per_cta=17), dict(warps_per_cta=-1), dict(ctas=-2), dict(stages=17),
    dict(load_path=4), dict(wait_timeout_ns=-5), dict(test_stall=2), dict(generic=2),
    dict(groups_per_cta=-1), dict(groups_per_cta=16), dict(sink_fusion=-1), dict(sink_fusion=3),
])
def test_rejects_bad_launch_options(abi, bad):
    opts = dict(warps_per_cta=0, ctas=0, stages=0, load_path=0, wait_timeout_ns=0, test_stall=0,
                generic=0, groups_per_cta=0, sink_fusion=0)
    opts.update(bad)
    lc = abi.FosLaunch(**opts)
    d = _desc(abi)
    st = abi.lib().fos_softmax_fwd(ctypes.byref(d), abi.FOS_BF16, FAKE, FAKE, FAKE, None,
                                   ctypes.byref(lc))
    assert st == abi.FOS_ERR_INVALID


def test_zero_rows_is_ok_and_launches_nothing(abi):
    d = _desc(abi, rows=0, batch=0)
    st = abi.lib().fos_softmax_fwd(ctypes.byref(d), abi.FOS_BF16, FAKE, FAKE, FAKE, None, None)
    assert st == abi.FOS_OK
    st = abi.lib().fos_softmax_bwd(ctypes.byref(d), abi.FOS_BF16, FAKE, FAKE, FAKE, None, None, None)
    assert st == abi.FOS_OK
    # empty tensors may have null data pointers
    st = abi.lib().fos_softmax_fwd(ctypes.byref(d), abi.FOS_BF16, None, None, None, None, None)
    assert st == abi.FOS_OK


def test_binding_refuses_cpu_tensors():
    import torch

    import deterministic_attention_softmax_gb300 as fos

    fos.build()
    with pytest.raises(ValueError):
        fos.fos_softmax_fwd(torch.zeros(4, 8))


def test_step_host_workspace_bytes(abi):
    lib = abi.lib()
    d = _desc(abi)  # 6 rows x 8 keys, 2 heads
    # LSE, delta and d_sink (256-byte aligned each), then 3 slots x 2 chunk tensors
    assert lib.fos_step_host_workspace_bytes(ctypes.byref(d), abi.FOS_BF16, 0) == 3 * 256 + 6 * 256
    big = _desc(abi, rows=4096, batch=1, heads=1, q_len=4096, ld=1000, key_len=1000)
    chunk = 100  # 100 rows of 2000 bytes -> 200,192 bytes per tensor after alignment
    t = -(-100 * 1000 * 2 // 256) * 256
    assert lib.fos_step_host_workspace_bytes(ctypes.byref(big), abi.FOS_BF16, chunk) == \
        2 * 16384 + 256 + 6 * t
    # the default chunk is about 16 MB of one tensor, capped at the row count
    assert lib.fos_step_host_workspace_bytes(ctypes.byref(big), abi.FOS_F32, 0) == \
        2 * 16384 + 256 + 6 * (4096 * 4000)
    for bad in (dict(rows=7), dict(ld=7)):
        assert lib.fos_step_host_workspace_bytes(ctypes.byref(_desc(abi, **bad)), abi.FOS_BF16, 0) == 0
    assert lib.fos_step_host_workspace_bytes(ctypes.byref(d), 9, 0) == 0
    assert lib.fos_step_host_workspace_bytes(ctypes.byref(d), abi.FOS_BF16, -1) == 0
    assert lib.fos_step_host_workspace_bytes(ctypes.byref(_desc(abi, rows=0, batch=0)),
                                             abi.FOS_BF16, 0) == 0


def test_step_host_refuses_before_any_cuda_call(abi):
    lib = abi.lib()
    d = _desc(abi)
    need = lib.fos_step_host_workspace_bytes(ctypes.byref(d), abi.FOS_BF16, 0)
    ws = ctypes.c_void_p(0x10000)  # 256-byte aligned, never dereferenced
    call = lambda dd, ws_, n, chunk=0, dsink=None: lib.fos_softmax_step_host(
        ctypes.byref(dd), abi.FOS_BF16, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, dsink, ws_, n, chunk,
        None, None)
    assert call(d, ws, need - 1) == abi.FOS_ERR_INVALID          # workspace too small
    assert call(d, ctypes.c_void_p(0x10010), need) == abi.FOS_ERR_INVALID  # misaligned
    assert call(d, None, need) == abi.FOS_ERR_INVALID            # no workspace
    assert call(d, ws, need, chunk=-3) == abi.FOS_ERR_INVALID
    assert call(d, ws, need, dsink=FAKE) == abi.FOS_ERR_INVALID  # d_sink without a sink
    assert call(_desc(abi, rows=7), ws, need) == abi.FOS_ERR_INVALID
    assert call(_desc(abi, rows=0, batch=0), None, 0) == abi.FOS_OK  # empty: nothing enqueued


def test_sink_grad_merge_adds_left_to_right_in_float32(abi):
    import numpy as np

    rng = np.random.default_rng(5)
    parts = (rng.standard_normal((3, 37)) * 10.0 ** rng.integers(-6, 6, (3, 37))).astype(np.float32)
    out = np.empty(3, dtype=np.float32)
    st = abi.lib().fos_sink_grad_merge(3, 37, parts.ctypes.data_as(ctypes.c_void_p),
                                       out.ctypes.data_as(ctypes.c_void_p))
    assert st == abi.FOS_OK
    for h in range(3):  # the same additions, one float32 rounding each
        t = np.float32(0.0)
        for c in range(37):
            t = np.float32(t + parts[h, c])
        assert out[h].tobytes() == t.tobytes()
    lib = abi.lib()
    assert lib.fos_sink_grad_merge(-1, 3, None, None) == abi.FOS_ERR_INVALID
    assert lib.fos_sink_grad_merge(2, 3, None, out.ctypes.data_as(ctypes.c_void_p)) == abi.FOS_ERR_INVALID
    assert lib.fos_sink_grad_merge(0, 3, None, None) == abi.FOS_OK
    zero = np.full(2, 7.0, dtype=np.float32)  # no chunks: d_sink = +0
    assert lib.fos_sink_grad_merge(2, 0, None, zero.ctypes.data_as(ctypes.c_void_p)) == abi.FOS_OK
    assert zero.tobytes() == np.zeros(2, dtype=np.float32).tobytes()


@pytest.mark.parametrize("b0,b1", [
    (1, 4),    # starts at position 384: not on the 256 grid
    (0, 1),    # ends at 384 and is not the last shard
    (2, 1), (0, 5), (-1, 2),
])
def test_sink_grad_partials_refuses_misaligned_or_bad_shards(abi, b0, b1):
    # refused before any CUDA call (never run a valid shard with these fake pointers)
    d = _desc(abi, rows=4 * 3 * 384, batch=4, heads=3, q_len=384, ld=512, key_len=512, sink=FAKE)
    st = abi.lib().fos_sink_grad_partials(ctypes.byref(d), b0, b1, FAKE, FAKE, FAKE, None, None)
    assert st == abi.FOS_ERR_INVALID


def test_sink_grad_partials_empty_shard_and_missing_sink(abi):
    lib = abi.lib()
    d = _desc(abi, rows=4 * 3 * 384, batch=4, heads=3, q_len=384, ld=512, key_len=512, sink=FAKE)
    assert lib.fos_sink_grad_partials(ctypes.byref(d), 3, 3, FAKE, FAKE, FAKE, None, None) == abi.FOS_OK
    nosink = _desc(abi, rows=4 * 3 * 384, batch=4, heads=3, q_len=384, ld=512, key_len=512)
    assert lib.fos_sink_grad_partials(ctypes.byref(nosink), 0, 2, FAKE, FAKE, FAKE, None,
                                      None) == abi.FOS_ERR_INVALID


def test_batch_shards_start_on_the_chunk_grid():
    from deterministic_attention_softmax_gb300.shard import batch_shards

    for batch, q_len, parts in ((4, 384, 2), (4, 384, 3), (2, 2048, 2), (7, 100, 3), (64, 257, 4),
                                (1, 16384, 2), (9, 256, 4)):
        sh = batch_shards(batch, q_len, parts)
        assert len(sh) == parts and sh[0][0] == 0 and sh[-1][1] == batch
        for (a, b), (c, _) in zip(sh, sh[1:]):
            assert b == c and a <= b
        for a, b in sh:
            assert a == b or (a * q_len) % 256 == 0

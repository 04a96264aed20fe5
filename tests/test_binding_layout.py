"""The binding's host-side marshalling, on the CPU: how a tensor's shape and strides become
(rows, key_len, ld), how the [batch][heads][q_len] geometry is inferred, and which mask / sink
tensors the descriptor refuses.  These decide which rows and stride the kernels see; no CUDA
call is made."""

import pytest
import torch

from deterministic_attention_softmax_gb300 import binding


def test_two_dimensional_rows():
    x = torch.zeros(12, 300)
    assert binding._rows_layout(x, "x") == (12, 300, 300)


def test_narrowed_view_keeps_the_buffer_stride():
    buf = torch.zeros(12, 320)
    assert binding._rows_layout(buf[:, :300], "x") == (12, 300, 320)
    assert binding._rows_layout(buf[3:9, 5:300], "x") == (6, 295, 320)


def test_four_dimensional_rows_and_inferred_geometry():
    x = torch.zeros(2, 3, 5, 64)
    assert binding._rows_layout(x, "x") == (30, 64, 64)
    assert binding._geometry(x, None, None, None) == (30, 64, 64, 2, 3, 5)
    # explicit geometry wins; q_len defaults to rows / (batch * heads)
    assert binding._geometry(x, 6, 1, None) == (30, 64, 64, 6, 1, 5)
    assert binding._geometry(x.view(30, 64), 2, 3, None) == (30, 64, 64, 2, 3, 5)


def test_four_dimensional_view_of_a_padded_buffer():
    buf = torch.zeros(2, 3, 5, 72)
    x = buf[..., :64]
    assert binding._rows_layout(x, "x") == (30, 64, 72)


def test_every_other_row_is_a_uniform_stride():
    assert binding._rows_layout(torch.zeros(2, 10, 64)[:, ::2], "x") == (10, 64, 128)


def test_single_row_and_broadcast_free_dims():
    assert binding._rows_layout(torch.zeros(1, 100), "x") == (1, 100, 100)
    assert binding._rows_layout(torch.zeros(1, 1, 7, 16), "x") == (7, 16, 16)


@pytest.mark.parametrize("make", [
    lambda: torch.zeros(300),                                   # no row dimension
    lambda: torch.zeros(300, 12).t(),                           # keys not contiguous
    lambda: torch.zeros(3, 2, 5, 64).permute(1, 0, 2, 3),       # heads before batch in memory
    lambda: torch.zeros(2, 6, 64)[:, :5],                       # batch stride != 5 rows
])
def test_layouts_that_do_not_collapse_to_rows_are_refused(make):
    with pytest.raises(ValueError):
        binding._rows_layout(make(), "x")


def desc(**kw):
    base = dict(rows=6, L=8, ld=8, batch=2, heads=3, q_len=1, causal=False, kv_valid_len=None,
                key_mask=None, sink=None)
    base.update(kw)
    return binding._desc(**base)


def test_descriptor_fields():
    kv = torch.tensor([3, 8], dtype=torch.int32)
    km = torch.ones(2, 8, dtype=torch.uint8)
    sink = torch.zeros(3)
    d = desc(causal=True, kv_valid_len=kv, key_mask=km, sink=sink)
    assert (d.rows, d.ld, d.key_len, d.batch, d.heads, d.q_len, d.causal, d.reserved) == \
        (6, 8, 8, 2, 3, 1, 1, 0)
    assert d.kv_valid_len == kv.data_ptr() and d.key_mask == km.data_ptr()
    assert d.sink == sink.data_ptr()
    assert desc().kv_valid_len is None and desc().sink is None


@pytest.mark.parametrize("kw", [
    dict(kv_valid_len=torch.tensor([3, 8], dtype=torch.int64)),       # not int32
    dict(kv_valid_len=torch.tensor([3, 8, 8], dtype=torch.int32)),    # not one per batch entry
    dict(kv_valid_len=torch.zeros(4, dtype=torch.int32)[::2]),        # not contiguous
    dict(key_mask=torch.ones(2, 7, dtype=torch.uint8)),               # not batch * key_len
    dict(key_mask=torch.ones(2, 8, dtype=torch.float32)),             # not uint8 / bool
    dict(sink=torch.zeros(3, dtype=torch.float64)),                   # not float32
    dict(sink=torch.zeros(4)),                                        # not one per head
])
def test_descriptor_refuses_bad_masks_and_sinks(kw):
    with pytest.raises(ValueError):
        desc(**kw)


def test_boolean_key_mask_is_accepted():
    km = torch.ones(2, 8, dtype=torch.bool)
    assert desc(key_mask=km).key_mask == km.data_ptr()

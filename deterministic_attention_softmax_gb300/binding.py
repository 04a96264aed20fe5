"""PyTorch-facing binding of the C ABI, with the same names as ``include/fos_softmax.h``.

Argument marshalling only: tensors are checked for device, dtype and layout, their device
pointers and the current CUDA stream are passed to ``libfos_softmax.so``, and a non-OK status
becomes a ``FosError``.  PyTorch provides device memory and streams; all arithmetic happens in
the library's CUDA kernels.

Row layout: ``scores`` (and P, dP, dScores) is a tensor whose last dimension holds the keys
(stride 1) and whose leading dimensions collapse to rows with one uniform row stride ``ld``
(``ld >= key_len``): a 2-D ``[rows, key_len]`` tensor, a narrowed view of a wider buffer, or a
``[batch, heads, q_len, key_len]`` tensor.  Rows are ordered ``[batch][heads][q_len]``.
"""

from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _abi

_DTYPES = {torch.float32: _abi.FOS_F32, torch.bfloat16: _abi.FOS_BF16,
           torch.float16: _abi.FOS_F16}


class FosError(RuntimeError):
    """A non-OK ``fos_status``; ``.status`` holds the code."""

    def __init__(self, status: int, where: str):
        self.status = int(status)
        msg = _abi.lib().fos_status_string(self.status).decode()
        super().__init__(f"{where}: {msg}")


@dataclass
class Launch:
    """Optional launch geometry (none of it changes a result bit); 0 means the default."""

    warps_per_cta: int = 0
    ctas: int = 0
    stages: int = 0
    load_path: int = 0  # 0 auto, 1 bulk copy (TMA) only, 2 plain loads only
    wait_timeout_ns: int = 0
    test_stall: int = 0
    generic: int = 0  # 1: never the kernel specialised for the common case
    groups_per_cta: int = 0  # forward row groups per CTA (0: chosen by the library)
    sink_fusion: int = 0  # fos_softmax_bwd_sink: 0 library's choice, 1 fuse where possible, 2 never

    def _c(self) -> _abi.FosLaunch:
        return _abi.FosLaunch(self.warps_per_cta, self.ctas, self.stages, self.load_path,
                              self.wait_timeout_ns, self.test_stall, self.generic,
                              self.groups_per_cta, self.sink_fusion)


def _rows_layout(t: torch.Tensor, name: str):
    """(rows, key_len, ld) of a row-major key tensor, or raise."""
    if t.dim() < 2:
        raise ValueError(f"{name} must have at least 2 dimensions (rows x keys)")
    if t.stride(-1) != 1 and t.shape[-1] > 1:
        raise ValueError(f"{name}: the key dimension must have stride 1")
    L = t.shape[-1]
    ld = t.stride(-2) if t.shape[-2] > 1 else max(L, t.stride(-2))
    rows = 1
    for d in t.shape[:-1]:
        rows *= d
    expect = ld
    for i in range(t.dim() - 2, -1, -1):
        if t.shape[i] > 1 and t.stride(i) != expect:
            raise ValueError(f"{name}: leading dimensions do not collapse to one row stride")
        expect *= t.shape[i]
    return rows, L, ld


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_cuda(t, name, device):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _geometry(x, batch, heads, q_len):
    rows, L, ld = _rows_layout(x, "scores")
    if x.dim() == 4 and batch is None and heads is None and q_len is None:
        batch, heads, q_len = x.shape[0], x.shape[1], x.shape[2]
    batch = 1 if batch is None else int(batch)
    heads = 1 if heads is None else int(heads)
    if q_len is None:
        q_len = rows // max(1, batch * heads)
    return rows, L, ld, batch, heads, int(q_len)


def _desc(rows, L, ld, batch, heads, q_len, causal, kv_valid_len, key_mask, sink):
    if kv_valid_len is not None and (kv_valid_len.dtype != torch.int32 or
                                     not kv_valid_len.is_contiguous()):
        raise ValueError("kv_valid_len must be a contiguous int32 tensor [batch]")
    if key_mask is not None:
        if key_mask.dtype not in (torch.uint8, torch.bool) or not key_mask.is_contiguous():
            raise ValueError("key_mask must be a contiguous uint8/bool tensor [batch, key_len]")
        if key_mask.numel() != batch * L:
            raise ValueError("key_mask must have batch * key_len entries")
    if sink is not None:
        if sink.dtype != torch.float32 or not sink.is_contiguous() or sink.numel() != heads:
            raise ValueError("sink must be a contiguous float32 tensor [heads]")
    if kv_valid_len is not None and kv_valid_len.numel() != batch:
        raise ValueError("kv_valid_len must have one entry per batch")
    return _abi.FosDesc(rows, ld, L, batch, heads, q_len, int(bool(causal)), 0,
                        None if kv_valid_len is None else kv_valid_len.data_ptr(),
                        None if key_mask is None else key_mask.data_ptr(),
                        None if sink is None else sink.data_ptr())


def _like(x):
    return torch.empty_strided(x.shape, x.stride(), dtype=x.dtype, device=x.device)


def _same_layout(a, b, na, nb):
    if a.shape != b.shape or a.stride() != b.stride() or a.dtype != b.dtype:
        raise ValueError(f"{nb} must have the shape, strides and dtype of {na}")


def fos_softmax_fwd(scores, probs=None, lse=None, *, batch=None, heads=None, q_len=None,
                    causal=False, kv_valid_len=None, key_mask=None, sink=None, stream=None,
                    launch: Launch | None = None):
    """Fixed-order softmax forward.  Returns ``(probs, lse)``; see ``fos_softmax_fwd`` in the
    C header for the arithmetic.  ``probs`` may be ``scores`` itself (in place)."""
    if scores.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {scores.dtype}")
    dev = scores.device
    rows, L, ld, batch, heads, q_len = _geometry(scores, batch, heads, q_len)
    if probs is None:
        probs = _like(scores)
    if lse is None:
        lse = torch.empty(rows, dtype=torch.float32, device=dev)
    _same_layout(scores, probs, "scores", "probs")
    if lse.dtype != torch.float32 or lse.numel() != rows or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 tensor with one entry per row")
    for t, n in ((scores, "scores"), (probs, "probs"), (lse, "lse"), (kv_valid_len, "kv_valid_len"),
                 (key_mask, "key_mask"), (sink, "sink")):
        _check_cuda(t, n, dev)
    d = _desc(rows, L, ld, batch, heads, q_len, causal, kv_valid_len, key_mask, sink)
    lc = None if launch is None else ctypes.byref(launch._c())
    with torch.cuda.device(dev):
        st = _abi.lib().fos_softmax_fwd(ctypes.byref(d), _DTYPES[scores.dtype], _ptr(scores),
                                        _ptr(probs), _ptr(lse), _stream_handle(stream, dev), lc)
    if st != _abi.FOS_OK:
        raise FosError(st, "fos_softmax_fwd")
    return probs, lse


def fos_softmax_bwd(probs, dprobs, dscores=None, delta=None, *, batch=None, heads=None,
                    q_len=None, causal=False, kv_valid_len=None, key_mask=None, stream=None,
                    want_delta=True, launch: Launch | None = None):
    """Softmax VJP on the given P.  Returns ``(dscores, delta)`` (delta is None when neither
    given nor wanted).  ``dscores`` may be ``dprobs`` itself (in place)."""
    if probs.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {probs.dtype}")
    dev = probs.device
    rows, L, ld, batch, heads, q_len = _geometry(probs, batch, heads, q_len)
    _same_layout(probs, dprobs, "probs", "dprobs")
    if dscores is None:
        dscores = _like(probs)
    _same_layout(probs, dscores, "probs", "dscores")
    if delta is None and want_delta:
        delta = torch.empty(rows, dtype=torch.float32, device=dev)
    if delta is not None and (delta.dtype != torch.float32 or delta.numel() != rows or
                              not delta.is_contiguous()):
        raise ValueError("delta must be a contiguous float32 tensor with one entry per row")
    for t, n in ((probs, "probs"), (dprobs, "dprobs"), (dscores, "dscores"), (delta, "delta"),
                 (kv_valid_len, "kv_valid_len"), (key_mask, "key_mask")):
        _check_cuda(t, n, dev)
    d = _desc(rows, L, ld, batch, heads, q_len, causal, kv_valid_len, key_mask, None)
    lc = None if launch is None else ctypes.byref(launch._c())
    with torch.cuda.device(dev):
        st = _abi.lib().fos_softmax_bwd(ctypes.byref(d), _DTYPES[probs.dtype], _ptr(probs),
                                        _ptr(dprobs), _ptr(dscores), _ptr(delta),
                                        _stream_handle(stream, dev), lc)
    if st != _abi.FOS_OK:
        raise FosError(st, "fos_softmax_bwd")
    return dscores, delta


def fos_softmax_bwd_sink(probs, dprobs, lse, sink, dscores=None, d_sink=None, delta=None, *,
                         batch=None, heads=None, q_len=None, causal=False, kv_valid_len=None,
                         key_mask=None, workspace=None, stream=None,
                         launch: Launch | None = None):
    """Backward and sink gradient in one call (the sink gradient taken along by the backward
    where its kernels allow, otherwise the two launches; the same bits either way).  Returns
    ``(dscores, d_sink, delta)``; delta is written only when given."""
    if probs.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {probs.dtype}")
    dev = probs.device
    rows, L, ld, batch, heads, q_len = _geometry(probs, batch, heads, q_len)
    _same_layout(probs, dprobs, "probs", "dprobs")
    if dscores is None:
        dscores = _like(probs)
    _same_layout(probs, dscores, "probs", "dscores")
    for t, n in ((lse, "lse"), (delta, "delta")):
        if t is not None and (t.dtype != torch.float32 or t.numel() != rows or
                              not t.is_contiguous()):
            raise ValueError(f"{n} must be a contiguous float32 tensor with one entry per row")
    if sink is None:
        raise ValueError("sink is required")
    if d_sink is None:
        d_sink = torch.empty(heads, dtype=torch.float32, device=dev)
    if d_sink.dtype != torch.float32 or d_sink.numel() != heads or not d_sink.is_contiguous():
        raise ValueError("d_sink must be a contiguous float32 tensor [heads]")
    for t, n in ((probs, "probs"), (dprobs, "dprobs"), (dscores, "dscores"), (lse, "lse"),
                 (delta, "delta"), (sink, "sink"), (d_sink, "d_sink"),
                 (kv_valid_len, "kv_valid_len"), (key_mask, "key_mask"), (workspace, "workspace")):
        _check_cuda(t, n, dev)
    d = _desc(rows, L, ld, batch, heads, q_len, causal, kv_valid_len, key_mask, sink)
    need = int(_abi.lib().fos_bwd_sink_workspace_bytes(ctypes.byref(d)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    lc = None if launch is None else ctypes.byref(launch._c())
    with torch.cuda.device(dev):
        st = _abi.lib().fos_softmax_bwd_sink(
            ctypes.byref(d), _DTYPES[probs.dtype], _ptr(probs), _ptr(dprobs), _ptr(dscores),
            _ptr(delta), _ptr(lse), _ptr(d_sink), _ptr(workspace), ws_bytes,
            _stream_handle(stream, dev), lc)
    if st != _abi.FOS_OK:
        raise FosError(st, "fos_softmax_bwd_sink")
    return dscores, d_sink, delta


def fos_sink_grad(lse, delta, sink, d_sink=None, *, batch, heads, q_len, key_len=1,
                  stream=None, launch: Launch | None = None):
    """Per-head sink gradient from the forward's LSE and the backward's delta."""
    dev = lse.device
    rows = int(batch) * int(heads) * int(q_len)
    for t, n in ((lse, "lse"), (delta, "delta")):
        if t.dtype != torch.float32 or t.numel() != rows or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous float32 tensor of batch*heads*q_len")
    if d_sink is None:
        d_sink = torch.empty(int(heads), dtype=torch.float32, device=dev)
    if d_sink.dtype != torch.float32 or d_sink.numel() != heads or not d_sink.is_contiguous():
        raise ValueError("d_sink must be a contiguous float32 tensor [heads]")
    for t, n in ((lse, "lse"), (delta, "delta"), (sink, "sink"), (d_sink, "d_sink")):
        _check_cuda(t, n, dev)
    if sink is None:
        raise ValueError("sink is required")
    L = max(1, int(key_len))
    d = _desc(rows, L, L, int(batch), int(heads), int(q_len), False, None, None, sink)
    lc = None if launch is None else ctypes.byref(launch._c())
    with torch.cuda.device(dev):
        st = _abi.lib().fos_sink_grad(ctypes.byref(d), _ptr(lse), _ptr(delta), _ptr(d_sink),
                                      _stream_handle(stream, dev), lc)
    if st != _abi.FOS_OK:
        raise FosError(st, "fos_sink_grad")
    return d_sink


def sink_chunk_range(q_len: int, batch_begin: int, batch_end: int) -> tuple[int, int]:
    """[c0, c1): the 256-position chunks of one head covered by batch entries [b0, b1)."""
    p0, p1 = int(batch_begin) * int(q_len), int(batch_end) * int(q_len)
    return p0 // 256, -(-p1 // 256)


def fos_sink_grad_partials(lse, delta, sink, partials=None, *, batch, heads, q_len,
                           batch_begin, batch_end, stream=None, launch: Launch | None = None):
    """Chunk partials ``[heads, c1 - c0]`` of the sink gradient for batch entries
    ``[batch_begin, batch_end)``; ``lse`` and ``delta`` hold those entries' rows only."""
    dev = lse.device
    n = (int(batch_end) - int(batch_begin)) * int(heads) * int(q_len)
    for t, nm in ((lse, "lse"), (delta, "delta")):
        if t.dtype != torch.float32 or t.numel() != n or not t.is_contiguous():
            raise ValueError(f"{nm} must be a contiguous float32 tensor of the shard's rows")
    c0, c1 = sink_chunk_range(q_len, batch_begin, batch_end)
    if partials is None:
        partials = torch.empty((int(heads), max(0, c1 - c0)), dtype=torch.float32, device=dev)
    if partials.dtype != torch.float32 or partials.numel() != heads * max(0, c1 - c0) or \
            not partials.is_contiguous():
        raise ValueError("partials must be a contiguous float32 tensor [heads, c1 - c0]")
    for t, nm in ((lse, "lse"), (delta, "delta"), (sink, "sink"), (partials, "partials")):
        _check_cuda(t, nm, dev)
    if sink is None:
        raise ValueError("sink is required")
    rows = int(batch) * int(heads) * int(q_len)
    d = _desc(rows, 1, 1, int(batch), int(heads), int(q_len), False, None, None, sink)
    lc = None if launch is None else ctypes.byref(launch._c())
    with torch.cuda.device(dev):
        st = _abi.lib().fos_sink_grad_partials(ctypes.byref(d), int(batch_begin), int(batch_end),
                                               _ptr(lse), _ptr(delta), _ptr(partials),
                                               _stream_handle(stream, dev), lc)
    if st != _abi.FOS_OK:
        raise FosError(st, "fos_sink_grad_partials")
    return partials


def fos_sink_grad_merge(partials):
    """d_sink ``[heads]`` (CPU) from every shard's chunk partials, ``[heads, n_chunks]`` CPU
    float32 in chunk order, added left to right by the library's host merge."""
    if partials.is_cuda or partials.dtype != torch.float32 or partials.dim() != 2:
        raise ValueError("partials must be a CPU float32 tensor [heads, n_chunks]")
    partials = partials.contiguous()
    heads, nchunks = partials.shape
    out = torch.empty(heads, dtype=torch.float32)
    st = _abi.lib().fos_sink_grad_merge(int(heads), int(nchunks), _ptr(partials), _ptr(out))
    if st != _abi.FOS_OK:
        raise FosError(st, "fos_sink_grad_merge")
    return out


def _check_host(t, name):
    if t is not None and t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")


def fos_step_host_workspace_bytes(scores, *, batch=None, heads=None, q_len=None,
                                  chunk_rows: int = 0) -> int:
    """Device workspace bytes ``fos_softmax_step_host`` needs for the problem of ``scores``
    (host arithmetic only; 0 for an empty problem)."""
    if scores.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {scores.dtype}")
    rows, L, ld, batch, heads, q_len = _geometry(scores, batch, heads, q_len)
    d = _abi.FosDesc(rows, ld, L, batch, heads, q_len, 0, 0, None, None, None)
    return int(_abi.lib().fos_step_host_workspace_bytes(ctypes.byref(d), _DTYPES[scores.dtype],
                                                        int(chunk_rows)))


def fos_softmax_step_host(scores, dprobs, probs=None, lse=None, dscores=None, delta=None, *,
                          batch=None, heads=None, q_len=None, causal=False, kv_valid_len=None,
                          key_mask=None, sink=None, d_sink=None, want_d_sink=True,
                          workspace=None, chunk_rows: int = 0, device=None, stream=None,
                          launch: Launch | None = None):
    """Forward, backward and (with a sink) sink gradient of host-resident data, through the
    library's chunked upload / compute / download pipeline.  ``scores``, ``dprobs`` and the
    outputs are CPU tensors (page-locked ones let the copies overlap; new outputs are
    allocated page-locked); ``kv_valid_len``, ``key_mask``, ``sink`` and ``workspace`` are
    CUDA tensors of the device that runs the step.  Returns ``(probs, lse, dscores, delta,
    d_sink)`` (``d_sink`` is None without a sink); they are complete once the stream is."""
    if scores.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {scores.dtype}")
    if device is None:
        for t in (workspace, sink, kv_valid_len, key_mask):
            if t is not None and t.is_cuda:
                device = t.device
                break
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    rows, L, ld, batch, heads, q_len = _geometry(scores, batch, heads, q_len)
    _same_layout(scores, dprobs, "scores", "dprobs")

    def host_like(t):
        return torch.empty_strided(t.shape, t.stride(), dtype=t.dtype, pin_memory=True)

    probs = host_like(scores) if probs is None else probs
    dscores = host_like(scores) if dscores is None else dscores
    _same_layout(scores, probs, "scores", "probs")
    _same_layout(scores, dscores, "scores", "dscores")
    if lse is None:
        lse = torch.empty(rows, dtype=torch.float32, pin_memory=True)
    if delta is None:
        delta = torch.empty(rows, dtype=torch.float32, pin_memory=True)
    for t, n in ((lse, "lse"), (delta, "delta")):
        if t.dtype != torch.float32 or t.numel() != rows or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous float32 tensor with one entry per row")
    if sink is not None and want_d_sink and d_sink is None:
        d_sink = torch.empty(heads, dtype=torch.float32, pin_memory=True)
    if d_sink is not None and (d_sink.dtype != torch.float32 or d_sink.numel() != heads or
                               not d_sink.is_contiguous()):
        raise ValueError("d_sink must be a contiguous float32 tensor [heads]")
    for t, n in ((scores, "scores"), (dprobs, "dprobs"), (probs, "probs"), (dscores, "dscores"),
                 (lse, "lse"), (delta, "delta"), (d_sink, "d_sink")):
        _check_host(t, n)
    for t, n in ((kv_valid_len, "kv_valid_len"), (key_mask, "key_mask"), (sink, "sink"),
                 (workspace, "workspace")):
        _check_cuda(t, n, dev)
    d = _desc(rows, L, ld, batch, heads, q_len, causal, kv_valid_len, key_mask, sink)
    dt = _DTYPES[scores.dtype]
    need = int(_abi.lib().fos_step_host_workspace_bytes(ctypes.byref(d), dt, int(chunk_rows)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    lc = None if launch is None else ctypes.byref(launch._c())
    with torch.cuda.device(dev):
        st = _abi.lib().fos_softmax_step_host(
            ctypes.byref(d), dt, _ptr(scores), _ptr(dprobs), _ptr(probs), _ptr(lse),
            _ptr(dscores), _ptr(delta), _ptr(d_sink), _ptr(workspace), ws_bytes,
            int(chunk_rows), _stream_handle(stream, dev), lc)
    if st != _abi.FOS_OK:
        raise FosError(st, "fos_softmax_step_host")
    return probs, lse, dscores, delta, d_sink


def fos_qk_scores(q, k, scale: float = 1.0, scores=None, *, out_dtype=torch.float32,
                  ld_scores=None, tile_n: int = 0, stream=None):
    """Scores ``[B, Hq, Sq, Skv]`` = scale * Q K^T on the tensor cores (see ``fos_qk_scores``
    in the C header).  ``q`` is ``[B, Hq, Sq, D]``, ``k`` ``[B, Hkv, Skv, D]``, both dense and of
    one 16-bit dtype; ``scores`` (optional) is a ``[B, Hq, Sq, Skv]`` view whose rows are
    ``ld_scores`` elements apart (a narrowed wider buffer).  When omitted it is allocated with
    rows padded to 16 bytes (the tensor stores need it) and returned as the narrowed view."""
    if q.dtype not in (torch.bfloat16, torch.float16) or k.dtype != q.dtype:
        raise ValueError("q and k must share one dtype, bfloat16 or float16")
    if q.dim() != 4 or k.dim() != 4 or not q.is_contiguous() or not k.is_contiguous():
        raise ValueError("q and k must be dense [B, H, S, D] tensors")
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Skv, Dk = k.shape
    if Bk != B or Dk != D:
        raise ValueError("q and k must agree in batch and head dimension")
    dev = q.device
    _check_cuda(k, "k", dev)
    if scores is None:
        per16 = 16 // torch.tensor([], dtype=out_dtype).element_size()
        ld_pad = max(per16, -(-Skv // per16) * per16)
        scores = torch.empty((B, Hq, Sq, ld_pad), dtype=out_dtype, device=dev)[..., :Skv]
    if scores.dtype not in _DTYPES or tuple(scores.shape) != (B, Hq, Sq, Skv) or \
            scores.stride(-1) != 1:
        raise ValueError("scores must be [B, Hq, Sq, Skv] with unit key stride")
    _check_cuda(scores, "scores", dev)
    if scores.numel() == 0:  # no score to compute (strides of an empty tensor say nothing)
        return scores
    ld = scores.stride(2) if ld_scores is None else int(ld_scores)
    if scores.stride(1) != Sq * ld or scores.stride(0) != Hq * Sq * ld:
        raise ValueError("scores rows must be ld_scores apart and densely packed otherwise")
    d = _abi.FosQkDesc(B, Hq, Hkv, Sq, Skv, D, ld, float(scale), int(tile_n))
    with torch.cuda.device(dev):
        st = _abi.lib().fos_qk_scores(ctypes.byref(d), _DTYPES[q.dtype], _DTYPES[scores.dtype],
                                      _ptr(q), _ptr(k), _ptr(scores), _stream_handle(stream, dev))
    if st != _abi.FOS_OK:
        raise FosError(st, "fos_qk_scores")
    return scores


def fos_pv_out(probs, v, out=None, *, scale: float = 1.0, out_dtype=torch.float32, stream=None):
    """Output ``[B, Hq, Sq, D]`` = scale * P V on the tensor cores (see ``fos_pv_out`` in the C
    header).  ``probs`` is a ``[B, Hq, Sq, Skv]`` view whose rows are ``ld`` elements apart
    (``ld`` a multiple of 8), ``v`` a dense ``[B, Hkv, Skv, D]`` of the same 16-bit dtype."""
    if probs.dtype not in (torch.bfloat16, torch.float16) or v.dtype != probs.dtype:
        raise ValueError("probs and v must share one dtype, bfloat16 or float16")
    if probs.dim() != 4 or v.dim() != 4 or not v.is_contiguous() or probs.stride(-1) != 1:
        raise ValueError("probs must be [B, H, Sq, Skv] with unit key stride, v dense "
                         "[B, Hkv, Skv, D]")
    B, Hq, Sq, Skv = probs.shape
    Bv, Hkv, Skv_v, D = v.shape
    if Bv != B or Skv_v != Skv:
        raise ValueError("probs and v must agree in batch and key count")
    dev = probs.device
    _check_cuda(v, "v", dev)
    if out is None:
        out = torch.empty((B, Hq, Sq, D), dtype=out_dtype, device=dev)
    if out.dtype not in _DTYPES or tuple(out.shape) != (B, Hq, Sq, D) or not out.is_contiguous():
        raise ValueError("out must be a dense [B, Hq, Sq, D] tensor")
    _check_cuda(out, "out", dev)
    if out.numel() == 0:
        return out
    ld = probs.stride(2)
    if probs.stride(1) != Sq * ld or probs.stride(0) != Hq * Sq * ld:
        raise ValueError("probs rows must be one stride apart and densely packed otherwise")
    d = _abi.FosPvDesc(B, Hq, Hkv, Sq, Skv, D, ld, float(scale))
    with torch.cuda.device(dev):
        st = _abi.lib().fos_pv_out(ctypes.byref(d), _DTYPES[probs.dtype], _DTYPES[out.dtype],
                                   _ptr(probs), _ptr(v), _ptr(out), _stream_handle(stream, dev))
    if st != _abi.FOS_OK:
        raise FosError(st, "fos_pv_out")
    return out


def fos_grad_kv(a, m, kv_heads: int, scale: float = 1.0, out=None, *, out_dtype=torch.float32,
                stream=None):
    """Output ``[B, Hkv, Skv, D]`` = scale * a^T m summed over each key head's query heads (see
    ``fos_grad_kv`` in the C header): dV from ``(P, dO)``, dK from ``(dScores, Q, scale)``.
    ``a`` is a ``[B, Hq, Sq, Skv]`` view whose rows are ``ld`` elements apart (``ld`` a multiple
    of 8), ``m`` a dense ``[B, Hq, Sq, D]`` of the same 16-bit dtype."""
    if a.dtype not in (torch.bfloat16, torch.float16) or m.dtype != a.dtype:
        raise ValueError("a and m must share one dtype, bfloat16 or float16")
    if a.dim() != 4 or m.dim() != 4 or not m.is_contiguous() or a.stride(-1) != 1:
        raise ValueError("a must be [B, Hq, Sq, Skv] with unit key stride, m dense [B, Hq, Sq, D]")
    B, Hq, Sq, Skv = a.shape
    Bm, Hm, Sm, D = m.shape
    if (Bm, Hm, Sm) != (B, Hq, Sq):
        raise ValueError("a and m must agree in batch, query heads and query positions")
    kv_heads = int(kv_heads)
    if kv_heads < 1 or Hq % kv_heads != 0:
        raise ValueError("kv_heads must divide the query heads")
    dev = a.device
    _check_cuda(m, "m", dev)
    if out is None:
        out = torch.empty((B, kv_heads, Skv, D), dtype=out_dtype, device=dev)
    if out.dtype not in _DTYPES or tuple(out.shape) != (B, kv_heads, Skv, D) or \
            not out.is_contiguous():
        raise ValueError("out must be a dense [B, Hkv, Skv, D] tensor")
    _check_cuda(out, "out", dev)
    if out.numel() == 0:
        return out
    ld = a.stride(2) if Sq > 0 else max(Skv, a.stride(2))
    if Sq > 0 and (a.stride(1) != Sq * ld or a.stride(0) != Hq * Sq * ld):
        raise ValueError("a rows must be one stride apart and densely packed otherwise")
    d = _abi.FosPvDesc(B, Hq, kv_heads, Sq, Skv, D, ld, float(scale))
    with torch.cuda.device(dev):
        st = _abi.lib().fos_grad_kv(ctypes.byref(d), _DTYPES[a.dtype], _DTYPES[out.dtype],
                                    _ptr(a), _ptr(m), _ptr(out), _stream_handle(stream, dev))
    if st != _abi.FOS_OK:
        raise FosError(st, "fos_grad_kv")
    return out


def fos_device_error(stream=None, device=None) -> int:
    """Synchronise the stream and return (and clear) the device error status code."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        return int(_abi.lib().fos_device_error(_stream_handle(stream, dev)))


def fos_status_string(status: int) -> str:
    return _abi.lib().fos_status_string(int(status)).decode()


def fos_contract_fingerprint() -> str:
    return _abi.lib().fos_contract_fingerprint().decode()

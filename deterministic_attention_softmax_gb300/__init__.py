"""Fixed-order, batch-invariant row softmax for GB300 (sm_103a).

The operation between the QK and AV GEMMs of joint attention ("[WS1][kernels] Add fixed-order
joint-attention softmax for Qwen-Image", Summary): forward P and LSE with optional causal /
valid-length / key masks and a per-head sink logit; backward delta and dScores; the per-head
sink gradient without atomics; and the fixed-order QK and PV contractions around it, on the
tensor cores.  The compute lives in ``libfos_softmax.so`` (C ABI in
``include/fos_softmax.h``); this package is its PyTorch binding, plus ``fixed_order_softmax``,
the same kernels as a differentiable op.
"""

from ._build import build
from .autograd import (FixedOrderAttention, FixedOrderSoftmax, fixed_order_attention,
                       fixed_order_softmax)
from .binding import (FosError, Launch, fos_contract_fingerprint, fos_device_error,
                      fos_grad_kv, fos_pv_out, fos_qk_scores, fos_sink_grad, fos_sink_grad_merge,
                      fos_sink_grad_partials, fos_softmax_bwd, fos_softmax_bwd_sink,
                      fos_softmax_fwd, fos_softmax_step_host, fos_status_string,
                      fos_step_host_workspace_bytes, sink_chunk_range)

__all__ = [
    "FixedOrderAttention", "FixedOrderSoftmax", "FosError", "Launch", "build",
    "fixed_order_attention", "fixed_order_softmax",
    "fos_contract_fingerprint", "fos_device_error", "fos_grad_kv", "fos_pv_out", "fos_qk_scores",
    "fos_sink_grad", "fos_sink_grad_merge", "fos_sink_grad_partials", "fos_softmax_bwd",
    "fos_softmax_bwd_sink", "fos_softmax_fwd", "fos_softmax_step_host", "fos_status_string",
    "fos_step_host_workspace_bytes", "sink_chunk_range",
]

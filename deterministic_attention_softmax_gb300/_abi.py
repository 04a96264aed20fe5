"""ctypes view of ``include/fos_softmax.h`` (argument marshalling only).

The library is loaded on first use.  If it has not been built the first call raises: there is
no fallback of any kind, every operation runs in the CUDA kernels of ``libfos_softmax.so``.
"""

from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
# FOS_LIBRARY=debug selects the build whose kernels check their indices (FOS_DEBUG); it is
# built on demand by ``_build.build(debug=True)`` and used by the tests only.
DEBUG_LIB_PATH = os.path.join(_PKG, "libfos_softmax_debug.so")
LIB_PATH = DEBUG_LIB_PATH if os.environ.get("FOS_LIBRARY") == "debug" else \
    os.path.join(_PKG, "libfos_softmax.so")

# fos_dtype
FOS_F32, FOS_BF16, FOS_F16 = 0, 1, 2
# fos_status
FOS_OK, FOS_ERR_INVALID, FOS_ERR_UNSUPPORTED, FOS_ERR_CUDA, FOS_ERR_TIMEOUT = 0, 1, 2, 3, 4
FOS_ERR_INDEX = 5
STATUS_NAMES = {0: "FOS_OK", 1: "FOS_ERR_INVALID", 2: "FOS_ERR_UNSUPPORTED", 3: "FOS_ERR_CUDA",
                4: "FOS_ERR_TIMEOUT", 5: "FOS_ERR_INDEX"}

# Every symbol include/fos_softmax.h declares.
EXPORTED = ("fos_softmax_fwd", "fos_softmax_bwd", "fos_sink_grad", "fos_sink_grad_partials",
            "fos_sink_grad_merge", "fos_softmax_step_host",
            "fos_step_host_workspace_bytes", "fos_softmax_step_host_static", "fos_qk_scores",
            "fos_pv_out", "fos_grad_kv",
            "fos_softmax_bwd_sink", "fos_bwd_sink_workspace_bytes", "fos_device_error",
            "fos_status_string", "fos_contract_fingerprint")


class FosDesc(ctypes.Structure):
    _fields_ = [
        ("rows", ctypes.c_int64),
        ("ld", ctypes.c_int64),
        ("key_len", ctypes.c_int32),
        ("batch", ctypes.c_int32),
        ("heads", ctypes.c_int32),
        ("q_len", ctypes.c_int32),
        ("causal", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("kv_valid_len", ctypes.c_void_p),
        ("key_mask", ctypes.c_void_p),
        ("sink", ctypes.c_void_p),
    ]


class FosQkDesc(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("q_heads", ctypes.c_int32),
        ("kv_heads", ctypes.c_int32),
        ("q_len", ctypes.c_int32),
        ("kv_len", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("ld_scores", ctypes.c_int64),
        ("scale", ctypes.c_float),
        ("tile_n", ctypes.c_int32),
    ]


class FosPvDesc(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("q_heads", ctypes.c_int32),
        ("kv_heads", ctypes.c_int32),
        ("q_len", ctypes.c_int32),
        ("kv_len", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("ld_probs", ctypes.c_int64),
        ("scale", ctypes.c_float),
    ]


class FosLaunch(ctypes.Structure):
    _fields_ = [
        ("warps_per_cta", ctypes.c_int32),
        ("ctas", ctypes.c_int32),
        ("stages", ctypes.c_int32),
        ("load_path", ctypes.c_int32),
        ("wait_timeout_ns", ctypes.c_int64),
        ("test_stall", ctypes.c_int32),
        ("generic", ctypes.c_int32),
        ("groups_per_cta", ctypes.c_int32),
        ("sink_fusion", ctypes.c_int32),
    ]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it was never built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; "
                "g.build()'); this package has no non-CUDA fallback")
        L = ctypes.CDLL(LIB_PATH)
        vp, dp, lp = ctypes.c_void_p, ctypes.POINTER(FosDesc), ctypes.POINTER(FosLaunch)
        L.fos_softmax_fwd.argtypes = [dp, ctypes.c_int, vp, vp, vp, vp, lp]
        L.fos_softmax_fwd.restype = ctypes.c_int
        L.fos_softmax_bwd.argtypes = [dp, ctypes.c_int, vp, vp, vp, vp, vp, lp]
        L.fos_softmax_bwd.restype = ctypes.c_int
        L.fos_sink_grad.argtypes = [dp, vp, vp, vp, vp, lp]
        L.fos_sink_grad.restype = ctypes.c_int
        L.fos_sink_grad_partials.argtypes = [dp, ctypes.c_int32, ctypes.c_int32, vp, vp, vp, vp,
                                             lp]
        L.fos_sink_grad_partials.restype = ctypes.c_int
        L.fos_sink_grad_merge.argtypes = [ctypes.c_int32, ctypes.c_int64, vp, vp]
        L.fos_sink_grad_merge.restype = ctypes.c_int
        L.fos_softmax_step_host.argtypes = [dp, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp,
                                            ctypes.c_size_t, ctypes.c_int64, vp, lp]
        L.fos_softmax_step_host.restype = ctypes.c_int
        L.fos_step_host_workspace_bytes.argtypes = [dp, ctypes.c_int, ctypes.c_int64]
        L.fos_step_host_workspace_bytes.restype = ctypes.c_size_t
        L.fos_softmax_step_host_static.argtypes = [dp, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp,
                                                   ctypes.c_int64, vp, lp]
        L.fos_softmax_step_host_static.restype = ctypes.c_int
        L.fos_softmax_bwd_sink.argtypes = [dp, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp,
                                           ctypes.c_size_t, vp, lp]
        L.fos_softmax_bwd_sink.restype = ctypes.c_int
        L.fos_bwd_sink_workspace_bytes.argtypes = [dp]
        L.fos_bwd_sink_workspace_bytes.restype = ctypes.c_size_t
        L.fos_qk_scores.argtypes = [ctypes.POINTER(FosQkDesc), ctypes.c_int, ctypes.c_int, vp, vp,
                                    vp, vp]
        L.fos_qk_scores.restype = ctypes.c_int
        L.fos_pv_out.argtypes = [ctypes.POINTER(FosPvDesc), ctypes.c_int, ctypes.c_int, vp, vp, vp,
                                 vp]
        L.fos_pv_out.restype = ctypes.c_int
        L.fos_grad_kv.argtypes = [ctypes.POINTER(FosPvDesc), ctypes.c_int, ctypes.c_int, vp, vp,
                                  vp, ctypes.c_void_p]
        L.fos_grad_kv.restype = ctypes.c_int
        L.fos_device_error.argtypes = [vp]
        L.fos_device_error.restype = ctypes.c_int
        L.fos_status_string.argtypes = [ctypes.c_int]
        L.fos_status_string.restype = ctypes.c_char_p
        L.fos_contract_fingerprint.argtypes = []
        L.fos_contract_fingerprint.restype = ctypes.c_char_p
        _lib = L
        return L

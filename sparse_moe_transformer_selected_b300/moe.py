"""Python binding of libmoe_b300.so: the C entry points of include/moe.h with the
same names and argument order.

Only argument marshalling happens here: a torch tensor argument is passed as
its data pointer (an int is passed through as a raw device address), the
stream defaults to torch's current stream, and a non-OK status raises
MoEError carrying the library's message.  Every step of the block runs in the
library's CUDA kernels; if the library is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_b300.so")

STATUS = {0: "MOE_OK", 1: "MOE_ERR_NULL", 2: "MOE_ERR_SHAPE", 3: "MOE_ERR_ALIGN",
          4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_UNSUPPORTED", 6: "MOE_ERR_CUDA",
          7: "MOE_ERR_TIMEOUT", 8: "MOE_ERR_DEVICE_BOUNDS"}

# moe_workspace_region `which` values
REGIONS = {"topk_idx": 0, "topk_w": 1, "offsets": 2, "perm": 3, "inv": 4,
           "x_perm": 5, "h_hi": 6, "h_lo": 7, "y": 8}

# Every symbol include/moe.h declares.
EXPORTS = ("moe_workspace_bytes", "moe_forward", "moe_block_forward", "moe_route",
           "moe_poll_status", "moe_last_error", "moe_workspace_region", "moe_set_trace_events",
           "moe_forward_noalloc", "moe_poll_status_noalloc", "moe_hidden_format",
           "moe_set_wait_limit", "moe_set_fault_injection", "moe_debug_combine",
           "moe_mma_peak")

# Scratch built into the library for moe_forward_noalloc (MOE_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 16 << 20


class MoEError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None


def load() -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing; build it with "
                           "`python -m sparse_moe_transformer_selected_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I32, F32, SZ = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                            ctypes.c_size_t)
    lib.moe_workspace_bytes.argtypes = [I64, I32, I32, I32, I32]
    lib.moe_workspace_bytes.restype = SZ
    lib.moe_forward.argtypes = [P, I64, I32, I32, P, P, P, P, P, P, P, P, I32, I32, F32, F32,
                                P, P, SZ, P]
    lib.moe_forward.restype = I32
    lib.moe_block_forward.argtypes = [P, I64, I32, I32, P, F32, P, P, P, P, P, P, P, P, I32,
                                      I32, F32, F32, P, P, SZ, P]
    lib.moe_block_forward.restype = I32
    lib.moe_route.argtypes = [P, I64, I32, P, P, I32, I32, P, P, P, P, P, P, SZ, P]
    lib.moe_route.restype = I32
    lib.moe_poll_status.argtypes = [P, P]
    lib.moe_poll_status.restype = I32
    lib.moe_last_error.argtypes = []
    lib.moe_last_error.restype = ctypes.c_char_p
    lib.moe_workspace_region.argtypes = [I64, I32, I32, I32, I32, I32,
                                         ctypes.POINTER(SZ), ctypes.POINTER(SZ)]
    lib.moe_workspace_region.restype = I32
    lib.moe_set_trace_events.argtypes = [ctypes.POINTER(P), I32]
    lib.moe_set_trace_events.restype = I32
    lib.moe_forward_noalloc.argtypes = [P, I64, I32, I32, P, P, P, P, P, P, P, P, I32, I32, F32,
                                        F32, P, P]
    lib.moe_forward_noalloc.restype = I32
    lib.moe_set_wait_limit.argtypes = [ctypes.c_double]
    lib.moe_set_wait_limit.restype = I32
    lib.moe_set_fault_injection.argtypes = [I32]
    lib.moe_set_fault_injection.restype = I32
    lib.moe_debug_combine.argtypes = [P, P, P, P, I64, I32, I32, P, P, SZ, P]
    lib.moe_debug_combine.restype = I32
    lib.moe_mma_peak.argtypes = [I32, I32, ctypes.POINTER(ctypes.c_double), P, P]
    lib.moe_mma_peak.restype = I32
    lib.moe_poll_status_noalloc.argtypes = [P]
    lib.moe_poll_status_noalloc.restype = I32
    lib.moe_hidden_format.argtypes = [I64, I32, I32, I32, I32, F32, ctypes.POINTER(I32),
                                      ctypes.POINTER(I32)]
    lib.moe_hidden_format.restype = I32
    _lib = lib
    return lib


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return a.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int) -> int:
    if status != 0:
        raise MoEError(status, moe_last_error())
    return status


def moe_last_error() -> str:
    return load().moe_last_error().decode("utf-8", "replace")


def moe_workspace_bytes(T: int, d: int, W: int, E: int, k: int) -> int:
    return int(load().moe_workspace_bytes(T, d, W, E, k))


def moe_workspace_region(T: int, d: int, W: int, E: int, k: int, which) -> tuple[int, int]:
    which = REGIONS[which] if isinstance(which, str) else which
    off, nb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(load().moe_workspace_region(T, d, W, E, k, which, ctypes.byref(off), ctypes.byref(nb)))
    return off.value, nb.value


def moe_forward(x_bf16, T, d, W, router_w, router_b, w_gu_fp4, w_gu_scale, b_gu_bf16,
                w_dn_fp4, w_dn_scale, b_dn_bf16, E, k, limit, alpha, out_bf16, workspace,
                workspace_bytes, stream=None) -> int:
    return _check(load().moe_forward(
        _ptr(x_bf16), T, d, W, _ptr(router_w), _ptr(router_b), _ptr(w_gu_fp4),
        _ptr(w_gu_scale), _ptr(b_gu_bf16), _ptr(w_dn_fp4), _ptr(w_dn_scale), _ptr(b_dn_bf16),
        E, k, limit, alpha, _ptr(out_bf16), _ptr(workspace), workspace_bytes, _stream(stream)))


def moe_block_forward(x_bf16, T, d, W, norm_w, eps, router_w, router_b, w_gu_fp4, w_gu_scale,
                      b_gu_bf16, w_dn_fp4, w_dn_scale, b_dn_bf16, E, k, limit, alpha, out_bf16,
                      workspace, workspace_bytes, stream=None) -> int:
    """out = x + MoE(RMSNorm(x)); see include/moe.h."""
    return _check(load().moe_block_forward(
        _ptr(x_bf16), T, d, W, _ptr(norm_w), eps, _ptr(router_w), _ptr(router_b),
        _ptr(w_gu_fp4), _ptr(w_gu_scale), _ptr(b_gu_bf16), _ptr(w_dn_fp4), _ptr(w_dn_scale),
        _ptr(b_dn_bf16), E, k, limit, alpha, _ptr(out_bf16), _ptr(workspace), workspace_bytes,
        _stream(stream)))


def moe_route(x_bf16, T, d, router_w, router_b, E, k, topk_idx, topk_w, offsets, perm, inv,
              workspace, workspace_bytes, stream=None) -> int:
    return _check(load().moe_route(
        _ptr(x_bf16), T, d, _ptr(router_w), _ptr(router_b), E, k, _ptr(topk_idx), _ptr(topk_w),
        _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(workspace), workspace_bytes, _stream(stream)))


def moe_poll_status(workspace, stream=None) -> int:
    return _check(load().moe_poll_status(_ptr(workspace), _stream(stream)))


# Number formats of h between the two GEMMs (moe_hidden_format).
HIDDEN_BF16_PAIR, HIDDEN_F16_PAIR, HIDDEN_E4M3_TERMS = 0, 1, 2


def moe_hidden_format(T: int, d: int, W: int, E: int, k: int, limit: float) -> tuple:
    """(format, exponent): how moe_forward carries h on this shape and clamp.

    HIDDEN_BF16_PAIR / HIDDEN_F16_PAIR: h = hi + lo; HIDDEN_E4M3_TERMS:
    h = (t0 + t1/16 + t2/256 + t3/4096) * 2**exponent.
    """
    f = ctypes.c_int(0)
    x = ctypes.c_int(0)
    _check(load().moe_hidden_format(T, d, W, E, k, limit, ctypes.byref(f), ctypes.byref(x)))
    return f.value, x.value


def moe_set_trace_events(events) -> int:
    """events: a sequence of 7 torch.cuda.Event (or raw cudaEvent_t ints), or None."""
    if not events:
        return _check(load().moe_set_trace_events(None, 0))
    handles = [e if isinstance(e, int) else e.cuda_event for e in events]
    arr = (ctypes.c_void_p * len(handles))(*handles)
    return _check(load().moe_set_trace_events(arr, len(handles)))


def moe_forward_noalloc(x_bf16, T, d, W, router_w, router_b, w_gu_fp4, w_gu_scale, b_gu_bf16,
                        w_dn_fp4, w_dn_scale, b_dn_bf16, E, k, limit, alpha, out_bf16,
                        stream=None) -> int:
    """moe_forward with the library's built-in scratch instead of a workspace,
    for callers that cannot allocate device memory; see include/moe.h."""
    return _check(load().moe_forward_noalloc(
        _ptr(x_bf16), T, d, W, _ptr(router_w), _ptr(router_b), _ptr(w_gu_fp4),
        _ptr(w_gu_scale), _ptr(b_gu_bf16), _ptr(w_dn_fp4), _ptr(w_dn_scale), _ptr(b_dn_bf16),
        E, k, limit, alpha, _ptr(out_bf16), _stream(stream)))


def moe_poll_status_noalloc(stream=None) -> int:
    """moe_poll_status for the built-in scratch of moe_forward_noalloc."""
    return _check(load().moe_poll_status_noalloc(_stream(stream)))


def moe_set_wait_limit(seconds: float) -> int:
    """Wait limit of the GEMMs' bounded waits for later calls (0: default 2 s)."""
    return _check(load().moe_set_wait_limit(seconds))


def moe_set_fault_injection(mode: int) -> int:
    """Test hook (include/moe.h): 1 makes gate_up's weight producer issue nothing."""
    return _check(load().moe_set_fault_injection(mode))


def moe_debug_combine(y, perm, inv, topk_w, T, d, k, out_bf16, workspace, workspace_bytes,
                      stream=None) -> int:
    """Test hook: the fused combine on caller tables (include/moe.h)."""
    return _check(load().moe_debug_combine(
        _ptr(y), _ptr(perm), _ptr(inv), _ptr(topk_w), T, d, k, _ptr(out_bf16), _ptr(workspace),
        workspace_bytes, _stream(stream)))


MMA_KINDS = {"f16": 0, "mxf8f6f4": 1, "f16_tmem_a_n128": 2, "f16_tmem_a_n256": 3}


def moe_mma_peak(kind, iters, workspace, stream=None) -> float:
    """Dense TFLOP/s of an MMA form (a key of MMA_KINDS); include/moe.h."""
    kind = MMA_KINDS[kind] if isinstance(kind, str) else kind
    out = ctypes.c_double(0.0)
    _check(load().moe_mma_peak(kind, iters, ctypes.byref(out), _ptr(workspace), _stream(stream)))
    return out.value

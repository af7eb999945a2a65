"""Python binding of the GB300 MoE layer library (``libmoe.so``).

Argument marshalling only: each function below passes device pointers, sizes
and the CUDA stream to the C entry point of the same name declared in
``include/moe.h``; every step of the layer runs in the library's CUDA kernels.
PyTorch supplies device memory and streams.  There is no fallback: if the
library is missing or fails to load, every call raises.

Tensor arguments are ``torch.Tensor`` objects (contiguous, on the current
device) or ``None`` where the C call accepts NULL.  bf16 layers take
``torch.bfloat16`` tensors, fp32 layers ``torch.float32``.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "MoeDesc", "MoeError", "MOE_F32", "MOE_BF16", "MOE_FLAG_HOST_IO", "MOE_FLAG_SIMT_FFN",
    "MOE_FLAG_NO_DECODE", "MOE_FLAG_SIMT_ROUTER", "MOE_FLAG_GEMM_SINGLE", "MOE_FLAG_GEMM_PAIR", "MOE_FLAG_SWIGLU",
    "MOE_FLAG_TEST_WAIT_TIMEOUT", "MOE_FLAG_GEMM_ROWS", "MOE_FLAG_FFN_SPLIT", "MOE_FLAG_REROUTE", "MOE_FLAG_FUSED_COMBINE", "MOE_FLAG_DECODE_SPLIT", "MOE_FLAG_GATHER_GEMM", "lib",
    "library_path", "make_desc", "moe_reroute",
    "moe_status_string", "moe_capacity_default", "moe_max_rows", "moe_workspace_size",
    "moe_router_topk", "moe_dispatch", "moe_dispatch_noalloc", "moe_expert_ffn", "moe_combine", "moe_aux_loss",
    "moe_layer_forward", "moe_get_device_error", "moe_profile_events", "moe_layer_launches", "moe_ffn_kernel", "moe_layer_decode_fused",
    "MOE_FFN_STREAM", "MOE_FFN_SIMT", "MOE_FFN_TC_SINGLE", "MOE_FFN_TC_PAIRS", "MOE_FFN_TC_FUSED",
    "MOE_FFN_STREAM_SPLIT", "workspace", "MOE_OK", "MOE_ERR_INVALID", "MOE_ERR_UNSUPPORTED", "MOE_ERR_WORKSPACE",
    "MOE_ERR_CUDA", "MOE_ERR_TIMEOUT", "MOE_ERR_DEVICE",
]

MOE_F32, MOE_BF16 = 0, 1
MOE_FLAG_HOST_IO = 1 << 0
MOE_FLAG_SIMT_FFN = 1 << 1
MOE_FLAG_NO_DECODE = 1 << 2
MOE_FLAG_SIMT_ROUTER = 1 << 3
MOE_FLAG_GEMM_SINGLE = 1 << 4
MOE_FLAG_GEMM_PAIR = 1 << 5
MOE_FLAG_SWIGLU = 1 << 6
MOE_FLAG_TEST_WAIT_TIMEOUT = 1 << 7
MOE_FLAG_GEMM_ROWS = 1 << 8
MOE_FLAG_FFN_SPLIT = 1 << 9
MOE_FLAG_REROUTE = 1 << 10
MOE_FLAG_FUSED_COMBINE = 1 << 11
MOE_FLAG_DECODE_SPLIT = 1 << 12
MOE_FLAG_GATHER_GEMM = 1 << 13
# moe_ffn_kernel results
MOE_FFN_STREAM, MOE_FFN_SIMT, MOE_FFN_TC_SINGLE, MOE_FFN_TC_PAIRS, MOE_FFN_TC_FUSED, MOE_FFN_STREAM_SPLIT = 0, 1, 2, 3, 4, 5

# status codes (MoeError.code)
MOE_OK = 0
MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE = \
    -1, -2, -3, -4, -5, -6

_PKG = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_PKG, "_lib", "libmoe.so")


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {moe_status_string(code)} ({code})")
        self.code = code


class MoeDesc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
                ("K", ctypes.c_int32), ("F", ctypes.c_int32), ("capacity", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("flags", ctypes.c_uint32), ("temperature", ctypes.c_float)]


_P = ctypes.c_void_p
_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_capacity_default": (ctypes.c_int64, [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]),
    "moe_max_rows": (ctypes.c_int64, [ctypes.POINTER(MoeDesc)]),
    "moe_workspace_size": (ctypes.c_int, [ctypes.POINTER(MoeDesc), ctypes.POINTER(ctypes.c_size_t)]),
    "moe_router_topk": (ctypes.c_int, [ctypes.POINTER(MoeDesc)] + [_P] * 8 + [ctypes.c_size_t, _P]),
    "moe_dispatch": (ctypes.c_int, [ctypes.POINTER(MoeDesc)] + [_P] * 9 + [ctypes.c_size_t, _P]),
    "moe_dispatch_noalloc": (ctypes.c_int, [ctypes.POINTER(MoeDesc)] + [_P] * 10),
    "moe_reroute": (ctypes.c_int, [ctypes.POINTER(MoeDesc)] + [_P] * 7 + [ctypes.c_size_t, _P]),
    "moe_expert_ffn": (ctypes.c_int, [ctypes.POINTER(MoeDesc)] + [_P] * 9 + [ctypes.c_size_t, _P]),
    "moe_combine": (ctypes.c_int, [ctypes.POINTER(MoeDesc)] + [_P] * 5),
    "moe_aux_loss": (ctypes.c_int, [ctypes.POINTER(MoeDesc)] + [_P] * 4),
    "moe_layer_forward": (ctypes.c_int, [ctypes.POINTER(MoeDesc)] + [_P] * 12 + [ctypes.c_size_t, _P]),
    "moe_get_device_error": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int32), _P]),
    "moe_profile_events": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]),
    "moe_layer_launches": (ctypes.c_int, [ctypes.POINTER(MoeDesc)]),
    "moe_ffn_kernel": (ctypes.c_int, [ctypes.POINTER(MoeDesc)]),
    "moe_layer_decode_fused": (ctypes.c_int, [ctypes.POINTER(MoeDesc)]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Load ``libmoe.so`` (built by ``build.py``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(f"MoE CUDA library not built: {library_path} is missing "
                               "(run __graft_entry__.build() or python -m "
                               "sparse_mixture_experts_topk_gb300.build)")
        L = ctypes.CDLL(library_path)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, rc):
    if rc != MOE_OK:
        raise MoeError(fn, rc)


def make_desc(T, H, E, K, F, capacity=0, dtype=MOE_BF16, flags=0, temperature=1.0) -> MoeDesc:
    return MoeDesc(int(T), int(H), int(E), int(K), int(F), int(capacity), int(dtype), int(flags),
                   float(temperature))


def moe_status_string(code: int) -> str:
    return lib().moe_status_string(int(code)).decode()


def moe_capacity_default(T: int, E: int, K: int) -> int:
    return int(lib().moe_capacity_default(int(T), int(E), int(K)))


def moe_max_rows(desc: MoeDesc) -> int:
    return int(lib().moe_max_rows(ctypes.byref(desc)))


def moe_workspace_size(desc: MoeDesc) -> int:
    n = ctypes.c_size_t(0)
    _check("moe_workspace_size", lib().moe_workspace_size(ctypes.byref(desc), ctypes.byref(n)))
    return int(n.value)


def workspace(desc: MoeDesc, device=None):
    """A zero-filled device workspace of ``moe_workspace_size(desc)`` bytes."""
    import torch
    return torch.zeros(max(moe_workspace_size(desc), 256), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def moe_router_topk(desc, x, Wg, gate_bias, logits, ids, w, psum, ws, stream=None):
    _check("moe_router_topk", lib().moe_router_topk(
        ctypes.byref(desc), _ptr(x), _ptr(Wg), _ptr(gate_bias), _ptr(logits), _ptr(ids), _ptr(w),
        _ptr(psum), _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream)))


def moe_dispatch(desc, ids, x, count, offs, src, pos, x_perm, dropped, ws, stream=None):
    _check("moe_dispatch", lib().moe_dispatch(
        ctypes.byref(desc), _ptr(ids), _ptr(x), _ptr(count), _ptr(offs), _ptr(src), _ptr(pos),
        _ptr(x_perm), _ptr(dropped), _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream)))


def moe_dispatch_noalloc(desc, ids, x, count, offs, src, pos, x_perm, dropped, device_error,
                         stream=None):
    """``moe_dispatch`` for callers that cannot allocate device memory: the
    scratch is a fixed 64 KiB array inside the library, so no workspace is
    passed.  Calls on one device must not overlap on the GPU."""
    _check("moe_dispatch_noalloc", lib().moe_dispatch_noalloc(
        ctypes.byref(desc), _ptr(ids), _ptr(x), _ptr(count), _ptr(offs), _ptr(src), _ptr(pos),
        _ptr(x_perm), _ptr(dropped), _ptr(device_error), _stream(stream)))


def moe_reroute(desc, logits, ids, pos, offs, ids_out, dropped, ws, stream=None):
    _check("moe_reroute", lib().moe_reroute(
        ctypes.byref(desc), _ptr(logits), _ptr(ids), _ptr(pos), _ptr(offs), _ptr(ids_out), _ptr(dropped),
        _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream)))


def moe_expert_ffn(desc, x_perm, offs, W1, b1, W2, b2, h_perm, y_perm, ws, stream=None):
    _check("moe_expert_ffn", lib().moe_expert_ffn(
        ctypes.byref(desc), _ptr(x_perm), _ptr(offs), _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2),
        _ptr(h_perm), _ptr(y_perm), _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream)))


def moe_combine(desc, y_perm, pos, w, out, stream=None):
    _check("moe_combine", lib().moe_combine(
        ctypes.byref(desc), _ptr(y_perm), _ptr(pos), _ptr(w), _ptr(out), _stream(stream)))


def moe_aux_loss(desc, psum, count, loss, stream=None):
    _check("moe_aux_loss", lib().moe_aux_loss(
        ctypes.byref(desc), _ptr(psum), _ptr(count), _ptr(loss), _stream(stream)))


def moe_layer_forward(desc, x, Wg, gate_bias, W1, b1, W2, b2, out, aux, count, dropped, ws,
                      stream=None):
    _check("moe_layer_forward", lib().moe_layer_forward(
        ctypes.byref(desc), _ptr(x), _ptr(Wg), _ptr(gate_bias), _ptr(W1), _ptr(b1), _ptr(W2),
        _ptr(b2), _ptr(out), _ptr(aux), _ptr(count), _ptr(dropped), _ptr(ws),
        ws.numel() if ws is not None else 0, _stream(stream)))


def moe_layer_launches(desc: MoeDesc) -> int:
    """Number of kernels one ``moe_layer_forward`` with ``desc`` launches."""
    n = int(lib().moe_layer_launches(ctypes.byref(desc)))
    if n < 0:
        _check("moe_layer_launches", n)
    return n


def moe_ffn_kernel(desc: MoeDesc) -> int:
    """Which expert-FFN kernel (``MOE_FFN_*``) a call with ``desc`` runs."""
    k = int(lib().moe_ffn_kernel(ctypes.byref(desc)))
    if k < 0:
        _check("moe_ffn_kernel", k)
    return k


def moe_layer_decode_fused(desc: MoeDesc) -> bool:
    """Whether ``moe_layer_forward`` runs ``desc`` as the one-launch decode layer."""
    k = int(lib().moe_layer_decode_fused(ctypes.byref(desc)))
    if k < 0:
        _check("moe_layer_decode_fused", k)
    return k == 1


def moe_get_device_error(ws, stream=None) -> int:
    code = ctypes.c_int32(0)
    _check("moe_get_device_error", lib().moe_get_device_error(_ptr(ws), ctypes.byref(code),
                                                              _stream(stream)))
    return int(code.value)


_prof_events = None


def moe_profile_events(events) -> None:
    """Record the 6 given ``torch.cuda.Event`` objects at the stage boundaries of
    every later ``moe_layer_forward`` on this thread; ``None`` switches it off."""
    global _prof_events
    if not events:
        _check("moe_profile_events", lib().moe_profile_events(None, 0))
        _prof_events = None
        return
    events = list(events)
    for ev in events:            # torch creates the CUDA event on first record
        if not ev.cuda_event:
            ev.record()
    arr = (ctypes.c_void_p * len(events))(*[ev.cuda_event for ev in events])
    _check("moe_profile_events", lib().moe_profile_events(arr, len(events)))
    _prof_events = events        # the library records these handles until switched off

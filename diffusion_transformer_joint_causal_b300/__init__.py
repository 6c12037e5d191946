"""Python binding of the dit_attn C-ABI library (argument marshalling only).

Every step of the attention forward runs in the CUDA kernels of
``libdit_attn.so``; this module only checks tensors, passes their device
pointers and the current CUDA stream through ctypes, and turns status codes
into exceptions.  PyTorch supplies device memory and streams.  There is no
fallback: if the library is missing, importing the names below raises.

    import diffusion_transformer_joint_causal_b300 as dit
    dit.create()                      # once per device
    out = dit.forward(q, k, v)        # q,k,v: bf16 CUDA tensors [B, H, L, d]

    # e4m3 queries/keys: quantise after the RMS norm, then the e4m3-QK forward
    s = math.sqrt(128) / 448          # |rms-normalised value| <= sqrt(d)
    q8 = dit.rmsnorm_e4m3(q, out_scale=1 / s)
    k8 = dit.rmsnorm_e4m3(k, out_scale=1 / s)
    out = dit.forward_qk8(q8, k8, v, q_scale=s, k_scale=s)

    # e4m3 values too (P rounded to e4m3 before P.V); v_scale from calibration
    v_scale = float(v.abs().max()) / 448
    v8 = dit.quantize_e4m3(v, out_scale=1 / v_scale)
    out = dit.forward_fp8(q8, k8, v8, q_scale=s, k_scale=s, v_scale=v_scale)
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

__all__ = ["create", "destroy", "forward", "forward_ptr", "status_string", "get_device_error",
           "check_wait_timeout", "rmsnorm", "rmsnorm_ptr", "forward_qk8", "forward_qk8_ptr",
           "rmsnorm_e4m3", "rmsnorm_e4m3_ptr", "forward_ws_ptr", "forward_qk8_ws_ptr",
           "workspace_size", "forward_noalloc", "forward_noalloc_ptr", "forward_fp8",
           "forward_fp8_ptr", "forward_fp8_ws_ptr", "quantize_e4m3", "quantize_e4m3_ptr",
           "check_exp2", "last_cuda_error", "version", "library_path", "DitAttnError", "STATUS",
           "EXPORTED_SYMBOLS"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libdit_attn.so")

STATUS = {
    0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "NOT_INITIALIZED",
    4: "NO_DEVICE", 5: "CUDA", 6: "TIMEOUT",
}

EXPORTED_SYMBOLS = ("dit_attn_version", "dit_attn_create", "dit_attn_forward",
                    "dit_attn_destroy", "dit_attn_status_string", "dit_attn_get_device_error",
                    "dit_attn_check_wait_timeout", "dit_attn_last_cuda_error", "dit_attn_rmsnorm",
                    "dit_attn_forward_qk8", "dit_attn_rmsnorm_e4m3", "dit_attn_forward_ws",
                    "dit_attn_forward_qk8_ws", "dit_attn_workspace_size",
                    "dit_attn_forward_noalloc", "dit_attn_forward_fp8",
                    "dit_attn_forward_fp8_ws", "dit_attn_quantize_e4m3", "dit_attn_check_exp2")

_lock = threading.Lock()
_lib = None


class DitAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status_string(status)})")


def library_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise ImportError(
                    f"{_LIB_PATH} is missing; build it with "
                    "`python -m diffusion_transformer_joint_causal_b300.build`")
            lib = ctypes.CDLL(_LIB_PATH)
            c_int, vp = ctypes.c_int, ctypes.c_void_p
            lib.dit_attn_version.restype = c_int
            lib.dit_attn_version.argtypes = []
            lib.dit_attn_create.restype = c_int
            lib.dit_attn_create.argtypes = []
            lib.dit_attn_destroy.restype = c_int
            lib.dit_attn_destroy.argtypes = []
            lib.dit_attn_forward.restype = c_int
            lib.dit_attn_forward.argtypes = [vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int,
                                             ctypes.c_float, vp]
            lib.dit_attn_status_string.restype = ctypes.c_char_p
            lib.dit_attn_status_string.argtypes = [c_int]
            lib.dit_attn_get_device_error.restype = c_int
            lib.dit_attn_get_device_error.argtypes = [vp]
            lib.dit_attn_check_wait_timeout.restype = c_int
            lib.dit_attn_check_wait_timeout.argtypes = [c_int, vp]
            lib.dit_attn_rmsnorm.restype = c_int
            lib.dit_attn_rmsnorm.argtypes = [vp, vp, vp, ctypes.c_longlong, c_int, ctypes.c_float, vp]
            lib.dit_attn_forward_qk8.restype = c_int
            lib.dit_attn_forward_qk8.argtypes = [vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int,
                                                 ctypes.c_float, ctypes.c_float, ctypes.c_float, vp]
            lib.dit_attn_rmsnorm_e4m3.restype = c_int
            lib.dit_attn_rmsnorm_e4m3.argtypes = [vp, vp, vp, ctypes.c_longlong, c_int,
                                                  ctypes.c_float, ctypes.c_float, vp]
            lib.dit_attn_forward_ws.restype = c_int
            lib.dit_attn_forward_ws.argtypes = [vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int,
                                                ctypes.c_float, vp, ctypes.c_longlong, vp]
            lib.dit_attn_forward_qk8_ws.restype = c_int
            lib.dit_attn_forward_qk8_ws.argtypes = [vp, vp, vp, vp, c_int, c_int, c_int, c_int,
                                                    c_int, ctypes.c_float, ctypes.c_float,
                                                    ctypes.c_float, vp, ctypes.c_longlong, vp]
            lib.dit_attn_forward_noalloc.restype = c_int
            lib.dit_attn_forward_noalloc.argtypes = [vp, vp, vp, vp, c_int, c_int, c_int, c_int,
                                                     c_int, ctypes.c_float, vp]
            lib.dit_attn_workspace_size.restype = c_int
            lib.dit_attn_workspace_size.argtypes = [c_int, c_int, c_int, c_int, c_int, c_int,
                                                    ctypes.POINTER(ctypes.c_longlong)]
            lib.dit_attn_forward_fp8.restype = c_int
            lib.dit_attn_forward_fp8.argtypes = [vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int,
                                                 ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                                 ctypes.c_float, vp]
            lib.dit_attn_forward_fp8_ws.restype = c_int
            lib.dit_attn_forward_fp8_ws.argtypes = [vp, vp, vp, vp, c_int, c_int, c_int, c_int,
                                                    c_int, ctypes.c_float, ctypes.c_float,
                                                    ctypes.c_float, ctypes.c_float, vp,
                                                    ctypes.c_longlong, vp]
            lib.dit_attn_quantize_e4m3.restype = c_int
            lib.dit_attn_quantize_e4m3.argtypes = [vp, vp, ctypes.c_longlong, ctypes.c_float, vp]
            lib.dit_attn_check_exp2.restype = c_int
            lib.dit_attn_check_exp2.argtypes = [vp, vp, vp, ctypes.c_longlong, c_int, vp]
            lib.dit_attn_last_cuda_error.restype = c_int
            lib.dit_attn_last_cuda_error.argtypes = []
            _lib = lib
    return _lib


def version() -> int:
    return _load().dit_attn_version()


def status_string(status: int) -> str:
    return _load().dit_attn_status_string(int(status)).decode()


def last_cuda_error() -> int:
    return _load().dit_attn_last_cuda_error()


def create() -> None:
    """Prepare the current CUDA device (idempotent)."""
    rc = _load().dit_attn_create()
    if rc:
        raise DitAttnError(rc, "dit_attn_create")


def destroy() -> None:
    _ws_sizes.clear()
    rc = _load().dit_attn_destroy()
    if rc:
        raise DitAttnError(rc, "dit_attn_destroy")


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))


def get_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the kernels' error word."""
    return _load().dit_attn_get_device_error(_stream_handle(stream))


def check_wait_timeout(limit_us: int, stream=None) -> int:
    """Enqueue the bounded-wait self-test kernel; returns the launch status."""
    return _load().dit_attn_check_wait_timeout(int(limit_us), _stream_handle(stream))


def check_exp2(x, degree: int, stream=None):
    """(y_fma, y_mufu) for a float32 CUDA tensor x: the softmax's FMA-pipe 2^x of
    the given degree (2 or 3) and the MUFU ex2.approx it stands in for."""
    import torch
    if not isinstance(x, torch.Tensor) or x.dtype != torch.float32 or not x.is_cuda:
        raise TypeError("x must be a float32 CUDA tensor")
    x = x.contiguous()
    y_fma, y_mufu = torch.empty_like(x), torch.empty_like(x)
    with torch.cuda.device(x.device):
        rc = _load().dit_attn_check_exp2(ctypes.c_void_p(x.data_ptr()),
                                         ctypes.c_void_p(y_fma.data_ptr()),
                                         ctypes.c_void_p(y_mufu.data_ptr()),
                                         ctypes.c_longlong(x.numel()), int(degree),
                                         _stream_handle(stream))
    if rc:
        raise DitAttnError(rc, "dit_attn_check_exp2")
    return y_fma, y_mufu


def forward_ptr(q: int, k: int, v: int, out: int, B: int, H: int, Lq: int, Lk: int, d: int,
                scale: float, stream=0) -> int:
    """Raw C-ABI call with integer device pointers; returns the status code."""
    s = stream if isinstance(stream, ctypes.c_void_p) else ctypes.c_void_p(int(stream))
    return _load().dit_attn_forward(ctypes.c_void_p(q), ctypes.c_void_p(k), ctypes.c_void_p(v),
                                    ctypes.c_void_p(out), B, H, Lq, Lk, d,
                                    ctypes.c_float(scale), s)


def _check_qkv(q, k, v, qk_dtypes, v_dtypes=None):
    import torch
    v_dtypes = v_dtypes or (torch.bfloat16,)
    for name, t, dtypes in (("q", q, qk_dtypes), ("k", k, qk_dtypes), ("v", v, v_dtypes)):
        if not isinstance(t, torch.Tensor) or t.dtype not in dtypes or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor of dtype {' or '.join(map(str, dtypes))}")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, H, L, d] tensor")
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    if tuple(k.shape) != (B, H, Lk, d) or tuple(v.shape) != (B, H, Lk, d):
        raise ValueError("k and v must be [B, H, Lk, d] with q's B, H and d")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be on one device")
    return B, H, Lq, Lk, d


def _out_like(out, q, shape):
    import torch
    if out is None:
        return torch.empty(shape, dtype=torch.bfloat16, device=q.device)
    if (out.dtype != torch.bfloat16 or tuple(out.shape) != tuple(shape)
            or not out.is_contiguous() or out.device != q.device):
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    return out


def workspace_size(B: int, H: int, Lq: int, Lk: int, d: int, qk8: bool = False,
                   variant: int | None = None) -> int:
    """Bytes of split-tail workspace the forward uses for these sizes (0: none).
    variant: 0 forward, 1 forward_qk8, 2 forward_fp8 (default: 1 if qk8 else 0)."""
    if variant is None:
        variant = 1 if qk8 else 0
    nb = ctypes.c_longlong(0)
    rc = _load().dit_attn_workspace_size(B, H, Lq, Lk, d, int(variant), ctypes.byref(nb))
    if rc:
        raise DitAttnError(rc, "dit_attn_workspace_size")
    return nb.value


_ws_sizes = {}   # (device index, sizes, variant) -> workspace bytes; fixed once a device is created


def _workspace(workspace, device, B, H, Lq, Lk, d, variant, stream):
    """(tensor, pointer, bytes) of the workspace: "auto" allocates what the
    library asks for through torch's caching allocator, ordered on the stream
    the call runs on; None runs unsplit; a uint8 CUDA tensor is used as given."""
    import torch
    if workspace is None:
        return None, 0, 0
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError('workspace must be "auto", None or a uint8 CUDA tensor')
        key = (device.index, B, H, Lq, Lk, d, int(variant))
        nb = _ws_sizes.get(key)
        if nb is None:   # the caller has made `device` current
            nb = 0 if d == 64 else workspace_size(B, H, Lq, Lk, d, variant=int(variant))
            _ws_sizes[key] = nb
        if nb == 0:
            return None, 0, 0
        workspace = torch.empty(nb, dtype=torch.uint8, device=device)
        if stream is not None:
            # the block returns to the pool only once work on `stream` is done
            workspace.record_stream(stream if isinstance(stream, torch.cuda.Stream)
                                    else torch.cuda.ExternalStream(int(stream), device=device))
    if (not isinstance(workspace, torch.Tensor) or workspace.dtype != torch.uint8
            or workspace.device != device or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous uint8 tensor on the inputs' device")
    return workspace, workspace.data_ptr(), workspace.numel()


def forward_ws_ptr(q: int, k: int, v: int, out: int, B: int, H: int, Lq: int, Lk: int, d: int,
                   scale: float, workspace: int, workspace_bytes: int, stream=0) -> int:
    """Raw C-ABI call of dit_attn_forward_ws with integer device pointers; returns the status."""
    s = stream if isinstance(stream, ctypes.c_void_p) else ctypes.c_void_p(int(stream))
    return _load().dit_attn_forward_ws(ctypes.c_void_p(q), ctypes.c_void_p(k), ctypes.c_void_p(v),
                                       ctypes.c_void_p(out), B, H, Lq, Lk, d,
                                       ctypes.c_float(scale), ctypes.c_void_p(workspace),
                                       ctypes.c_longlong(workspace_bytes), s)


def forward(q, k, v, scale: float | None = None, out=None, stream=None, workspace="auto"):
    """out = softmax(q k^T * scale) v over every (batch, head); bf16 in and out.

    q: [B, H, Lq, d], k and v: [B, H, Lk, d], contiguous bf16 CUDA tensors on
    one device; d is 64 or 128; scale defaults to 1/sqrt(d).  Enqueued on
    ``stream`` (default: torch's current stream); returns ``out``.
    ``workspace``: "auto" (default) gives the split tail the scratch it asks
    for, None runs without splitting, or pass a uint8 CUDA tensor.
    """
    import torch
    B, H, Lq, Lk, d = _check_qkv(q, k, v, (torch.bfloat16,))
    out = _out_like(out, q, (B, H, Lq, d))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with torch.cuda.device(q.device):
        ws, ws_ptr, ws_bytes = _workspace(workspace, q.device, B, H, Lq, Lk, d, 0, stream)
        rc = forward_ws_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                            B, H, Lq, Lk, d, float(scale), ws_ptr, ws_bytes,
                            _stream_handle(stream))
    if rc:
        raise DitAttnError(rc, "dit_attn_forward_ws")
    return out


def rmsnorm_ptr(x: int, y: int, weight: int, rows: int, d: int, eps: float, stream=0) -> int:
    """Raw C-ABI call of dit_attn_rmsnorm with integer device pointers; returns the status."""
    s = stream if isinstance(stream, ctypes.c_void_p) else ctypes.c_void_p(int(stream))
    return _load().dit_attn_rmsnorm(ctypes.c_void_p(x), ctypes.c_void_p(y),
                                    ctypes.c_void_p(weight) if weight else None,
                                    ctypes.c_longlong(rows), d, ctypes.c_float(eps), s)


def rmsnorm(x, weight=None, eps: float = 1e-6, out=None, stream=None):
    """out = bf16(x / sqrt(mean(x^2, last dim) + eps) * weight) for a bf16 CUDA tensor
    whose last dimension (64 or 128) is the head dimension; ``out=x`` works in place."""
    import torch
    if not isinstance(x, torch.Tensor) or x.dtype != torch.bfloat16 or not x.is_cuda:
        raise TypeError("x must be a bfloat16 CUDA tensor")
    if not x.is_contiguous() or x.dim() < 1:
        raise ValueError("x must be contiguous")
    d = x.shape[-1]
    if weight is not None and (weight.dtype != torch.bfloat16 or tuple(weight.shape) != (d,)
                               or not weight.is_contiguous() or weight.device != x.device):
        raise ValueError("weight must be a contiguous bf16 [d] tensor on x's device")
    if out is None:
        out = torch.empty_like(x)
    elif (out.dtype != torch.bfloat16 or out.shape != x.shape or not out.is_contiguous()
          or out.device != x.device):
        raise ValueError("out must be a contiguous bf16 tensor shaped like x on x's device")
    with torch.cuda.device(x.device):
        rc = rmsnorm_ptr(x.data_ptr(), out.data_ptr(), weight.data_ptr() if weight is not None else 0,
                         x.numel() // d, d, float(eps), _stream_handle(stream))
    if rc:
        raise DitAttnError(rc, "dit_attn_rmsnorm")
    return out


def forward_qk8_ptr(q8: int, k8: int, v: int, out: int, B: int, H: int, Lq: int, Lk: int, d: int,
                    scale: float, q_scale: float, k_scale: float, stream=0) -> int:
    """Raw C-ABI call of dit_attn_forward_qk8 with integer device pointers; returns the status."""
    s = stream if isinstance(stream, ctypes.c_void_p) else ctypes.c_void_p(int(stream))
    return _load().dit_attn_forward_qk8(ctypes.c_void_p(q8), ctypes.c_void_p(k8),
                                        ctypes.c_void_p(v), ctypes.c_void_p(out), B, H, Lq, Lk, d,
                                        ctypes.c_float(scale), ctypes.c_float(q_scale),
                                        ctypes.c_float(k_scale), s)


def forward_qk8_ws_ptr(q8: int, k8: int, v: int, out: int, B: int, H: int, Lq: int, Lk: int,
                       d: int, scale: float, q_scale: float, k_scale: float, workspace: int,
                       workspace_bytes: int, stream=0) -> int:
    """Raw C-ABI call of dit_attn_forward_qk8_ws with integer device pointers."""
    s = stream if isinstance(stream, ctypes.c_void_p) else ctypes.c_void_p(int(stream))
    return _load().dit_attn_forward_qk8_ws(ctypes.c_void_p(q8), ctypes.c_void_p(k8),
                                           ctypes.c_void_p(v), ctypes.c_void_p(out), B, H, Lq,
                                           Lk, d, ctypes.c_float(scale), ctypes.c_float(q_scale),
                                           ctypes.c_float(k_scale), ctypes.c_void_p(workspace),
                                           ctypes.c_longlong(workspace_bytes), s)


def forward_qk8(q8, k8, v, q_scale: float, k_scale: float, scale: float | None = None, out=None,
                stream=None, workspace="auto"):
    """out = softmax((q_scale*q8)(k_scale*k8)^T * scale) v with e4m3 q8, k8.

    q8: [B, H, Lq, 128], k8: [B, H, Lk, 128], contiguous CUDA tensors of e4m3
    codes (torch.float8_e4m3fn or uint8); v: [B, H, Lk, 128] bf16.  scale
    defaults to 1/sqrt(d); ``workspace`` as for forward.  Returns the bf16
    output ``out``.
    """
    import torch
    B, H, Lq, Lk, d = _check_qkv(q8, k8, v, (torch.float8_e4m3fn, torch.uint8))
    out = _out_like(out, v, (B, H, Lq, d))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with torch.cuda.device(v.device):
        ws, ws_ptr, ws_bytes = _workspace(workspace, v.device, B, H, Lq, Lk, d, 1, stream)
        rc = forward_qk8_ws_ptr(q8.data_ptr(), k8.data_ptr(), v.data_ptr(), out.data_ptr(),
                                B, H, Lq, Lk, d, float(scale), float(q_scale), float(k_scale),
                                ws_ptr, ws_bytes, _stream_handle(stream))
    if rc:
        raise DitAttnError(rc, "dit_attn_forward_qk8_ws")
    return out


def rmsnorm_e4m3_ptr(x: int, y8: int, weight: int, rows: int, d: int, eps: float,
                     out_scale: float, stream=0) -> int:
    """Raw C-ABI call of dit_attn_rmsnorm_e4m3 with integer device pointers; returns the status."""
    s = stream if isinstance(stream, ctypes.c_void_p) else ctypes.c_void_p(int(stream))
    return _load().dit_attn_rmsnorm_e4m3(ctypes.c_void_p(x), ctypes.c_void_p(y8),
                                         ctypes.c_void_p(weight) if weight else None,
                                         ctypes.c_longlong(rows), d, ctypes.c_float(eps),
                                         ctypes.c_float(out_scale), s)


def rmsnorm_e4m3(x, out_scale: float, weight=None, eps: float = 1e-6, out=None, stream=None):
    """out = e4m3(x / sqrt(mean(x^2, last dim) + eps) * weight * out_scale), saturating at 448,
    for a bf16 CUDA tensor whose last dimension (64 or 128) is the head dimension.
    Returns a torch.float8_e4m3fn tensor shaped like x (or fills ``out``)."""
    import torch
    if not isinstance(x, torch.Tensor) or x.dtype != torch.bfloat16 or not x.is_cuda:
        raise TypeError("x must be a bfloat16 CUDA tensor")
    if not x.is_contiguous() or x.dim() < 1:
        raise ValueError("x must be contiguous")
    d = x.shape[-1]
    if weight is not None and (weight.dtype != torch.bfloat16 or tuple(weight.shape) != (d,)
                               or not weight.is_contiguous() or weight.device != x.device):
        raise ValueError("weight must be a contiguous bf16 [d] tensor on x's device")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.float8_e4m3fn, device=x.device)
    elif (out.dtype not in (torch.float8_e4m3fn, torch.uint8) or out.shape != x.shape
          or not out.is_contiguous() or out.device != x.device):
        raise ValueError("out must be a contiguous e4m3 (or uint8) tensor shaped like x")
    with torch.cuda.device(x.device):
        rc = rmsnorm_e4m3_ptr(x.data_ptr(), out.data_ptr(),
                              weight.data_ptr() if weight is not None else 0,
                              x.numel() // d, d, float(eps), float(out_scale),
                              _stream_handle(stream))
    if rc:
        raise DitAttnError(rc, "dit_attn_rmsnorm_e4m3")
    return out


def forward_noalloc_ptr(q: int, k: int, v: int, out: int, B: int, H: int, Lq: int, Lk: int, d: int,
                        scale: float, stream=0) -> int:
    """Raw C-ABI call of dit_attn_forward_noalloc with integer device pointers."""
    s = stream if isinstance(stream, ctypes.c_void_p) else ctypes.c_void_p(int(stream))
    return _load().dit_attn_forward_noalloc(ctypes.c_void_p(q), ctypes.c_void_p(k),
                                            ctypes.c_void_p(v), ctypes.c_void_p(out), B, H, Lq,
                                            Lk, d, ctypes.c_float(scale), s)


def forward_noalloc(q, k, v, out, scale: float | None = None, stream=None):
    """forward() with the split tail's scratch held by the library: no memory is
    allocated by the call (``out`` must be given).  Calls must not overlap."""
    import torch
    B, H, Lq, Lk, d = _check_qkv(q, k, v, (torch.bfloat16,))
    if out is None:
        raise ValueError("forward_noalloc needs an output tensor")
    out = _out_like(out, q, (B, H, Lq, d))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with torch.cuda.device(q.device):
        rc = forward_noalloc_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                 B, H, Lq, Lk, d, float(scale), _stream_handle(stream))
    if rc:
        raise DitAttnError(rc, "dit_attn_forward_noalloc")
    return out


def forward_fp8_ptr(q8: int, k8: int, v8: int, out: int, B: int, H: int, Lq: int, Lk: int, d: int,
                    scale: float, q_scale: float, k_scale: float, v_scale: float, stream=0) -> int:
    """Raw C-ABI call of dit_attn_forward_fp8 with integer device pointers; returns the status."""
    s = stream if isinstance(stream, ctypes.c_void_p) else ctypes.c_void_p(int(stream))
    return _load().dit_attn_forward_fp8(ctypes.c_void_p(q8), ctypes.c_void_p(k8),
                                        ctypes.c_void_p(v8), ctypes.c_void_p(out), B, H, Lq, Lk,
                                        d, ctypes.c_float(scale), ctypes.c_float(q_scale),
                                        ctypes.c_float(k_scale), ctypes.c_float(v_scale), s)


def forward_fp8_ws_ptr(q8: int, k8: int, v8: int, out: int, B: int, H: int, Lq: int, Lk: int,
                       d: int, scale: float, q_scale: float, k_scale: float, v_scale: float,
                       workspace: int, workspace_bytes: int, stream=0) -> int:
    """Raw C-ABI call of dit_attn_forward_fp8_ws with integer device pointers."""
    s = stream if isinstance(stream, ctypes.c_void_p) else ctypes.c_void_p(int(stream))
    return _load().dit_attn_forward_fp8_ws(ctypes.c_void_p(q8), ctypes.c_void_p(k8),
                                           ctypes.c_void_p(v8), ctypes.c_void_p(out), B, H, Lq,
                                           Lk, d, ctypes.c_float(scale), ctypes.c_float(q_scale),
                                           ctypes.c_float(k_scale), ctypes.c_float(v_scale),
                                           ctypes.c_void_p(workspace),
                                           ctypes.c_longlong(workspace_bytes), s)


def forward_fp8(q8, k8, v8, q_scale: float, k_scale: float, v_scale: float,
                scale: float | None = None, out=None, stream=None, workspace="auto"):
    """out = v_scale * softmax((q_scale*q8)(k_scale*k8)^T * scale) v8, all three e4m3,
    with the probabilities rounded to e4m3 before the product with v8.

    q8: [B, H, Lq, 128], k8 and v8: [B, H, Lk, 128], contiguous CUDA tensors of
    e4m3 codes (torch.float8_e4m3fn or uint8).  scale defaults to 1/sqrt(d);
    ``workspace`` as for forward.  Returns the bf16 output ``out``.
    """
    import torch
    e4m3 = (torch.float8_e4m3fn, torch.uint8)
    B, H, Lq, Lk, d = _check_qkv(q8, k8, v8, e4m3, e4m3)
    out = _out_like(out, v8, (B, H, Lq, d))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with torch.cuda.device(v8.device):
        ws, ws_ptr, ws_bytes = _workspace(workspace, v8.device, B, H, Lq, Lk, d, 2, stream)
        rc = forward_fp8_ws_ptr(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), out.data_ptr(),
                                B, H, Lq, Lk, d, float(scale), float(q_scale), float(k_scale),
                                float(v_scale), ws_ptr, ws_bytes, _stream_handle(stream))
    if rc:
        raise DitAttnError(rc, "dit_attn_forward_fp8_ws")
    return out


def quantize_e4m3_ptr(x: int, y8: int, n: int, out_scale: float, stream=0) -> int:
    """Raw C-ABI call of dit_attn_quantize_e4m3 with integer device pointers; returns the status."""
    s = stream if isinstance(stream, ctypes.c_void_p) else ctypes.c_void_p(int(stream))
    return _load().dit_attn_quantize_e4m3(ctypes.c_void_p(x), ctypes.c_void_p(y8),
                                          ctypes.c_longlong(n), ctypes.c_float(out_scale), s)


def quantize_e4m3(x, out_scale: float, out=None, stream=None):
    """out = e4m3(x * out_scale) (fp32 product, nearest even, saturating at 448) for a
    contiguous bf16 CUDA tensor; returns a torch.float8_e4m3fn tensor shaped like x
    (or fills ``out``).  The dequantisation scale to hand the forward is 1/out_scale."""
    import torch
    if not isinstance(x, torch.Tensor) or x.dtype != torch.bfloat16 or not x.is_cuda:
        raise TypeError("x must be a bfloat16 CUDA tensor")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.float8_e4m3fn, device=x.device)
    elif (out.dtype not in (torch.float8_e4m3fn, torch.uint8) or out.shape != x.shape
          or not out.is_contiguous() or out.device != x.device):
        raise ValueError("out must be a contiguous e4m3 (or uint8) tensor shaped like x")
    with torch.cuda.device(x.device):
        rc = quantize_e4m3_ptr(x.data_ptr(), out.data_ptr(), x.numel(), float(out_scale),
                               _stream_handle(stream))
    if rc:
        raise DitAttnError(rc, "dit_attn_quantize_e4m3")
    return out

"""Python binding of libfa.so (the C ABI in include/fa.h).

Argument marshalling only: torch tensors become device pointers and sizes,
the ``stream`` keyword (a torch CUDA stream; by default the current one)
becomes the library's stream argument, and non-OK status codes become
``FaError``.  Every step of attention runs in the library's CUDA kernels;
there is no other code path.  PyTorch supplies device memory (outputs and
workspaces, allocated on the stream the call runs on) and streams.
"""

from __future__ import annotations

import contextlib
import ctypes
import math
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa.so")

FA_OK, FA_ERR_INVALID, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)
FA_DTYPE_F32, FA_DTYPE_BF16 = 0, 1

EXPORTS = ("fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_bwd_static_workspace", "fa_fwd_key_major",
           "fa_fwd_key_major_workspace_bytes", "fa_fwd_f32_3xtf32", "fa_fwd_f32_3xtf32_workspace_bytes",
           "fa_last_device_status", "fa_set_wait_limit_us", "fa_selftest_wait_timeout", "fa_status_string",
           "fa_version")


class FaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {lib.fa_status_string(status).decode()}")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m exact_tiled_attention_02_gb300.build` "
                          "(or __graft_entry__.build()); there is no fallback implementation")
    L = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
    L.fa_fwd.restype = i
    L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, sz, vp]
    L.fa_bwd.restype = i
    L.fa_bwd_static_workspace.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
    L.fa_bwd_static_workspace.restype = i
    L.fa_bwd_workspace_bytes.argtypes = [i, i, i, i]
    L.fa_bwd_workspace_bytes.restype = sz
    L.fa_fwd_key_major.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, sz, vp]
    L.fa_fwd_key_major.restype = i
    L.fa_fwd_key_major_workspace_bytes.argtypes = [i, i, i, i]
    L.fa_fwd_key_major_workspace_bytes.restype = sz
    L.fa_fwd_f32_3xtf32.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, sz, vp]
    L.fa_fwd_f32_3xtf32.restype = i
    L.fa_fwd_f32_3xtf32_workspace_bytes.argtypes = [i, i, i, i]
    L.fa_fwd_f32_3xtf32_workspace_bytes.restype = sz
    L.fa_last_device_status.argtypes = [vp]
    L.fa_last_device_status.restype = i
    L.fa_set_wait_limit_us.argtypes = [ctypes.c_longlong]
    L.fa_set_wait_limit_us.restype = ctypes.c_longlong
    L.fa_selftest_wait_timeout.argtypes = [i, vp]
    L.fa_selftest_wait_timeout.restype = i
    L.fa_status_string.argtypes = [i]
    L.fa_status_string.restype = ctypes.c_char_p
    L.fa_version.argtypes = []
    L.fa_version.restype = i
    return L


lib = _load()


def _torch():
    import torch
    return torch


def _stream_ptr(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _alloc_on(stream):
    """Context for the tensors a call allocates (outputs, workspace): on the
    stream its kernels run on.  The caching allocator hands a freed block out
    again in the order of the stream it was allocated on; a workspace
    allocated on the current stream and dropped on return, while the kernels
    still run on another stream, could otherwise be reused at once."""
    torch = _torch()
    return contextlib.nullcontext() if stream is None else torch.cuda.stream(stream)


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return FA_DTYPE_BF16
    if t.dtype == torch.float32:
        return FA_DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}: use torch.bfloat16 or torch.float32")


def _check_qkv(*ts):
    ref = ts[0]
    if ref.dim() != 4:
        raise ValueError("tensors must be [B, H, N, d]")
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")
        if t.shape != ref.shape or t.dtype != ref.dtype or t.device != ref.device:
            raise ValueError("q, k, v (and o, dO, grads) must share shape, dtype and device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous [B, H, N, d]")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def fa_status_string(status: int) -> str:
    return lib.fa_status_string(int(status)).decode()


def fa_version() -> int:
    return lib.fa_version()


def fa_set_wait_limit_us(limit_us: int) -> int:
    return lib.fa_set_wait_limit_us(int(limit_us))


def fa_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return lib.fa_bwd_workspace_bytes(B, H, N, d)


def fa_fwd_key_major_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return lib.fa_fwd_key_major_workspace_bytes(B, H, N, d)


def fa_fwd_f32_3xtf32_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return lib.fa_fwd_f32_3xtf32_workspace_bytes(B, H, N, d)


def fa_last_device_status(stream=None) -> int:
    return lib.fa_last_device_status(_stream_ptr(stream))


def fa_selftest_wait_timeout(limit_us: int, stream=None) -> int:
    return lib.fa_selftest_wait_timeout(int(limit_us), _stream_ptr(stream))


def fa_fwd(q, k, v, scale: float | None = None, window: int = 0, o=None, lse=None, want_lse: bool = True,
           stream=None):
    """O = softmax(Q K^T * scale) V on the GPU; returns ``(o, lse)``.

    ``q, k, v``: contiguous [B, H, N, d] bf16 (d in {64, 96, 128, 256}) or float32
    (d <= 128) CUDA tensors.  ``scale`` defaults to 1/sqrt(d).  ``window``:
    0 = unmasked, else the odd full width of the local window.  ``o``/``lse``
    may be given to write into existing buffers; ``lse`` is float32 [B, H, N]
    (None when ``want_lse`` is false and none is given).
    """
    torch = _torch()
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with _alloc_on(stream):
        if o is None:
            o = torch.empty_like(q)
        if lse is None and want_lse:
            lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    _check_qkv(q, o)
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous() or lse.numel() != B * H * N):
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor")
    st = lib.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(scale), int(window),
                    _dtype_code(q), _stream_ptr(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd")
    return o, lse


def fa_fwd_key_major(q, k, v, scale: float | None = None, window: int = 0, o=None, lse=None, want_lse: bool = True,
                     workspace=None, stream=None):
    """The forward pass in the key-major loop order (a comparison schedule,
    bf16 with d = 64 or 128); same results as ``fa_fwd``.  The fp32 workspace
    for the running statistics is taken from ``workspace`` (a CUDA uint8
    tensor of at least ``fa_fwd_key_major_workspace_bytes`` bytes) or
    allocated here with torch."""
    torch = _torch()
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with _alloc_on(stream):
        if o is None:
            o = torch.empty_like(q)
        if lse is None and want_lse:
            lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
        if workspace is None:
            workspace = torch.empty(fa_fwd_key_major_workspace_bytes(B, H, N, d), device=q.device, dtype=torch.uint8)
    _check_qkv(q, o)
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous() or lse.numel() != B * H * N):
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor")
    st = lib.fa_fwd_key_major(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(scale), int(window),
                              _dtype_code(q), _ptr(workspace), workspace.numel() * workspace.element_size(),
                              _stream_ptr(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_key_major")
    return o, lse


def fa_fwd_f32_3xtf32(q, k, v, scale: float | None = None, window: int = 0, o=None, lse=None, want_lse: bool = True,
                      workspace=None, stream=None):
    """float32 forward on the tensor cores by the 3xTF32 split (d <= 64);
    same operation and outputs as ``fa_fwd`` on float32 tensors.  The
    workspace (split copies of Q, K, V) is taken from ``workspace`` (a CUDA
    uint8 tensor of at least ``fa_fwd_f32_3xtf32_workspace_bytes`` bytes) or
    allocated here with torch."""
    torch = _torch()
    _check_qkv(q, k, v)
    if q.dtype != torch.float32:
        raise TypeError("fa_fwd_f32_3xtf32 takes float32 tensors")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with _alloc_on(stream):
        if o is None:
            o = torch.empty_like(q)
        if lse is None and want_lse:
            lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
        if workspace is None:
            workspace = torch.empty(fa_fwd_f32_3xtf32_workspace_bytes(B, H, N, d), device=q.device, dtype=torch.uint8)
    _check_qkv(q, o)
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous() or lse.numel() != B * H * N):
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor")
    st = lib.fa_fwd_f32_3xtf32(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(scale), int(window),
                               _ptr(workspace), workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_f32_3xtf32")
    return o, lse


def fa_bwd(q, k, v, o, lse, do, scale: float | None = None, window: int = 0, dq=None, dk=None, dv=None,
           workspace=None, stream=None):
    """Gradients (dQ, dK, dV) of the forward above, by recomputation.

    ``o`` and ``lse`` are the forward's outputs; ``do`` is dL/dO.  The
    workspace (float32 dQ accumulator + row sums) is taken from ``workspace``
    (a CUDA uint8 tensor of at least ``fa_bwd_workspace_bytes`` bytes) or
    allocated here with torch.
    """
    torch = _torch()
    _check_qkv(q, k, v, o, do)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if lse.dtype != torch.float32 or not lse.is_contiguous() or lse.numel() != B * H * N:
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor")
    need = fa_bwd_workspace_bytes(B, H, N, d)
    with _alloc_on(stream):
        dq = torch.empty_like(q) if dq is None else dq
        dk = torch.empty_like(q) if dk is None else dk
        dv = torch.empty_like(q) if dv is None else dv
        if workspace is None:
            workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    _check_qkv(q, dq, dk, dv)
    st = lib.fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                    B, H, N, d, float(scale), int(window), _dtype_code(q), _ptr(workspace),
                    workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    if st != FA_OK:
        raise FaError(st, "fa_bwd")
    return dq, dk, dv


def fa_bwd_static_workspace(q, k, v, o, lse, do, dq, dk, dv, scale: float | None = None, window: int = 0,
                            stream=None):
    """fa_bwd without a workspace argument, for callers that cannot allocate
    device memory: the library's fixed 64 MiB scratch array stands in for the
    workspace, and neither this wrapper nor the library allocates anything
    (the caller passes the dq, dk, dv outputs).  Calls that overlap on the GPU
    share that array and race; problems needing more than 64 MiB of workspace
    raise FaError(FA_ERR_UNSUPPORTED)."""
    torch = _torch()
    _check_qkv(q, k, v, o, do, dq, dk, dv)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if lse.dtype != torch.float32 or not lse.is_contiguous() or lse.numel() != B * H * N:
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor")
    st = lib.fa_bwd_static_workspace(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk),
                                     _ptr(dv), B, H, N, d, float(scale), int(window), _dtype_code(q),
                                     _stream_ptr(stream))
    if st != FA_OK:
        raise FaError(st, "fa_bwd_static_workspace")
    return dq, dk, dv

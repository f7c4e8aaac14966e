"""ctypes binding to libfa2_gb300.so (declared in include/fa2.h).

Argument marshalling only: shape/dtype checks, raw pointers, the current CUDA
stream.  Every step of the forward pass runs in the library's kernels; there
is no fallback.  Importing this module raises ImportError if the library has
not been built (``python -m io_aware_exact_fa2_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

# FA2_NOALLOC_SCRATCH_BYTES of include/fa2.h: the fixed workspace of fa2_fwd_noalloc
NOALLOC_SCRATCH_BYTES = 48 << 20

STATUS = {0: "FA2_OK", 1: "FA2_ERR_INVALID_ARG", 2: "FA2_ERR_UNSUPPORTED",
          3: "FA2_ERR_CUDA", 4: "FA2_ERR_TIMEOUT"}


class Fa2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where} failed: {STATUS.get(status, status)}")


def library_path() -> str:
    return LIB_PATH


def load_library() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"CUDA library {LIB_PATH} is missing: build it with "
            "`python -m io_aware_exact_fa2_gb300.build` (there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa2_fwd.restype = i
    lib.fa2_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    lib.fa2_fwd_from_host.restype = i
    lib.fa2_fwd_from_host.argtypes = [vp] * 10 + [i, i, i, i, i, i, f, vp]
    lib.fa2_workspace_size.restype = i
    lib.fa2_workspace_size.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
    lib.fa2_fwd_ws.restype = i
    lib.fa2_fwd_ws.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp, ctypes.c_size_t, vp]
    lib.fa2_fwd_window.restype = i
    lib.fa2_fwd_window.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    ll3 = ctypes.POINTER(ctypes.c_longlong)
    lib.fa2_fwd_ex.restype = i
    lib.fa2_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ll3, ll3, ll3, ll3, i, i, f, vp,
                               ctypes.c_size_t, vp]
    lib.fa2_bwd_ex.restype = i
    lib.fa2_bwd_ex.argtypes = [vp] * 9 + [i, i, i, i, i] + [ll3] * 8 + [i, i, f, vp, ctypes.c_size_t, vp]
    lib.fa2_fwd_fp8.restype = i
    lib.fa2_fwd_fp8.argtypes = [vp] * 8 + [i, i, i, i, i, i, f, vp, ctypes.c_size_t, vp]
    lib.fa2_fwd_noalloc.restype = i
    lib.fa2_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    lib.fa2_bwd_workspace_size.restype = i
    lib.fa2_bwd_workspace_size.argtypes = [i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
    lib.fa2_bwd.restype = i
    lib.fa2_bwd.argtypes = [vp] * 9 + [i, i, i, i, i, i, f, vp, ctypes.c_size_t, vp]
    lib.fa2_bwd_window.restype = i
    lib.fa2_bwd_window.argtypes = [vp] * 9 + [i, i, i, i, i, i, f, vp, ctypes.c_size_t, vp]
    lib.fa2_get_device_error.restype = i
    lib.fa2_get_device_error.argtypes = [vp, ctypes.POINTER(i)]
    lib.fa2_status_string.restype = ctypes.c_char_p
    lib.fa2_status_string.argtypes = [i]
    lib.fa2_version.restype = i
    lib.fa2_version.argtypes = []
    return lib


_lib = load_library()


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check_shapes(q, k, v, o, lse):
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D (B, H, L, D)")
    B, H, Lq, D = q.shape
    if tuple(k.shape[:2]) != (B, H) or k.shape[3] != D or tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)}")
    if tuple(o.shape) != (B, H, Lq, D) or tuple(lse.shape) != (B, H, Lq):
        raise ValueError("o must be (B, H, Lq, D) and lse (B, H, Lq)")
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16), ("v", v, torch.bfloat16),
                        ("o", o, torch.bfloat16), ("lse", lse, torch.float32)):
        if t.dtype != dt:
            raise TypeError(f"{name} must be {dt}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    return B, H, Lq, k.shape[2], D


def fa2_workspace_size(B: int, H: int, Lq: int, Lk: int, D: int, causal: bool, device: int = 0) -> int:
    """Bytes of workspace fa2_fwd_ws needs on `device` (0 when the pass uses none)."""
    n = ctypes.c_size_t(0)
    st = _lib.fa2_workspace_size(B, H, Lq, Lk, D, int(bool(causal)), int(device), ctypes.byref(n))
    if st != 0:
        raise Fa2Error(st, "fa2_workspace_size")
    return int(n.value)


def fa2_workspace(q, k, causal: bool):
    """A zero-filled uint8 CUDA tensor sized for fa2_fwd_ws on q's problem (None if not needed)."""
    import torch
    B, H, Lq, D = q.shape
    n = fa2_workspace_size(B, H, Lq, k.shape[2], D, causal, q.device.index or 0)
    return torch.zeros(n, dtype=torch.uint8, device=q.device) if n else None


def fa2_fwd(q, k, v, o, lse, causal: bool, scale: float | None = None, stream=None,
            workspace=None) -> None:
    """Forward pass on CUDA tensors: writes o (bf16) and lse (fp32, natural log).

    With `workspace` (from fa2_workspace) a non-causal pass balances its key
    tiles evenly over the SMs (fa2_fwd_ws); without it, whole query tiles are
    scheduled (fa2_fwd).
    """
    B, H, Lq, Lk, D = _check_shapes(q, k, v, o, lse)
    for t in (q, k, v, o, lse):
        if not t.is_cuda or t.device != q.device:
            raise ValueError("all tensors must be on the same CUDA device")
    if scale is None:
        scale = D ** -0.5
    if workspace is None:
        st = _lib.fa2_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          B, H, Lq, Lk, D, int(bool(causal)), float(scale), _stream_handle(stream, q.device))
        where = "fa2_fwd"
    else:
        if not workspace.is_cuda or workspace.device != q.device:
            raise ValueError("workspace must be on q's CUDA device")
        st = _lib.fa2_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                             B, H, Lq, Lk, D, int(bool(causal)), float(scale), workspace.data_ptr(),
                             workspace.numel() * workspace.element_size(), _stream_handle(stream, q.device))
        where = "fa2_fwd_ws"
    if st != 0:
        raise Fa2Error(st, where)


def fa2_fwd_fp8(q8, k8, v8, descale_q, descale_k, descale_v, o, lse, causal: bool, scale: float | None = None,
                stream=None, workspace=None) -> None:
    """Forward pass on e4m3 inputs (fa2_fwd_fp8): q8 (B, H, Lq, 128), k8 and v8 (B, H, Lk, 128)
    float8_e4m3fn CUDA tensors, each with a float32 (B, H) CUDA tensor of descales (the real
    input is the stored value times its head's descale).  Writes o (bf16) and lse (fp32).
    `workspace` as for fa2_fwd (fa2_workspace on a D = 128 problem of the same shape)."""
    import torch
    if q8.dim() != 4 or k8.dim() != 4 or v8.dim() != 4:
        raise ValueError("q8, k8, v8 must be 4-D (B, H, L, D)")
    B, H, Lq, D = q8.shape
    Lk = k8.shape[2]
    if tuple(k8.shape) != (B, H, Lk, D) or tuple(v8.shape) != (B, H, Lk, D):
        raise ValueError(f"shape mismatch: q {tuple(q8.shape)} k {tuple(k8.shape)} v {tuple(v8.shape)}")
    if tuple(o.shape) != (B, H, Lq, D) or tuple(lse.shape) != (B, H, Lq):
        raise ValueError("o must be (B, H, Lq, D) and lse (B, H, Lq)")
    for name, t, dt in (("q8", q8, torch.float8_e4m3fn), ("k8", k8, torch.float8_e4m3fn),
                        ("v8", v8, torch.float8_e4m3fn), ("o", o, torch.bfloat16), ("lse", lse, torch.float32),
                        ("descale_q", descale_q, torch.float32), ("descale_k", descale_k, torch.float32),
                        ("descale_v", descale_v, torch.float32)):
        if t.dtype != dt:
            raise TypeError(f"{name} must be {dt}, got {t.dtype}")
        if not t.is_contiguous() or not t.is_cuda or t.device != q8.device:
            raise ValueError(f"{name} must be contiguous and on q8's CUDA device")
    for name, t in (("descale_q", descale_q), ("descale_k", descale_k), ("descale_v", descale_v)):
        if t.numel() != B * H:
            raise ValueError(f"{name} must hold one value per (batch, head)")
    if scale is None:
        scale = D ** -0.5
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = _lib.fa2_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), descale_q.data_ptr(), descale_k.data_ptr(),
                          descale_v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Lq, Lk, D, int(bool(causal)),
                          float(scale), ws_ptr, ws_bytes, _stream_handle(stream, q8.device))
    if st != 0:
        raise Fa2Error(st, "fa2_fwd_fp8")


def fa2_fwd_window(q, k, v, o, lse, window: int, scale: float | None = None, stream=None) -> None:
    """Causal forward restricted to the sliding window i - window <= j <= i (Lq <= Lk)."""
    B, H, Lq, Lk, D = _check_shapes(q, k, v, o, lse)
    for t in (q, k, v, o, lse):
        if not t.is_cuda or t.device != q.device:
            raise ValueError("all tensors must be on the same CUDA device")
    if scale is None:
        scale = D ** -0.5
    st = _lib.fa2_fwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                             B, H, Lq, Lk, D, int(window), float(scale), _stream_handle(stream, q.device))
    if st != 0:
        raise Fa2Error(st, "fa2_fwd_window")


def fa2_fwd_ex(q, k, v, o, lse, causal: bool, scale: float | None = None, window: int | None = None,
               workspace=None, stream=None) -> None:
    """Forward pass on strided (B, H, L, D) views (fa2_fwd_ex).

    q, k, v and o may be any views whose last dimension is contiguous and whose
    other strides are multiples of 8 elements -- e.g. `x.view(B, L, H, D).transpose(1, 2)`
    or slices of one packed QKV tensor.  lse must be contiguous (B, H, Lq).
    """
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4 or o.dim() != 4:
        raise ValueError("q, k, v, o must be 4-D (B, H, L, D) views")
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    if tuple(k.shape) != (B, H, Lk, D) or tuple(v.shape) != (B, H, Lk, D) or tuple(o.shape) != (B, H, Lq, D):
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)} o {tuple(o.shape)}")
    if tuple(lse.shape) != (B, H, Lq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 (B, H, Lq) tensor")
    arrays = []
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
        if t.stride(3) != 1:
            raise ValueError(f"{name}'s last dimension must be contiguous")
        if not t.is_cuda or t.device != q.device:
            raise ValueError("all tensors must be on the same CUDA device")
        arrays.append((ctypes.c_longlong * 3)(t.stride(0), t.stride(1), t.stride(2)))
    if scale is None:
        scale = D ** -0.5
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = _lib.fa2_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Lq, Lk, D,
                         *arrays, int(bool(causal)), -1 if window is None else int(window), float(scale),
                         ws_ptr, ws_bytes, _stream_handle(stream, q.device))
    if st != 0:
        raise Fa2Error(st, "fa2_fwd_ex")


def fa2_bwd_ex(q, k, v, o, lse, do, dq, dk, dv, causal: bool, scale: float | None = None,
               window: int | None = None, workspace=None, stream=None) -> None:
    """Backward pass on strided (B, H, L, D) views (fa2_bwd_ex): every tensor but lse may be
    a view whose last dimension is contiguous and whose other strides are multiples of 8
    elements; lse is the contiguous (B, H, Lq) output of the forward."""
    import torch
    tensors = (("q", q), ("k", k), ("v", v), ("o", o), ("do", do), ("dq", dq), ("dk", dk), ("dv", dv))
    if any(t.dim() != 4 for _, t in tensors):
        raise ValueError("q, k, v, o, do, dq, dk, dv must be 4-D (B, H, L, D) views")
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    for name, t in tensors:
        want = (B, H, Lk, D) if name in ("k", "v", "dk", "dv") else (B, H, Lq, D)
        if tuple(t.shape) != want:
            raise ValueError(f"{name} must have shape {want}, got {tuple(t.shape)}")
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
        if t.stride(3) != 1:
            raise ValueError(f"{name}'s last dimension must be contiguous")
        if not t.is_cuda or t.device != q.device:
            raise ValueError("all tensors must be on the same CUDA device")
    if tuple(lse.shape) != (B, H, Lq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 (B, H, Lq) tensor")
    arrays = [(ctypes.c_longlong * 3)(t.stride(0), t.stride(1), t.stride(2)) for _, t in tensors]
    if scale is None:
        scale = D ** -0.5
    if workspace is None:
        workspace = torch.empty(max(fa2_bwd_workspace_size(B, H, Lq, Lk, D), 16), dtype=torch.uint8,
                                device=q.device)
    st = _lib.fa2_bwd_ex(*(t.data_ptr() for _, t in tensors[:4]), lse.data_ptr(),
                         *(t.data_ptr() for _, t in tensors[4:]), B, H, Lq, Lk, D, *arrays,
                         int(bool(causal)), -1 if window is None else int(window), float(scale),
                         workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                         _stream_handle(stream, q.device))
    if st != 0:
        raise Fa2Error(st, "fa2_bwd_ex")


def fa2_fwd_noalloc(q, k, v, o, lse, causal: bool, scale: float | None = None, stream=None) -> None:
    """fa2_fwd with a workspace for callers that may not allocate device memory.

    Runs the same schedule as fa2_fwd(..., workspace=fa2_workspace(q, k, causal)),
    with the workspace taken from the library's fixed per-device scratch
    (NOALLOC_SCRATCH_BYTES) instead: neither this function nor the library
    allocates.  Calls that overlap on the GPU share that scratch and race.
    """
    B, H, Lq, Lk, D = _check_shapes(q, k, v, o, lse)
    for t in (q, k, v, o, lse):
        if not t.is_cuda or t.device != q.device:
            raise ValueError("all tensors must be on the same CUDA device")
    if scale is None:
        scale = D ** -0.5
    st = _lib.fa2_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                              B, H, Lq, Lk, D, int(bool(causal)), float(scale), _stream_handle(stream, q.device))
    if st == 2 and D in (64, 128, 256):
        need = fa2_workspace_size(B, H, Lq, Lk, D, causal, q.device.index or 0)
        raise Fa2Error(st, f"fa2_fwd_noalloc (needs {need} bytes of workspace, "
                           f"the fixed scratch holds {NOALLOC_SCRATCH_BYTES})")
    if st != 0:
        raise Fa2Error(st, "fa2_fwd_noalloc")


def fa2_bwd(q, k, v, o, lse, do, dq, dk, dv, causal: bool, scale: float | None = None, stream=None,
            workspace=None) -> None:
    """Backward pass on CUDA tensors: writes dq, dk, dv (bf16) from the forward's o and lse.

    workspace: a float32/uint8 CUDA tensor of at least fa2_bwd_workspace_size bytes
    (allocated here when not given).
    """
    _bwd(q, k, v, o, lse, do, dq, dk, dv, bool(causal), None, scale, stream, workspace)


def fa2_bwd_window(q, k, v, o, lse, do, dq, dk, dv, window: int, scale: float | None = None, stream=None,
                   workspace=None) -> None:
    """Backward pass of fa2_fwd_window (causal, query i sees keys i - window .. i; Lq <= Lk)."""
    _bwd(q, k, v, o, lse, do, dq, dk, dv, True, int(window), scale, stream, workspace)


def _bwd(q, k, v, o, lse, do, dq, dk, dv, causal, window, scale, stream, workspace) -> None:
    import torch
    B, H, Lq, Lk, D = _check_shapes(q, k, v, o, lse)
    for name, t, shape in (("do", do, (B, H, Lq, D)), ("dq", dq, (B, H, Lq, D)), ("dk", dk, (B, H, Lk, D)),
                           ("dv", dv, (B, H, Lk, D))):
        if tuple(t.shape) != shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor of shape {shape}")
    for t in (q, k, v, o, lse, do, dq, dk, dv):
        if not t.is_cuda or t.device != q.device:
            raise ValueError("all tensors must be on the same CUDA device")
    if scale is None:
        scale = D ** -0.5
    n = fa2_bwd_workspace_size(B, H, Lq, Lk, D)
    if workspace is None:
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr())
    ws = (workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_handle(stream, q.device))
    if window is None:
        st = _lib.fa2_bwd(*ptrs, B, H, Lq, Lk, D, int(causal), float(scale), *ws)
        name = "fa2_bwd"
    else:
        st = _lib.fa2_bwd_window(*ptrs, B, H, Lq, Lk, D, window, float(scale), *ws)
        name = "fa2_bwd_window"
    if st != 0:
        raise Fa2Error(st, name)


def fa2_bwd_workspace_size(B: int, H: int, Lq: int, Lk: int, D: int) -> int:
    n = ctypes.c_size_t(0)
    st = _lib.fa2_bwd_workspace_size(B, H, Lq, Lk, D, ctypes.byref(n))
    if st != 0:
        raise Fa2Error(st, "fa2_bwd_workspace_size")
    return int(n.value)


def fa2_fwd_from_host(q_host, k_host, v_host, o_host, lse_host, q_dev, k_dev, v_dev, o_dev, lse_dev,
                      causal: bool, scale: float | None = None, stream=None) -> None:
    """Host buffers in, host buffers out: copies and kernels overlapped over chunks of
    heads on the library's own streams, ordered after `stream`'s earlier work.

    The caller synchronises `stream` before reading o_host / lse_host.
    """
    B, H, Lq, Lk, D = _check_shapes(q_host, k_host, v_host, o_host, lse_host)
    _check_shapes(q_dev, k_dev, v_dev, o_dev, lse_dev)
    if scale is None:
        scale = D ** -0.5
    st = _lib.fa2_fwd_from_host(
        q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(), o_host.data_ptr(), lse_host.data_ptr(),
        q_dev.data_ptr(), k_dev.data_ptr(), v_dev.data_ptr(), o_dev.data_ptr(), lse_dev.data_ptr(),
        B, H, Lq, Lk, D, int(bool(causal)), float(scale), _stream_handle(stream, q_dev.device))
    if st != 0:
        raise Fa2Error(st, "fa2_fwd_from_host")


def fa2_get_device_error(stream=None) -> tuple[int, int]:
    """Synchronise, then read and clear the kernels' error word: (status, raw code)."""
    import torch
    detail = ctypes.c_int(0)
    st = _lib.fa2_get_device_error(_stream_handle(stream, torch.cuda.current_device()), ctypes.byref(detail))
    return st, detail.value


def fa2_status_string(status: int) -> str:
    return _lib.fa2_status_string(int(status)).decode()


def fa2_version() -> int:
    return _lib.fa2_version()

"""fp64 CPU oracle for exact scaled-dot-product attention (test infrastructure).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm are the only callers.  The CUDA
library never imports, links or calls anything here, and this package imports
nothing from the CUDA side.

The arithmetic lives in ``fa2_oracle.c`` (plain C, fp64, one materialised score
row and probability row per output row); this module only compiles it with gcc
and marshals arguments.  See that file's header for the definition it follows:

  O = softmax(scale * Q K^T [+ causal mask]) V,   LSE_i = ln sum_j exp(s_ij)

as stated in Olowookere, "FlashAttention-2 from scratch with a custom Triton
kernel" (section "The core idea: making attention IO-aware") and "Chapter 08:
Flash Attention -- blocked attention" (sections 3 and 4).

It also holds the backward definition of the same attention (Chapter 08,
section 6: Delta, the softmax backward, dV = P^T dO, dK = scale dS^T Q,
dQ = scale dS K), an fp64-input forward for numerical differentiation, and the
FP8 forward's reference: e4m3 inputs with per-(batch, head) descales, widened
exactly and fed to the same definition.

Every function here is pinned: the forward by ``tests/test_oracle_pins.py``
(closed forms, invariants, brute force, a library cross-check), the gradients
by ``tests/test_oracle_grad_pins.py`` (finite differences of the forward,
torch autograd, invariants, a closed form), the FP8 inputs by
``tests/test_oracle_fp8_pins.py`` (the e4m3 widening against torch's over all 256
codes, agreement with the bf16 path on shared values, descale laws, closed
forms); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa2_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libfa2_oracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, -O2, no fast-math). Returns the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.fa2_oracle_rows.restype = ctypes.c_int
            lib.fa2_oracle_rows.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.fa2_oracle_rows_w.restype = ctypes.c_int
            lib.fa2_oracle_rows_w.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_int64, ctypes.c_int, ctypes.c_int64, ctypes.c_double,
                ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.fa2_oracle_decode_bf16.restype = None
            lib.fa2_oracle_decode_bf16.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
            lib.fa2_oracle_decode_e4m3.restype = None
            lib.fa2_oracle_decode_e4m3.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
            lib.fa2_oracle_dequant_e4m3.restype = None
            lib.fa2_oracle_dequant_e4m3.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                                    ctypes.c_int64, ctypes.c_void_p]
            lib.fa2_oracle_rows_f64.restype = ctypes.c_int
            lib.fa2_oracle_rows_f64.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.fa2_oracle_max_threads.restype = ctypes.c_int
            lib.fa2_oracle_max_threads.argtypes = []
            i64, vp = ctypes.c_int64, ctypes.c_void_p
            lib.fa2_oracle_fwd_f64.restype = ctypes.c_int
            lib.fa2_oracle_fwd_f64.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, ctypes.c_int, i64,
                                               ctypes.c_double, vp, vp, ctypes.c_int]
            lib.fa2_oracle_bwd_f64.restype = ctypes.c_int
            lib.fa2_oracle_bwd_f64.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, ctypes.c_int, i64,
                                               ctypes.c_double, vp, vp, vp, vp, ctypes.c_int]
            _lib = lib
    return _lib


def _bf16_bits(t) -> np.ndarray:
    """bf16 torch tensor (CPU) -> contiguous uint16 numpy array of its bits."""
    import torch
    if t.dtype != torch.bfloat16:
        raise TypeError(f"oracle inputs must be bfloat16, got {t.dtype}")
    t = t.detach().to("cpu").contiguous()
    return t.view(torch.int16).numpy().view(np.uint16)


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp64 the way the oracle does internally."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().fa2_oracle_decode_bf16(bits.ctypes.data, out.ctypes.data, bits.size)
    return out


def _e4m3_bits(t) -> np.ndarray:
    """float8_e4m3fn (or uint8) torch tensor (CPU) -> contiguous uint8 numpy array of its bits."""
    import torch
    if t.dtype not in (torch.float8_e4m3fn, torch.uint8):
        raise TypeError(f"fp8 oracle inputs must be float8_e4m3fn, got {t.dtype}")
    t = t.detach().to("cpu").contiguous()
    return t.view(torch.uint8).numpy()


def decode_e4m3(bits: np.ndarray) -> np.ndarray:
    """Widen e4m3 bit patterns to fp64 the way the oracle does internally."""
    bits = np.ascontiguousarray(bits, dtype=np.uint8)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().fa2_oracle_decode_e4m3(bits.ctypes.data, out.ctypes.data, bits.size)
    return out


def dequant_e4m3(x, descale) -> np.ndarray:
    """Real values of an e4m3 tensor (B, H, L, D) with fp32 descales (B, H): stored value x descale."""
    bits = _e4m3_bits(x)
    B, H, L, D = bits.shape
    ds = np.ascontiguousarray(np.asarray(descale, dtype=np.float32).reshape(B * H))
    out = np.empty((B, H, L, D), dtype=np.float64)
    _load().fa2_oracle_dequant_e4m3(bits.ctypes.data, ds.ctypes.data, B * H, L * D, out.ctypes.data)
    return out


def rows_f64(q, k, v, causal: bool, scale: float, rows=None, threads: int = 0, window=None):
    """Attention rows of fp64 inputs (B, H, L, D): (o (n, D), lse (n,)), as attention_rows."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    if rows is None:
        rows = np.arange(B * H * Lq, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.size
    o = np.empty((n, D))
    lse = np.empty((n,))
    rc = _load().fa2_oracle_rows_f64(q.ctypes.data, k.ctypes.data, v.ctypes.data, B, H, Lq, Lk, D,
                                      int(bool(causal)), _window_arg(causal, window, Lq, Lk), float(scale),
                                      rows.ctypes.data if n else None, n, o.ctypes.data, lse.ctypes.data,
                                      int(threads))
    if rc != 0:
        raise RuntimeError(f"fa2_oracle_rows_f64 failed with code {rc}")
    return o, lse


def attention_fp8(q8, k8, v8, descale_q, descale_k, descale_v, causal: bool, scale: float, rows=None,
                  threads: int = 0):
    """Oracle for the FP8 forward: e4m3 q8 (B, H, Lq, D), k8, v8 (B, H, Lk, D) with fp32
    descales (B, H) each; the real inputs are stored value x descale ("Flash Attention:
    principles and implementation", section 4.3, names FlashAttention-3's FP8 mode; this
    per-(batch, head) descale is the reading taken).  Exact attention of the dequantised
    inputs in fp64.  rows: flat row ids (b*H + h)*Lq + i, None for all.
    Returns (o (n, D), lse (n,)) fp64."""
    q = dequant_e4m3(q8, descale_q)
    k = dequant_e4m3(k8, descale_k)
    v = dequant_e4m3(v8, descale_v)
    return rows_f64(q, k, v, causal, scale, rows, threads)


def max_threads() -> int:
    return int(_load().fa2_oracle_max_threads())


def _window_arg(causal: bool, window, Lq: int, Lk: int) -> int:
    """Sliding window (w, 0) of "Flash Attention: principles and implementation",
    section 6.3: needs causal, w >= 0, and Lq <= Lk so every row keeps key i."""
    if window is None:
        return -1
    if not causal or window < 0 or Lq > Lk:
        raise ValueError("a sliding window needs causal=True, window >= 0 and Lq <= Lk")
    return int(window)


def attention_rows(q, k, v, causal: bool, scale: float, rows=None,
                   return_p: bool = False, threads: int = 0, window=None):
    """Oracle output for selected rows.

    q: bf16 (B, H, Lq, D); k, v: bf16 (B, H, Lk, D) (torch CPU or CUDA tensors).
    rows: int64 array of flat row ids (b*H + h)*Lq + i; None means every row.
    window: None, or w for the causal sliding window i - w <= j <= i.
    Returns (o (n, D) fp64, lse (n,) fp64[, p (n, Lk) fp64]).
    """
    B, H, Lq, D = q.shape
    Bk, Hk, Lk, Dk = k.shape
    if (Bk, Hk, Dk) != (B, H, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("q, k, v shapes disagree")
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    if rows is None:
        rows = np.arange(B * H * Lq, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.size
    o = np.empty((n, D), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    p = np.empty((n, Lk), dtype=np.float64) if return_p else None
    w = _window_arg(causal, window, Lq, Lk)
    rc = _load().fa2_oracle_rows_w(
        qb.ctypes.data, kb.ctypes.data, vb.ctypes.data,
        B, H, Lq, Lk, D, int(bool(causal)), w, float(scale),
        rows.ctypes.data if n else None, n,
        o.ctypes.data, lse.ctypes.data, p.ctypes.data if return_p else None,
        int(threads))
    if rc != 0:
        raise RuntimeError(f"fa2_oracle_rows failed with code {rc}")
    return (o, lse, p) if return_p else (o, lse)


def attention(q, k, v, causal: bool, scale: float, threads: int = 0, window=None):
    """Full oracle output: O fp64 (B, H, Lq, D) and LSE fp64 (B, H, Lq)."""
    B, H, Lq, D = q.shape
    o, lse = attention_rows(q, k, v, causal, scale, None, False, threads, window)
    return o.reshape(B, H, Lq, D), lse.reshape(B, H, Lq)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def forward_f64(q, k, v, causal: bool, scale: float, threads: int = 0, window=None):
    """Forward definition on fp64 arrays (B, H, L, D): (O fp64 (B, H, Lq, D), LSE (B, H, Lq)).

    The same per-row arithmetic as ``attention`` without the bf16 widening, so a
    test can perturb the inputs by amounts bf16 cannot hold.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    o = np.empty((B, H, Lq, D))
    lse = np.empty((B, H, Lq))
    rc = _load().fa2_oracle_fwd_f64(q.ctypes.data, k.ctypes.data, v.ctypes.data, B, H, Lq, Lk, D,
                                     int(bool(causal)), _window_arg(causal, window, Lq, Lk), float(scale),
                                     o.ctypes.data, lse.ctypes.data, int(threads))
    if rc != 0:
        raise RuntimeError(f"fa2_oracle_fwd_f64 failed with code {rc}")
    return o, lse


def gradients_f64(q, k, v, do, causal: bool, scale: float, threads: int = 0, window=None):
    """Backward definition on fp64 arrays: (dQ, dK, dV, Delta) for L with dL/dO = do.

    Chapter 08, section 6: Delta = rowsum(dO * O), dS = P * (dO V^T - Delta),
    dV = P^T dO, dK = scale dS^T Q, dQ = scale dS K (see fa2_oracle.c).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    dq = np.empty((B, H, Lq, D))
    dk = np.empty((B, H, Lk, D))
    dv = np.empty((B, H, Lk, D))
    delta = np.empty((B, H, Lq))
    rc = _load().fa2_oracle_bwd_f64(q.ctypes.data, k.ctypes.data, v.ctypes.data, do.ctypes.data, B, H, Lq, Lk, D,
                                     int(bool(causal)), _window_arg(causal, window, Lq, Lk), float(scale),
                                     dq.ctypes.data, dk.ctypes.data,
                                     dv.ctypes.data, delta.ctypes.data, int(threads))
    if rc != 0:
        raise RuntimeError(f"fa2_oracle_bwd_f64 failed with code {rc}")
    return dq, dk, dv, delta


def gradients(q, k, v, do, causal: bool, scale: float, heads=None, threads: int = 0, window=None):
    """Backward definition for bf16 inputs (torch tensors, widened exactly to fp64).

    heads: optional list of flat head ids b*H + h to compute (default: all); the
    results then have shape (len(heads), L, D).  Returns (dQ, dK, dV, Delta) fp64.
    """
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    arrs = [decode_bf16(_bf16_bits(t)).reshape(B * H, t.shape[2], D) for t in (q, k, v, do)]
    if heads is not None:
        idx = np.asarray(heads, dtype=np.int64)
        arrs = [a[idx] for a in arrs]
    n = arrs[0].shape[0]
    dq, dk, dv, delta = gradients_f64(*(a.reshape(1, n, a.shape[1], D) for a in arrs), causal, scale, threads,
                                      window)
    if heads is None:
        return (dq.reshape(B, H, Lq, D), dk.reshape(B, H, Lk, D), dv.reshape(B, H, Lk, D), delta.reshape(B, H, Lq))
    return dq[0], dk[0], dv[0], delta[0]

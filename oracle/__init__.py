"""Float64 CPU oracle for multi-head scaled dot-product attention forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA product path shares no code with it and never calls it.

The arithmetic lives in ``attn_oracle.c`` (plain C loops, float64, OpenMP over
rows); this module only compiles it with gcc and marshals NumPy arrays through
ctypes.  It computes eq. (1) of "Attention Is All You Need" (section 3.2.1),
``softmax(Q K^T / sqrt(d_k) + M) V``, with M = -inf on forbidden connections
(section 3.2.3), plus the log-sum-exp of each row's scaled scores.  See the
header of ``attn_oracle.c`` for the definition written out, and
``tests/test_oracle.py`` for the pins that tie it to the pages.  The
backward (``attn_bwd``) is the gradient of that forward, pinned in
``tests/test_oracle_bwd.py`` by finite differences of the pinned forward.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_KEY_PADDING = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libattn_oracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``oracle/_build/libattn_oracle.so``.

    No -ffast-math: the oracle keeps IEEE float64 semantics.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            f = lib.oracle_attn_fwd_f64
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_long] * 6 + [
                ctypes.c_double, ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
            g = lib.oracle_attn_rows_f64
            g.restype = ctypes.c_int
            g.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_long] * 6 + [
                ctypes.c_double, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_long, ctypes.c_int]
            h = lib.oracle_attn_bwd_f64
            h.restype = ctypes.c_int
            h.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_long] * 6 + [
                ctypes.c_double, ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
            bd = lib.oracle_attn_band_f64
            bd.restype = ctypes.c_int
            bd.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_long] * 6 + [
                ctypes.c_double, ctypes.c_long, ctypes.c_long, ctypes.c_void_p, ctypes.c_long,
                ctypes.c_int]
            hb = lib.oracle_attn_bwd_band_f64
            hb.restype = ctypes.c_int
            hb.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_long] * 6 + [
                ctypes.c_double, ctypes.c_long, ctypes.c_long, ctypes.c_int]
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _as_f32(x) -> np.ndarray:
    """float32 C-contiguous copy-if-needed; bf16 values widen exactly."""
    if hasattr(x, "detach"):  # a torch tensor: go through float32 on the CPU
        x = x.detach().to("cpu").float().contiguous().numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def _prep(q, k, v, mask_kind, key_lens):
    q, k, v = _as_f32(q), _as_f32(k), _as_f32(v)
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, n, d]")
    B, H, n_q, d_k = q.shape
    if k.shape[:2] != (B, H) or v.shape[:2] != (B, H):
        raise ValueError("batch/head dims of q, k, v differ")
    n_k = k.shape[2]
    if k.shape[3] != d_k or v.shape[2] != n_k:
        raise ValueError("k must be [B,H,n_k,d_k] and v [B,H,n_k,d_v]")
    d_v = v.shape[3]
    kl = None
    if mask_kind == MASK_KEY_PADDING:
        if key_lens is None:
            raise ValueError("key padding needs key_lens")
        if hasattr(key_lens, "detach"):
            key_lens = key_lens.detach().to("cpu").numpy()
        kl = np.ascontiguousarray(key_lens, dtype=np.int32)
        if kl.shape != (B,):
            raise ValueError("key_lens must have one entry per batch")
    elif mask_kind not in (MASK_NONE, MASK_CAUSAL):
        raise ValueError(f"unknown mask kind {mask_kind}")
    return q, k, v, kl, (B, H, n_q, n_k, d_k, d_v)


def _ptr(a):
    return None if a is None else a.ctypes.data


def attn_fwd(q, k, v, scale: float, mask_kind: int = MASK_NONE,
             key_lens=None, threads: int = 0):
    """Every output row.  Returns (o [B,H,n_q,d_v] float64, lse [B,H,n_q] float64)."""
    q, k, v, kl, (B, H, n_q, n_k, d_k, d_v) = _prep(q, k, v, mask_kind, key_lens)
    o = np.empty((B, H, n_q, d_v), dtype=np.float64)
    lse = np.empty((B, H, n_q), dtype=np.float64)
    rc = _load().oracle_attn_fwd_f64(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, n_q, n_k, d_k, d_v,
        float(scale), int(mask_kind), _ptr(kl), int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_fwd_f64 failed ({rc})")
    return o, lse


def attn_rows(q, k, v, rows, scale: float, mask_kind: int = MASK_NONE,
              key_lens=None, threads: int = 0):
    """Only the flat rows ``(b*H + h)*n_q + i`` listed in ``rows``.

    Returns (o [len(rows), d_v] float64, lse [len(rows)] float64).
    """
    q, k, v, kl, (B, H, n_q, n_k, d_k, d_v) = _prep(q, k, v, mask_kind, key_lens)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    o = np.empty((rows.size, d_v), dtype=np.float64)
    lse = np.empty((rows.size,), dtype=np.float64)
    rc = _load().oracle_attn_rows_f64(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, n_q, n_k, d_k, d_v,
        float(scale), int(mask_kind), _ptr(kl), _ptr(rows), rows.size,
        int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_rows_f64 failed ({rc})")
    return o, lse


def attn_bwd(q, k, v, dout, scale: float, mask_kind: int = MASK_NONE, key_lens=None,
             threads: int = 0):
    """Gradients (dq, dk, dv), float64, of a loss whose gradient with
    respect to the forward's output O is ``dout`` [B,H,n_q,d_v]."""
    q, k, v, kl, (B, H, n_q, n_k, d_k, d_v) = _prep(q, k, v, mask_kind, key_lens)
    g = _as_f32(dout)
    if g.shape != (B, H, n_q, d_v):
        raise ValueError("dout must be [B,H,n_q,d_v]")
    dq = np.empty((B, H, n_q, d_k), dtype=np.float64)
    dk = np.empty((B, H, n_k, d_k), dtype=np.float64)
    dv = np.empty((B, H, n_k, d_v), dtype=np.float64)
    rc = _load().oracle_attn_bwd_f64(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(dq), _ptr(dk), _ptr(dv), B, H, n_q, n_k,
        d_k, d_v, float(scale), int(mask_kind), _ptr(kl), int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_bwd_f64 failed ({rc})")
    return dq, dk, dv


def attn_band(q, k, v, scale: float, left: int, right: int, rows=None, threads: int = 0):
    """Restricted self-attention: query i sees keys i-left <= j <= i+right.

    Every row (o [B,H,n_q,d_v], lse [B,H,n_q]) or, with ``rows``, only those
    flat rows (o [len(rows), d_v], lse [len(rows)]), float64.
    """
    q, k, v, _, (B, H, n_q, n_k, d_k, d_v) = _prep(q, k, v, MASK_NONE, None)
    if left < 0 or right < 0:
        raise ValueError("window sides must be >= 0")
    if rows is None:
        o = np.empty((B, H, n_q, d_v), dtype=np.float64)
        lse = np.empty((B, H, n_q), dtype=np.float64)
        rp, nr = None, 0
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        o = np.empty((rows.size, d_v), dtype=np.float64)
        lse = np.empty((rows.size,), dtype=np.float64)
        rp, nr = rows.ctypes.data, rows.size
    rc = _load().oracle_attn_band_f64(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, n_q, n_k, d_k, d_v, float(scale),
        int(left), int(right), rp, nr, int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_band_f64 failed ({rc})")
    return o, lse


def attn_bwd_band(q, k, v, dout, scale: float, left: int, right: int, threads: int = 0):
    """Gradients (dq, dk, dv), float64, of restricted self-attention (attn_band)."""
    q, k, v, _, (B, H, n_q, n_k, d_k, d_v) = _prep(q, k, v, MASK_NONE, None)
    if left < 0 or right < 0:
        raise ValueError("window sides must be >= 0")
    g = _as_f32(dout)
    if g.shape != (B, H, n_q, d_v):
        raise ValueError("dout must be [B,H,n_q,d_v]")
    dq = np.empty((B, H, n_q, d_k), dtype=np.float64)
    dk = np.empty((B, H, n_k, d_k), dtype=np.float64)
    dv = np.empty((B, H, n_k, d_v), dtype=np.float64)
    rc = _load().oracle_attn_bwd_band_f64(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(dq), _ptr(dk), _ptr(dv), B, H, n_q, n_k,
        d_k, d_v, float(scale), int(left), int(right), int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_bwd_band_f64 failed ({rc})")
    return dq, dk, dv

"""ctypes binding of the C ABI in ``include/attn.h``.

Argument marshalling only: every step of the attention runs in the CUDA
library.  PyTorch is used for device buffers and streams.  The library must
have been built (``transformer_head_scaled_gb300.build.build()``); if it is
missing, :func:`load` raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from .inputs import MASK_CAUSAL, MASK_KEY_PADDING, MASK_NONE  # noqa: F401

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build",
                        "libattn_gb300.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_CUDA = -3
ATTN_ERR_TIMEOUT = -4
ATTN_ERR_SCRATCH_TOO_SMALL = -5
MASK_WINDOW = 3  # attn_fwd_strided: the window of attn_fwd_window
DECODE_NOALLOC_SCRATCH_BYTES = 1 << 20

# Every entry point declared in include/attn.h.
EXPORTS = ("attn_fwd", "attn_fwd_f32", "attn_fwd_window", "attn_fwd_strided", "attn_fwd_host",
           "attn_fwd_host_buffer_bytes", "attn_decode", "attn_decode_strided",
           "attn_decode_workspace_bytes", "attn_decode_window",
           "attn_decode_window_workspace_bytes", "attn_decode_noalloc", "attn_bwd", "attn_bwd_window", "attn_bwd_strided",
           "attn_bwd_workspace_bytes",
           "attn_check", "attn_status_string",
           "attn_last_cuda_error", "attn_set_wait_limit_ns", "attn_launch_count",
           "attn_diag_tile", "attn_diag_wait_timeout")

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {status_string(status)} ({status})"
        if status == ATTN_ERR_CUDA and _lib is not None:
            msg += f", cudaError {_lib.attn_last_cuda_error()}"
        super().__init__(msg)


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (once) and declare the signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library {path} is missing: build it with "
                "transformer_head_scaled_gb300.build.build()")
        lib = ctypes.CDLL(path)
        vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        for name in ("attn_fwd", "attn_fwd_f32"):
            fn = getattr(lib, name)
            fn.restype = i32
            fn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp, vp]
        lib.attn_fwd_window.restype = i32
        lib.attn_fwd_window.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, i32,
                                        vp]
        lib.attn_fwd_strided.restype = i32
        lib.attn_fwd_strided.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp,
                                         vp, f32, i32, vp, i32, i32, vp]
        lib.attn_decode.restype = i32
        lib.attn_decode.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp,
                                    ctypes.c_size_t, vp]
        lib.attn_decode_noalloc.restype = i32
        lib.attn_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp,
                                            vp]
        lib.attn_decode_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
        lib.attn_decode_window.restype = i32
        lib.attn_decode_window.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp,
                                           i32, vp, ctypes.c_size_t, vp]
        lib.attn_decode_window_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_decode_window_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.attn_bwd.restype = i32
        lib.attn_bwd.argtypes = [vp] * 9 + [i32] * 5 + [f32, i32, vp, vp, ctypes.c_size_t, vp]
        lib.attn_decode_strided.restype = i32
        lib.attn_decode_strided.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, f32,
                                            vp, vp, ctypes.c_size_t, vp]
        lib.attn_fwd_host.restype = i32
        lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp,
                                      i32, i32, vp, ctypes.c_size_t, vp]
        lib.attn_fwd_host_buffer_bytes.restype = ctypes.c_size_t
        lib.attn_fwd_host_buffer_bytes.argtypes = [i32, i32, i32, i32, i32]
        lib.attn_bwd_strided.restype = i32
        lib.attn_bwd_strided.argtypes = [vp] * 9 + [i32] * 5 + [vp, f32, i32, vp, i32, i32, vp,
                                                                 ctypes.c_size_t, vp]
        lib.attn_bwd_window.restype = i32
        lib.attn_bwd_window.argtypes = [vp] * 9 + [i32] * 5 + [f32, i32, i32, vp, ctypes.c_size_t,
                                                                vp]
        lib.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_bwd_workspace_bytes.argtypes = [i32, i32, i32, i32]
        lib.attn_check.restype = i32
        lib.attn_check.argtypes = [vp]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_status_string.argtypes = [i32]
        lib.attn_last_cuda_error.restype = i32
        lib.attn_last_cuda_error.argtypes = []
        lib.attn_set_wait_limit_ns.restype = ctypes.c_uint64
        lib.attn_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        lib.attn_launch_count.restype = ctypes.c_uint64
        lib.attn_launch_count.argtypes = []
        lib.attn_diag_tile.restype = i32
        lib.attn_diag_tile.argtypes = [vp, vp, vp, vp, vp, vp, vp]
        lib.attn_diag_wait_timeout.restype = i32
        lib.attn_diag_wait_timeout.argtypes = [ctypes.c_uint64, vp]
        _lib = lib
        return lib


def status_string(status: int) -> str:
    if _lib is None:
        return str(status)
    return _lib.attn_status_string(int(status)).decode()


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


def attn_fwd_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, n_q, n_k, d_k, scale, mask_kind,
                 key_lens_ptr, stream_ptr, f32: bool = False) -> int:
    """The C call itself, on raw device pointers; returns the status code."""
    lib = load()
    fn = lib.attn_fwd_f32 if f32 else lib.attn_fwd
    return fn(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, n_q, n_k, d_k, float(scale),
              mask_kind, key_lens_ptr, stream_ptr)


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float | None = None,
             mask: int = MASK_NONE, key_lens: torch.Tensor | None = None,
             out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
             with_lse: bool = True, stream=None):
    """O = softmax(Q K^T * scale + M) V on the GPU, q/k/v [B, h, n, d] CUDA tensors.

    bf16 inputs run on the tensor cores (d = 64), float32 inputs on the CUDA
    cores.  scale defaults to 1/sqrt(d).  Returns (o, lse); lse is None when
    with_lse is False and no lse buffer is given.
    """
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if q.dtype != k.dtype or q.dtype != v.dtype or q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("q, k, v must all be bfloat16 or all float32")
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, h, n, d]")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    B, h, n_q, d = q.shape
    n_k = k.shape[2]
    if tuple(k.shape) != (B, h, n_k, d) or tuple(v.shape) != (B, h, n_k, d):
        raise ValueError("k and v must be [B, h, n_k, d] with q's B, h, d")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    kl = None
    if mask == MASK_KEY_PADDING:
        if key_lens is None:
            raise ValueError("key padding needs key_lens")
        kl = key_lens
        if kl.dtype != torch.int32 or not kl.is_cuda or kl.numel() != B or not kl.is_contiguous():
            raise ValueError("key_lens must be a contiguous int32 CUDA tensor of B entries")
    if out is None:
        out = torch.empty((B, h, n_q, d), dtype=q.dtype, device=q.device)
    if lse is None and with_lse:
        lse = torch.empty((B, h, n_q), dtype=torch.float32, device=q.device)
    rc = attn_fwd_raw(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, h, n_q, n_k, d, scale,
                      int(mask), _ptr(kl), _stream_ptr(stream), f32=q.dtype == torch.float32)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd")
    return out, lse


def attn_fwd_window_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, n_q, n_k, d_k, scale, left,
                       right, stream_ptr) -> int:
    """The C call itself, on raw device pointers; returns the status code."""
    return load().attn_fwd_window(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, n_q, n_k, d_k,
                                  float(scale), int(left), int(right), stream_ptr)


def attn_fwd_window(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, left: int, right: int,
                    scale: float | None = None, out: torch.Tensor | None = None,
                    lse: torch.Tensor | None = None, with_lse: bool = True, stream=None):
    """Restricted self-attention on the GPU: query i sees keys i-left .. i+right.

    q, k, v: contiguous bf16 CUDA [B, h, n, d] tensors, d in {16, 32, 64, 128}.
    Returns (o, lse).
    """
    for t in (q, k, v):
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous bf16 CUDA [B, h, n, d] tensors")
    B, h, n_q, d = q.shape
    n_k = k.shape[2]
    if tuple(k.shape) != (B, h, n_k, d) or tuple(v.shape) != (B, h, n_k, d):
        raise ValueError("k and v must be [B, h, n_k, d] with q's B, h, d")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and with_lse:
        lse = torch.empty((B, h, n_q), dtype=torch.float32, device=q.device)
    rc = attn_fwd_window_raw(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, h, n_q, n_k, d,
                             scale, left, right, _stream_ptr(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_window")
    return out, lse


def attn_fwd_strided_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, n_q, n_k, d_k, strides, scale,
                        mask_kind, lens_ptr, left, right, stream_ptr) -> int:
    """The C call itself; ``strides`` = four (b, h, n) element-stride triples for q, k, v, o."""
    arrs = [(ctypes.c_int64 * 3)(*[int(x) for x in st]) for st in strides]
    return load().attn_fwd_strided(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, n_q, n_k, d_k,
                                   *[ctypes.cast(a, ctypes.c_void_p) for a in arrs],
                                   float(scale), int(mask_kind), lens_ptr, int(left), int(right),
                                   stream_ptr)


def attn_fwd_strided(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float | None = None,
                     mask: int = MASK_NONE, key_lens: torch.Tensor | None = None,
                     window: tuple[int, int] | None = None, out: torch.Tensor | None = None,
                     lse: torch.Tensor | None = None, with_lse: bool = True, stream=None):
    """attn_fwd on [B, h, n, d] bf16 views with any strides over the first three
    dimensions and a contiguous last one (e.g. ``x.view(B, n, h, d).transpose(1, 2)``).
    ``window=(left, right)`` selects restricted self-attention; ``out`` may be a
    strided view too (default: contiguous)."""
    for t in (q, k, v):
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 4 or t.stride(-1) != 1:
            raise ValueError("q, k, v must be bf16 CUDA [B, h, n, d] views with unit last stride")
    B, h, n_q, d = q.shape
    n_k = k.shape[2]
    if tuple(k.shape) != (B, h, n_k, d) or tuple(v.shape) != (B, h, n_k, d):
        raise ValueError("k and v must be [B, h, n_k, d] with q's B, h, d")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    kl, left, right = None, 0, 0
    if window is not None:
        mask, (left, right) = MASK_WINDOW, window
    if mask == MASK_KEY_PADDING:
        if key_lens is None:
            raise ValueError("key padding needs key_lens")
        kl = key_lens
        if kl.dtype != torch.int32 or not kl.is_cuda or kl.numel() != B or not kl.is_contiguous():
            raise ValueError("key_lens must be a contiguous int32 CUDA tensor of B entries")
    if out is None:
        out = torch.empty((B, h, n_q, d), dtype=q.dtype, device=q.device)
    if tuple(out.shape) != (B, h, n_q, d) or out.stride(-1) != 1:
        raise ValueError("out must be a [B, h, n_q, d] view with unit last stride")
    if lse is None and with_lse:
        lse = torch.empty((B, h, n_q), dtype=torch.float32, device=q.device)
    strides = [t.stride()[:3] for t in (q, k, v, out)]
    rc = attn_fwd_strided_raw(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, h, n_q, n_k, d,
                              strides, scale, int(mask), _ptr(kl), left, right,
                              _stream_ptr(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_strided")
    return out, lse


def host_buffer_bytes(B: int, h: int, n_q: int, n_k: int, d: int = 64) -> int:
    """Device staging bytes attn_fwd_host needs (0 for unsupported sizes)."""
    return int(load().attn_fwd_host_buffer_bytes(B, h, n_q, n_k, d))


def attn_fwd_host_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, n_q, n_k, d_k, scale, mask_kind,
                      lens_ptr, left, right, buf_ptr, buf_bytes, stream_ptr) -> int:
    """The C call itself (host q, k, v, o, lse, lens; device staging); returns the status."""
    return load().attn_fwd_host(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, n_q, n_k, d_k,
                                float(scale), int(mask_kind), lens_ptr, int(left), int(right),
                                buf_ptr, int(buf_bytes), stream_ptr)


def attn_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float | None = None,
                  mask: int = MASK_NONE, key_lens: torch.Tensor | None = None,
                  window: tuple[int, int] | None = None, out: torch.Tensor | None = None,
                  lse: torch.Tensor | None = None, with_lse: bool = True,
                  buf: torch.Tensor | None = None, device=None, stream=None):
    """attn_fwd on host (CPU) bf16 [B, h, n, d] tensors, pinned for asynchronous copies:
    copies in, forward and copies out pipelined over batch slices on the device.
    Returns host (o, lse); they are complete once ``stream`` has reached the call's
    end (``check()`` synchronises)."""
    for t in (q, k, v):
        if t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous bf16 host [B, h, n, d] tensors")
    B, h, n_q, d = q.shape
    n_k = k.shape[2]
    if tuple(k.shape) != (B, h, n_k, d) or tuple(v.shape) != (B, h, n_k, d):
        raise ValueError("k and v must be [B, h, n_k, d] with q's B, h, d")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    kl, left, right = None, 0, 0
    if window is not None:
        mask, (left, right) = MASK_WINDOW, window
    if mask == MASK_KEY_PADDING:
        if key_lens is None:
            raise ValueError("key padding needs key_lens")
        kl = key_lens
        if kl.dtype != torch.int32 or kl.is_cuda or kl.numel() != B or not kl.is_contiguous():
            raise ValueError("key_lens must be a contiguous int32 host tensor of B entries")
    pin = q.is_pinned()
    if out is None:
        out = torch.empty((B, h, n_q, d), dtype=q.dtype, pin_memory=pin)
    if out.is_cuda or tuple(out.shape) != (B, h, n_q, d) or not out.is_contiguous():
        raise ValueError("out must be a contiguous host [B, h, n_q, d] tensor")
    if lse is None and with_lse:
        lse = torch.empty((B, h, n_q), dtype=torch.float32, pin_memory=pin)
    need = host_buffer_bytes(B, h, n_q, n_k, d)
    if buf is None or buf.numel() * buf.element_size() < need:
        dev = torch.device("cuda") if device is None else torch.device(device)
        buf = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    rc = attn_fwd_host_raw(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, h, n_q, n_k, d,
                           scale, int(mask), _ptr(kl), left, right, _ptr(buf),
                           buf.numel() * buf.element_size(), _stream_ptr(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_host")
    return out, lse


def attn_fwd_f32(q, k, v, **kw):
    """Float32 path (same as attn_fwd with float32 tensors)."""
    if q.dtype != torch.float32:
        raise ValueError("attn_fwd_f32 takes float32 tensors")
    return attn_fwd(q, k, v, **kw)


def decode_workspace_bytes(B: int, h: int, n_q: int, L_max: int, d: int = 64,
                           window: int | None = None) -> int:
    """Scratch bytes attn_decode (attn_decode_window when `window` is given)
    needs on the current device (0: none)."""
    if window is not None:
        return int(load().attn_decode_window_workspace_bytes(B, h, n_q, L_max, d, int(window)))
    return int(load().attn_decode_workspace_bytes(B, h, n_q, L_max, d))


def attn_decode_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, n_q, L_max, d, scale,
                    lens_ptr, ws_ptr, ws_bytes, stream_ptr) -> int:
    """The C call itself, on raw device pointers; returns the status code."""
    return load().attn_decode(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, n_q, L_max, d,
                              float(scale), lens_ptr, ws_ptr, int(ws_bytes), stream_ptr)


def attn_decode_window_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, n_q, L_max, d, scale,
                           lens_ptr, window, ws_ptr, ws_bytes, stream_ptr) -> int:
    """attn_decode_window on raw device pointers; returns the status code."""
    return load().attn_decode_window(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, n_q, L_max, d,
                                     float(scale), lens_ptr, int(window), ws_ptr, int(ws_bytes),
                                     stream_ptr)


def attn_decode_strided_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, n_q, L_max, d, strides,
                            scale, lens_ptr, ws_ptr, ws_bytes, stream_ptr) -> int:
    """The C call itself; ``strides`` = four (b, h, n) element-stride triples for q, k_cache,
    v_cache, o."""
    flat = (ctypes.c_int64 * 12)(*[int(x) for st in strides for x in st])
    return load().attn_decode_strided(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, n_q, L_max, d,
                                      ctypes.cast(flat, ctypes.c_void_p), float(scale), lens_ptr,
                                      ws_ptr, int(ws_bytes), stream_ptr)


def attn_decode_strided(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                        cache_lens: torch.Tensor | None = None, scale: float | None = None,
                        out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None, stream=None):
    """attn_decode on [B, h, n, d] bf16 views with any strides over the first three
    dimensions and a contiguous last one (e.g. a [B, L_max, h, d] cache seen as
    ``cache.transpose(1, 2)``); ``out`` may be a strided view too."""
    for t in (q, k_cache, v_cache):
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 4 or t.stride(-1) != 1:
            raise ValueError("q, k_cache, v_cache must be bf16 CUDA [B, h, n, d] views with unit "
                             "last stride")
    B, h, n_q, d = q.shape
    L_max = k_cache.shape[2]
    if tuple(k_cache.shape) != (B, h, L_max, d) or tuple(v_cache.shape) != (B, h, L_max, d):
        raise ValueError("caches must be [B, h, L_max, d] with q's B, h, d")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if cache_lens is not None and (cache_lens.dtype != torch.int32 or not cache_lens.is_cuda
                                   or cache_lens.numel() != B or not cache_lens.is_contiguous()):
        raise ValueError("cache_lens must be a contiguous int32 CUDA tensor of B entries")
    if out is None:
        out = torch.empty((B, h, n_q, d), dtype=q.dtype, device=q.device)
    if tuple(out.shape) != (B, h, n_q, d) or out.stride(-1) != 1:
        raise ValueError("out must be a [B, h, n_q, d] view with unit last stride")
    if lse is None:
        lse = torch.empty((B, h, n_q), dtype=torch.float32, device=q.device)
    need = decode_workspace_bytes(B, h, n_q, L_max, d)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    strides = [t.stride()[:3] for t in (q, k_cache, v_cache, out)]
    rc = attn_decode_strided_raw(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse), B,
                                 h, n_q, L_max, d, strides, scale, _ptr(cache_lens),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream_ptr(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode_strided")
    return out, lse


def attn_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                cache_lens: torch.Tensor | None = None, scale: float | None = None,
                out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                workspace: torch.Tensor | None = None, with_lse: bool = True, stream=None,
                window: int | None = None):
    """n_q <= 8 new queries q [B,h,n_q,d] against bf16 caches [B,h,L_max,d];
    query i sees the first cache_lens[b] keys (all L_max when None), or with
    `window` (attn_decode_window) only keys cache_lens[b]-1-window ..
    cache_lens[b]-1.  Returns (o, lse)."""
    for t in (q, k_cache, v_cache):
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError("q and the caches must be contiguous bf16 CUDA [B, h, n, d] tensors")
    B, h, n_q, d = q.shape
    L_max = k_cache.shape[2]
    if tuple(k_cache.shape) != (B, h, L_max, d) or tuple(v_cache.shape) != (B, h, L_max, d):
        raise ValueError("caches must be [B, h, L_max, d] with q's B, h, d")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if cache_lens is not None and (cache_lens.dtype != torch.int32 or not cache_lens.is_cuda
                                   or cache_lens.numel() != B or not cache_lens.is_contiguous()):
        raise ValueError("cache_lens must be a contiguous int32 CUDA tensor of B entries")
    if out is None:
        out = torch.empty((B, h, n_q, d), dtype=q.dtype, device=q.device)
    if lse is None and with_lse:
        lse = torch.empty((B, h, n_q), dtype=torch.float32, device=q.device)
    need = decode_workspace_bytes(B, h, n_q, L_max, d, window)
    if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if window is None:
        rc = attn_decode_raw(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse), B, h,
                             n_q, L_max, d, scale, _ptr(cache_lens), _ptr(workspace), ws_bytes,
                             _stream_ptr(stream))
    else:
        rc = attn_decode_window_raw(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse),
                                    B, h, n_q, L_max, d, scale, _ptr(cache_lens), window,
                                    _ptr(workspace), ws_bytes, _stream_ptr(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode" if window is None else "attn_decode_window")
    return out, lse


def bwd_workspace_bytes(B: int, h: int, n_q: int, d: int = 64) -> int:
    """Scratch bytes attn_bwd needs (0 for unsupported sizes)."""
    return int(load().attn_bwd_workspace_bytes(B, h, n_q, d))


def attn_bwd_raw(q_ptr, k_ptr, v_ptr, o_ptr, dout_ptr, lse_ptr, dq_ptr, dk_ptr, dv_ptr, B, h,
                 n_q, n_k, d, scale, mask_kind, lens_ptr, ws_ptr, ws_bytes, stream_ptr) -> int:
    """The C call itself, on raw device pointers; returns the status code."""
    return load().attn_bwd(q_ptr, k_ptr, v_ptr, o_ptr, dout_ptr, lse_ptr, dq_ptr, dk_ptr, dv_ptr,
                           B, h, n_q, n_k, d, float(scale), int(mask_kind), lens_ptr, ws_ptr,
                           int(ws_bytes), stream_ptr)


def attn_bwd_window_raw(q_ptr, k_ptr, v_ptr, o_ptr, dout_ptr, lse_ptr, dq_ptr, dk_ptr, dv_ptr, B,
                        h, n_q, n_k, d, scale, left, right, ws_ptr, ws_bytes, stream_ptr) -> int:
    """The C call itself, on raw device pointers; returns the status code."""
    return load().attn_bwd_window(q_ptr, k_ptr, v_ptr, o_ptr, dout_ptr, lse_ptr, dq_ptr, dk_ptr,
                                  dv_ptr, B, h, n_q, n_k, d, float(scale), int(left), int(right),
                                  ws_ptr, int(ws_bytes), stream_ptr)


def attn_bwd_strided_raw(q_ptr, k_ptr, v_ptr, o_ptr, dout_ptr, lse_ptr, dq_ptr, dk_ptr, dv_ptr, B,
                         h, n_q, n_k, d, strides, scale, mask_kind, lens_ptr, left, right, ws_ptr,
                         ws_bytes, stream_ptr) -> int:
    """The C call itself; ``strides`` = eight (b, h, n) element-stride triples for q, k, v, o,
    dout, dq, dk, dv."""
    flat = (ctypes.c_int64 * 24)(*[int(x) for st in strides for x in st])
    return load().attn_bwd_strided(q_ptr, k_ptr, v_ptr, o_ptr, dout_ptr, lse_ptr, dq_ptr, dk_ptr,
                                   dv_ptr, B, h, n_q, n_k, d, ctypes.cast(flat, ctypes.c_void_p),
                                   float(scale), int(mask_kind), lens_ptr, int(left), int(right),
                                   ws_ptr, int(ws_bytes), stream_ptr)


def attn_bwd_strided(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                     lse: torch.Tensor, dout: torch.Tensor, dq: torch.Tensor, dk: torch.Tensor,
                     dv: torch.Tensor, scale: float | None = None, mask: int = MASK_NONE,
                     key_lens: torch.Tensor | None = None,
                     window: tuple[int, int] | None = None,
                     workspace: torch.Tensor | None = None, stream=None):
    """attn_bwd on [B, h, n, d] bf16 views with any strides over the first three
    dimensions and a contiguous last one; the gradients are written into the
    given dq, dk, dv views (e.g. slices of one packed gradient buffer).
    ``window=(left, right)`` differentiates restricted self-attention."""
    for t in (q, k, v, o, dout, dq, dk, dv):
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 4 or t.stride(-1) != 1:
            raise ValueError("tensors must be bf16 CUDA [B, h, n, d] views with unit last stride")
    B, h, n_q, d = q.shape
    n_k = k.shape[2]
    for t in (k, v, dk, dv):
        if tuple(t.shape) != (B, h, n_k, d):
            raise ValueError("k, v, dk, dv must be [B, h, n_k, d] with q's B, h, d")
    for t in (o, dout, dq):
        if tuple(t.shape) != (B, h, n_q, d):
            raise ValueError("o, dout, dq must be shaped like q")
    if (lse is None or not lse.is_cuda or lse.dtype != torch.float32
            or tuple(lse.shape) != (B, h, n_q) or not lse.is_contiguous()):
        raise ValueError("lse must be the forward's contiguous float32 [B, h, n_q] CUDA tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    kl, left, right = None, 0, 0
    if window is not None:
        mask, (left, right) = MASK_WINDOW, window
    if mask == MASK_KEY_PADDING:
        if key_lens is None:
            raise ValueError("key padding needs key_lens")
        kl = key_lens
        if kl.dtype != torch.int32 or not kl.is_cuda or kl.numel() != B or not kl.is_contiguous():
            raise ValueError("key_lens must be a contiguous int32 CUDA tensor of B entries")
    need = bwd_workspace_bytes(B, h, n_q, d)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    strides = [t.stride()[:3] for t in (q, k, v, o, dout, dq, dk, dv)]
    rc = attn_bwd_strided_raw(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                              _ptr(dk), _ptr(dv), B, h, n_q, n_k, d, strides, scale, int(mask),
                              _ptr(kl), left, right, _ptr(workspace), ws_bytes,
                              _stream_ptr(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd_strided")
    return dq, dk, dv


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
             lse: torch.Tensor, dout: torch.Tensor, scale: float | None = None,
             mask: int = MASK_NONE, key_lens: torch.Tensor | None = None,
             dq: torch.Tensor | None = None, dk: torch.Tensor | None = None,
             dv: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
             window: tuple[int, int] | None = None, stream=None):
    """Gradients (dq, dk, dv) of attn_fwd for dout = dLoss/dO.

    q, k, v, o, dout: contiguous bf16 CUDA [B, h, n, d] tensors, d in {16, 32,
    64}; o and lse are what attn_fwd returned for q, k, v with the same scale
    and mask.
    A workspace of bwd_workspace_bytes(...) is allocated when none is given.
    ``window=(left, right)`` differentiates attn_fwd_window instead (mask and
    key_lens ignored).
    """
    for t in (q, k, v, o, dout):
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError("q, k, v, o, dout must be contiguous bf16 CUDA [B, h, n, d] tensors")
    B, h, n_q, d = q.shape
    n_k = k.shape[2]
    if tuple(k.shape) != (B, h, n_k, d) or tuple(v.shape) != (B, h, n_k, d):
        raise ValueError("k and v must be [B, h, n_k, d] with q's B, h, d")
    if tuple(o.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape):
        raise ValueError("o and dout must be shaped like q")
    if (lse is None or not lse.is_cuda or lse.dtype != torch.float32
            or tuple(lse.shape) != (B, h, n_q) or not lse.is_contiguous()):
        raise ValueError("lse must be the forward's contiguous float32 [B, h, n_q] CUDA tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    kl = None
    if mask == MASK_KEY_PADDING:
        if key_lens is None:
            raise ValueError("key padding needs key_lens")
        kl = key_lens
        if kl.dtype != torch.int32 or not kl.is_cuda or kl.numel() != B or not kl.is_contiguous():
            raise ValueError("key_lens must be a contiguous int32 CUDA tensor of B entries")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = bwd_workspace_bytes(B, h, n_q, d)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    if window is not None:
        rc = attn_bwd_window_raw(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                                 _ptr(dq), _ptr(dk), _ptr(dv), B, h, n_q, n_k, d, scale,
                                 window[0], window[1], _ptr(workspace), ws_bytes,
                                 _stream_ptr(stream))
    else:
        rc = attn_bwd_raw(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                          _ptr(dk), _ptr(dv), B, h, n_q, n_k, d, scale, int(mask), _ptr(kl),
                          _ptr(workspace), ws_bytes, _stream_ptr(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd_window" if window is not None else "attn_bwd")
    return dq, dk, dv


def check(stream=None) -> None:
    """Synchronise and raise if a kernel recorded an error (bounded wait ran out)."""
    rc = load().attn_check(_stream_ptr(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_check")


def set_wait_limit_ns(limit_ns: int) -> int:
    return int(load().attn_set_wait_limit_ns(int(limit_ns)))


def launch_count() -> int:
    return int(load().attn_launch_count())


def diag_tile(q, k, p, v, stream=None):
    """Single-tile tensor-core products (see attn_diag_tile in include/attn.h).

    q, k: bf16 [128, 64]; p: bf16 [128, 128]; v: bf16 [128, 64].
    Returns (s = q k^T float32 [128,128], o = p v float32 [128, 64]).
    """
    for t, shp in ((q, (128, 64)), (k, (128, 64)), (p, (128, 128)), (v, (128, 64))):
        if tuple(t.shape) != shp or t.dtype != torch.bfloat16 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"diag_tile: expected contiguous bf16 CUDA {shp}")
    s = torch.empty((128, 128), dtype=torch.float32, device=q.device)
    o = torch.empty((128, 64), dtype=torch.float32, device=q.device)
    rc = load().attn_diag_tile(_ptr(q), _ptr(k), _ptr(p), _ptr(v), _ptr(s), _ptr(o),
                               _stream_ptr(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_diag_tile")
    return s, o


def diag_wait_timeout(limit_ns: int, stream=None) -> None:
    rc = load().attn_diag_wait_timeout(int(limit_ns), _stream_ptr(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_diag_wait_timeout")

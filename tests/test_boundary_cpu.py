"""The C-ABI library without a GPU: it builds, loads, exports every symbol
include/attn.h declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import math
import os
import re

import pytest

from transformer_head_scaled_gb300 import binding
from transformer_head_scaled_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return binding.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert sorted(binding.EXPORTS) == _declared_functions()


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4):
        assert binding.status_string(code) not in ("", "unknown status")
    assert binding.status_string(7) == "unknown status"


def test_wait_limit_round_trip(lib):
    old = binding.set_wait_limit_ns(12345)
    assert binding.set_wait_limit_ns(old) == 12345
    assert binding.set_wait_limit_ns(0) == old      # 0 restores the default
    binding.set_wait_limit_ns(old)


# Fake, never-dereferenced device addresses: validation happens first.
A = 0x10000  # 16-byte aligned


def _call(f32=False, q=A, k=A, v=A, o=A, lse=None, B=1, h=1, n_q=8, n_k=8, d=64, scale=0.125,
          mask=0, lens=None):
    return binding.attn_fwd_raw(q, k, v, o, lse, B, h, n_q, n_k, d, scale, mask, lens, None, f32=f32)


@pytest.mark.parametrize("f32", [False, True])
def test_invalid_arguments_rejected_on_host(lib, f32):
    INV = binding.ATTN_ERR_INVALID_ARG
    assert _call(f32, q=None) == INV
    assert _call(f32, o=None) == INV
    assert _call(f32, k=A + 8) == INV            # misaligned
    assert _call(f32, lse=A + 2) == INV           # misaligned lse
    for field in ("B", "h", "n_q", "n_k"):
        assert _call(f32, **{field: 0}) == INV
        assert _call(f32, **{field: -3}) == INV
    assert _call(f32, scale=0.0) == INV
    assert _call(f32, scale=-1.0) == INV
    assert _call(f32, scale=math.nan) == INV
    assert _call(f32, scale=math.inf) == INV
    assert _call(f32, mask=3) == INV
    assert _call(f32, mask=-1) == INV
    assert _call(f32, mask=2, lens=None) == INV   # key padding needs lengths
    assert _call(f32, mask=2, lens=A + 2) == INV
    assert _call(f32, B=1 << 20, h=1 << 12) == INV  # B*h beyond 2^31


def test_unsupported_head_sizes(lib):
    UNS = binding.ATTN_ERR_UNSUPPORTED
    for d in (8, 48, 96, 256):
        assert _call(False, d=d) == UNS
    for d in (8, 48, 96, 256):
        assert _call(True, d=d) == UNS


def test_decode_arguments_rejected_on_host(lib):
    def call(q=A, k=A, v=A, o=A, lse=None, B=1, h=1, n_q=1, L=8, d=64, scale=0.125, lens=None,
             ws=None, ws_bytes=0):
        return binding.attn_decode_raw(q, k, v, o, lse, B, h, n_q, L, d, scale, lens, ws,
                                       ws_bytes, None)
    INV, UNS = binding.ATTN_ERR_INVALID_ARG, binding.ATTN_ERR_UNSUPPORTED
    assert call(q=None) == INV
    assert call(k=A + 4) == INV
    assert call(n_q=0) == INV and call(L=0) == INV and call(B=0) == INV
    assert call(scale=float("nan")) == INV
    assert call(lens=A + 2) == INV
    assert call(n_q=9) == UNS
    assert call(d=48) == UNS and call(d=256) == UNS   # head sizes 16, 32, 64, 128 only
    assert call(B=1 << 9, h=1 << 8) == UNS      # B*h beyond the grid's y extent
    assert lib.attn_decode_workspace_bytes(1, 1, 9, 8, 64) == 0   # unsupported sizes
    assert lib.attn_decode_workspace_bytes(1, 1, 1, 8, 48) == 0


def test_diag_entry_points_validate(lib):
    assert lib.attn_diag_tile(None, A, A, A, A, A, None) == binding.ATTN_ERR_INVALID_ARG
    assert lib.attn_diag_tile(A, A, A + 4, A, A, A, None) == binding.ATTN_ERR_INVALID_ARG
    assert lib.attn_diag_wait_timeout(0, None) == binding.ATTN_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        binding.attn_fwd(x, x, x)


def test_missing_library_fails_loudly(tmp_path):
    """No silent fallback: a missing library is an error."""
    saved = binding._lib
    binding._lib = None
    try:
        with pytest.raises(RuntimeError, match="missing"):
            binding.load(str(tmp_path / "nope.so"))
    finally:
        binding._lib = saved


def test_bwd_arguments_rejected_on_host(lib):
    def call(q=A, k=A, v=A, o=A, dout=A, lse=A, dq=A, dk=A, dv=A, B=1, h=1, n_q=8, n_k=8, d=64,
             scale=0.125, mask=0, lens=None, ws=A, ws_bytes=1 << 30):
        return binding.attn_bwd_raw(q, k, v, o, dout, lse, dq, dk, dv, B, h, n_q, n_k, d, scale,
                                    mask, lens, ws, ws_bytes, None)
    INV, UNS = binding.ATTN_ERR_INVALID_ARG, binding.ATTN_ERR_UNSUPPORTED
    for name in ("q", "k", "v", "o", "dout", "lse", "dq", "dk", "dv", "ws"):
        assert call(**{name: None}) == INV, name
    for name in ("q", "k", "v", "o", "dout", "dq", "dk", "dv", "ws"):
        assert call(**{name: A + 8}) == INV, name
    assert call(lse=A + 2) == INV
    assert call(n_q=0) == INV and call(n_k=0) == INV and call(B=0) == INV and call(h=-1) == INV
    assert call(scale=0.0) == INV and call(scale=float("nan")) == INV
    assert call(mask=2) == INV and call(mask=5) == INV
    assert call(d=48) == UNS and call(d=128) == UNS and call(d=8) == UNS
    need = lib.attn_bwd_workspace_bytes(2, 3, 200, 64)
    assert call(B=2, h=3, n_q=200, ws_bytes=need - 1) == INV


def test_bwd_workspace_size():
    binding.load()
    # per head and 128-query tile a 4 KB constant tile, then n_q x 64 float32
    assert binding.bwd_workspace_bytes(2, 3, 200) == 6 * (2 * 4096 + 200 * 64 * 4)
    assert binding.bwd_workspace_bytes(1, 1, 128) == 4096 + 128 * 64 * 4
    # d = 16, 32: the same constant tiles, n_q x d float32
    assert binding.bwd_workspace_bytes(1, 1, 8, 32) == 4096 + 8 * 32 * 4
    assert binding.bwd_workspace_bytes(2, 1, 300, 16) == 2 * (3 * 4096 + 300 * 16 * 4)
    assert binding.bwd_workspace_bytes(1, 1, 8, 128) == 0
    assert binding.bwd_workspace_bytes(1, 1, 8, 48) == 0
    assert binding.bwd_workspace_bytes(0, 1, 8) == 0


def test_window_arguments_rejected_on_host(lib):
    def call(left=4, right=4, d=64, q=A, n_q=8):
        return binding.attn_fwd_window_raw(q, A, A, A, None, 1, 1, n_q, 8, d, 0.125, left, right,
                                           None)
    assert call(left=-1) == binding.ATTN_ERR_INVALID_ARG
    assert call(right=-5) == binding.ATTN_ERR_INVALID_ARG
    assert call(q=None) == binding.ATTN_ERR_INVALID_ARG
    assert call(n_q=0) == binding.ATTN_ERR_INVALID_ARG
    assert call(d=48) == binding.ATTN_ERR_UNSUPPORTED


def test_strided_arguments_rejected_on_host(lib):
    good = [(8 * 64 * 8, 64, 8 * 64)] * 4   # [B, n, h, d] strides of a [B, h, n, d] view

    def call(strides=good, mask=0, lens=None, left=0, right=0, d=64, q=A):
        return binding.attn_fwd_strided_raw(q, A, A, A, None, 1, 8, 8, 8, d, strides, 0.125, mask,
                                            lens, left, right, None)
    INV = binding.ATTN_ERR_INVALID_ARG
    assert call(strides=[(8 * 64 * 8, 64, 8 * 64 + 4)] + good[1:]) == INV  # not 16-byte strides
    assert call(strides=good[:3] + [(0, 64, 512)]) == INV                   # zero stride
    assert call(strides=good[:1] + [(-512, 64, 512)] + good[2:]) == INV     # negative stride
    assert call(mask=3, left=-1) == INV
    assert call(mask=4) == INV
    assert call(mask=2, lens=None) == INV
    assert call(q=None) == INV
    assert call(d=48) == binding.ATTN_ERR_UNSUPPORTED


def test_bwd_window_arguments_rejected_on_host(lib):
    def call(left=4, right=4, d=64, q=A, ws_bytes=1 << 30):
        return binding.attn_bwd_window_raw(q, A, A, A, A, A, A, A, A, 1, 1, 8, 8, d, 0.125, left,
                                           right, A, ws_bytes, None)
    INV = binding.ATTN_ERR_INVALID_ARG
    assert call(left=-1) == INV and call(right=-1) == INV
    assert call(q=None) == INV
    assert call(ws_bytes=16) == INV
    assert call(d=128) == binding.ATTN_ERR_UNSUPPORTED
    # attn_bwd itself takes no window
    assert binding.attn_bwd_raw(A, A, A, A, A, A, A, A, A, 1, 1, 8, 8, 64, 0.125, 3, None, A,
                                1 << 30, None) == INV


def test_bwd_strided_arguments_rejected_on_host(lib):
    good = [(8 * 64 * 8, 64, 8 * 64)] * 8   # [B, n, h, d] strides of a [B, h, n, d] view

    def call(strides=good, mask=0, lens=None, left=0, right=0, d=64, q=A, ws_bytes=1 << 30):
        return binding.attn_bwd_strided_raw(q, A, A, A, A, A, A, A, A, 1, 8, 8, 8, d, strides,
                                            0.125, mask, lens, left, right, A, ws_bytes, None)
    INV = binding.ATTN_ERR_INVALID_ARG
    for i in range(8):   # every tensor's strides are checked: 16-byte multiples, positive
        bad = list(good)
        bad[i] = (8 * 64 * 8, 64, 8 * 64 + 4)
        assert call(strides=bad) == INV, i
        bad[i] = (0, 64, 512)
        assert call(strides=bad) == INV, i
    assert call(mask=3, left=-1) == INV
    assert call(mask=4) == INV
    assert call(mask=2, lens=None) == INV
    assert call(q=None) == INV
    assert call(ws_bytes=16) == INV
    assert call(d=128) == binding.ATTN_ERR_UNSUPPORTED
    assert lib.attn_bwd_strided(A, A, A, A, A, A, A, A, A, 1, 8, 8, 8, 64, None, 0.125, 0, None,
                                0, 0, A, 1 << 30, None) == INV   # no stride array


def test_fwd_host_arguments_rejected_on_host(lib):
    H = 0x20000  # a host address: only non-null is required of it

    def call(q=H, o=H, B=2, d=64, mask=0, lens=None, left=0, right=0, buf=A, nbytes=1 << 30):
        return binding.attn_fwd_host_raw(q, H, H, o, None, B, 2, 8, 8, d, 0.125, mask, lens, left,
                                         right, buf, nbytes, None)
    INV = binding.ATTN_ERR_INVALID_ARG
    assert call(q=None) == INV and call(o=None) == INV
    assert call(B=0) == INV
    assert call(mask=5) == INV and call(mask=3, left=-1) == INV
    assert call(mask=2, lens=None) == INV
    assert call(buf=A + 16) == INV            # staging must be 256-byte aligned
    assert call(buf=None) == INV
    assert call(nbytes=1024) == INV
    assert call(d=48) == binding.ATTN_ERR_UNSUPPORTED


def test_fwd_host_buffer_size():
    binding.load()
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    B, h, n_q, n_k, d = 3, 2, 100, 70, 64
    want = (up(B * h * n_q * d * 2) * 2 + up(B * h * n_k * d * 2) * 2 + up(B * h * n_q * 4)
            + up(B * 4))
    assert binding.host_buffer_bytes(B, h, n_q, n_k, d) == want
    assert binding.host_buffer_bytes(1, 1, 8, 8, 48) == 0
    assert binding.host_buffer_bytes(0, 1, 8, 8, 64) == 0


def test_decode_strided_arguments_rejected_on_host(lib):
    good = [(8 * 64 * 4, 64, 4 * 64)] * 4

    def call(strides=good, d=64, q=A):
        return binding.attn_decode_strided_raw(q, A, A, A, None, 1, 4, 1, 8, d, strides, 0.125,
                                               None, None, 0, None)
    INV = binding.ATTN_ERR_INVALID_ARG
    for i in range(4):
        bad = list(good)
        bad[i] = (8 * 64 * 4, 64 + 4, 4 * 64)
        assert call(strides=bad) == INV, i
        bad[i] = (8 * 64 * 4, 64, -256)
        assert call(strides=bad) == INV, i
    assert call(q=None) == INV
    assert call(d=48) == binding.ATTN_ERR_UNSUPPORTED
    assert lib.attn_decode_strided(A, A, A, A, None, 1, 4, 1, 8, 64, None, 0.125, None, None, 0,
                                   None) == INV


def test_decode_window_arguments_rejected_on_host(lib):
    def call(q=A, window=16, d=64, n_q=1, lens=None):
        return binding.attn_decode_window_raw(q, A, A, A, None, 1, 4, n_q, 8, d, 0.125, lens,
                                              window, None, 0, None)
    INV, UNS = binding.ATTN_ERR_INVALID_ARG, binding.ATTN_ERR_UNSUPPORTED
    assert call(window=-1) == INV and call(window=-100) == INV
    assert call(q=None) == INV
    assert call(lens=A + 2) == INV
    assert call(d=48) == UNS and call(n_q=9) == UNS
    assert lib.attn_decode_window_workspace_bytes(1, 1, 1, 8, 64, -1) == 0
    assert lib.attn_decode_window_workspace_bytes(1, 1, 9, 8, 64, 4) == 0   # unsupported sizes
    assert lib.attn_decode_window_workspace_bytes(1, 1, 1, 8, 48, 4) == 0

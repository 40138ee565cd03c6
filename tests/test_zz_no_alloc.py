"""attn_decode_noalloc: the decoding step for callers that cannot allocate.

Some callers may not allocate device memory while they run attention: an
engine that reserves all of its device memory before it starts serving, a
plug-in that is handed only its input and output buffers, or code that cannot
afford the device-wide synchronisation an allocation can cause.  For them the
library keeps a fixed scratch array of its own (1 MiB per device, held until
the process exits) and attn_decode_noalloc uses it in place of the workspace
that attn_decode takes from the caller.

These tests call it through the C ABI and check that it returns what
attn_decode returns with a caller-allocated workspace, within the tolerances
the other parity tests use, on two calls in a row (the second call finds the
first call's leftovers in the shared array), and that sizes whose partial
results do not fit the array are refused.  The file is collected last, so a
failure here never hides the outcome of another test; it also runs on its own
in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from transformer_head_scaled_gb300 import binding, inputs
from transformer_head_scaled_gb300.inputs import MASK_KEY_PADDING, Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from transformer_head_scaled_gb300.build import build
    build()
    return binding.load()


def _inputs(B, h, n_q, L_max, seed):
    w = Workload("na", B, h, n_q, L_max, 64, MASK_KEY_PADDING, "bf16", lens_lo=1, kind="decode")
    q, k, v, lens = inputs.make_inputs(w, device="cuda", seeds=(seed, seed + 1, seed + 2, seed + 3))
    return w, q, k, v, lens


def _noalloc(lib, w, q, k, v, lens):
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.h, w.n_q), dtype=torch.float32, device="cuda")
    rc = lib.attn_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), w.B, w.h, w.n_q, w.n_k, w.d,
                                 ctypes.c_float(w.scale), lens.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    return rc, o, lse


def _close(o, lse, o_ref, l_ref):
    err = (o.float() - o_ref.float()).abs()
    assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3
    assert torch.equal(torch.isneginf(lse), torch.isneginf(l_ref))
    fin = torch.isfinite(l_ref)
    assert (lse[fin] - l_ref[fin]).abs().max().item() <= 1e-3


def test_noalloc_matches_workspace_entry_point_twice(lib):
    # first a split cache (the partials go to the library's array), then a
    # different problem that reuses the array after it
    cases = [(1, 2, 2, 4096, 10), (3, 4, 1, 1000, 20)]
    assert binding.decode_workspace_bytes(*cases[0][:4]) > 0
    assert binding.decode_workspace_bytes(*cases[1][:4]) > 0
    for B, h, n_q, L, seed in cases:
        w, q, k, v, lens = _inputs(B, h, n_q, L, seed)
        o_ref, l_ref = binding.attn_decode(q, k, v, lens, scale=w.scale)
        rc, o, lse = _noalloc(lib, w, q, k, v, lens)
        assert rc == binding.ATTN_OK, binding.status_string(rc)
        binding.check()
        _close(o, lse, o_ref, l_ref)


def test_noalloc_refuses_sizes_beyond_its_array(lib):
    # 600 heads of 8 queries, split in two: 600 * 2 * 8 partials of 264 bytes
    w, q, k, v, lens = _inputs(75, 8, 8, 1024, 30)
    need = binding.decode_workspace_bytes(75, 8, 8, 1024)
    assert need > binding.DECODE_NOALLOC_SCRATCH_BYTES
    rc, _, _ = _noalloc(lib, w, q, k, v, lens)
    assert rc == binding.ATTN_ERR_SCRATCH_TOO_SMALL
    binding.check()

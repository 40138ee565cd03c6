"""attn_decode_noalloc: the decoding step for callers that cannot allocate.

Some callers may not allocate device memory while they run attention: an
engine that reserves all of its device memory before it starts serving, a
plug-in that is handed only its input and output buffers, or code that cannot
afford the device-wide synchronisation an allocation can cause.  For them the
library keeps a fixed scratch array of its own (1 MiB per device, held until
the process exits) and attn_decode_noalloc uses it in place of the workspace
that attn_decode takes from the caller.

These tests call it through the C ABI and check it against the float64
oracle (the decoding step is the forward with a key-padding mask over the
cache) and against attn_decode with a caller-allocated workspace, within the
tolerances the other parity tests use, on calls in a row that share the
array: a split cache, a second problem whose partials need more of the array
than the first one's, an empty cache entry, and the plain-load kernel of the
other head sizes.  Sizes whose partials do not fit the array are refused.
The file is collected last, so a failure here never hides the outcome of
another test; it also runs on its own in a fresh process.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from transformer_head_scaled_gb300 import binding, inputs
from transformer_head_scaled_gb300.inputs import MASK_KEY_PADDING, Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from transformer_head_scaled_gb300.build import build
    build()
    oracle.build()
    return binding.load()


def _inputs(B, h, n_q, L_max, seed, d=64, zero_first=False):
    w = Workload("na", B, h, n_q, L_max, d, MASK_KEY_PADDING, "bf16", lens_lo=1, kind="decode")
    q, k, v, lens = inputs.make_inputs(w, device="cuda", seeds=(seed, seed + 1, seed + 2, seed + 3))
    if zero_first:
        lens[0] = 0  # an empty cache: O = 0, LSE = -inf
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


def _close_oracle(w, q, k, v, lens, o, lse):
    o_ref, l_ref = oracle.attn_fwd(q, k, v, w.scale, MASK_KEY_PADDING, lens)
    _close(o.cpu(), lse.cpu(), torch.from_numpy(o_ref), torch.from_numpy(l_ref))


# B, h, n_q, L_max, seed, d, empty first cache
CASES = [
    (1, 2, 2, 4096, 10, 64, False),   # long split cache (TMA-fed kernel)
    (3, 4, 1, 1000, 20, 64, True),    # a second problem over the array, one empty cache
    (2, 8, 4, 8192, 40, 64, False),   # more partials than both calls before it
    (2, 3, 2, 3000, 50, 128, True),   # plain-load kernel (d = 128), split, one empty cache
    (2, 4, 1, 2500, 60, 32, False),   # plain-load kernel (d = 32), split
]


def test_noalloc_matches_oracle_and_workspace_entry_point(lib):
    needs = []
    for B, h, n_q, L, seed, d, zero in CASES:
        need = binding.decode_workspace_bytes(B, h, n_q, L, d)
        assert 0 < need <= binding.DECODE_NOALLOC_SCRATCH_BYTES
        needs.append(need)
        w, q, k, v, lens = _inputs(B, h, n_q, L, seed, d, zero)
        o_ref, l_ref = binding.attn_decode(q, k, v, lens, scale=w.scale)
        rc, o, lse = _noalloc(lib, w, q, k, v, lens)
        assert rc == binding.ATTN_OK, binding.status_string(rc)
        binding.check()
        _close(o, lse, o_ref, l_ref)
        _close_oracle(w, q, k, v, lens, o, lse)
    assert needs[2] > max(needs[0], needs[1])  # a later call uses more of the array


def test_noalloc_unsplit_cache_needs_no_array(lib):
    # one chunk per head: no partials, the array is not used
    w, q, k, v, lens = _inputs(512, 8, 1, 256, 70, 64, True)
    assert binding.decode_workspace_bytes(512, 8, 1, 256, 64) == 0
    rc, o, lse = _noalloc(lib, w, q, k, v, lens)
    assert rc == binding.ATTN_OK, binding.status_string(rc)
    binding.check()
    _close_oracle(w, q, k, v, lens, o, lse)


def test_noalloc_refuses_sizes_beyond_its_array(lib):
    # 600 heads of 8 queries over 1024-key caches: more partials than the array holds
    w, q, k, v, lens = _inputs(75, 8, 8, 1024, 30)
    need = binding.decode_workspace_bytes(75, 8, 8, 1024)
    assert need > binding.DECODE_NOALLOC_SCRATCH_BYTES
    rc, _, _ = _noalloc(lib, w, q, k, v, lens)
    assert rc == binding.ATTN_ERR_SCRATCH_TOO_SMALL
    binding.check()

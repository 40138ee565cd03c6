"""attn_fwd_host (host buffers in and out, copies pipelined with the forward
over batch slices) against attn_fwd on the device: the same kernel computes
every (b, h), so O and LSE must be equal bit for bit; and against the float64
oracle on one case under the forward's tolerances."""
import numpy as np
import pytest
import torch

import oracle
from transformer_head_scaled_gb300 import binding, inputs
from transformer_head_scaled_gb300.inputs import (MASK_CAUSAL, MASK_KEY_PADDING, MASK_NONE,
                                                  Workload)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from transformer_head_scaled_gb300.build import build
    build()
    oracle.build()
    return binding.load()


def _host(B, h, n_q, n_k, d, seed, pin=True):
    w = Workload("host", B, h, n_q, n_k, d, MASK_NONE, "bf16")
    q, k, v, _ = inputs.make_inputs(w, device="cpu", seeds=(seed, seed + 1, seed + 2, seed + 3))
    if pin:
        q, k, v = (t.pin_memory() for t in (q, k, v))
    return q, k, v


CASES = [
    # B, h, n_q, n_k, d, mask, lens, window
    (11, 2, 200, 300, 64, MASK_NONE, None, None),          # 8 uneven slices
    (8, 3, 256, 256, 64, MASK_CAUSAL, None, None),
    (5, 2, 130, 400, 64, MASK_KEY_PADDING, [0, 1, 129, 400, 77], None),
    (9, 2, 600, 600, 64, MASK_NONE, None, (100, 50)),
    (1, 4, 384, 384, 128, MASK_CAUSAL, None, None),        # a single slice
    (16, 2, 300, 300, 32, MASK_NONE, None, None),
]


@pytest.mark.parametrize("B,h,n_q,n_k,d,mask,lens,window", CASES)
def test_fwd_host_equals_device_path(B, h, n_q, n_k, d, mask, lens, window):
    q, k, v = _host(B, h, n_q, n_k, d, seed=40)
    kl_host = None if lens is None else torch.tensor(lens, dtype=torch.int32)
    o, lse = binding.attn_fwd_host(q, k, v, mask=mask, key_lens=kl_host, window=window)
    binding.check()
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    if window is not None:
        o_ref, lse_ref = binding.attn_fwd_window(qd, kd, vd, window[0], window[1])
    else:
        o_ref, lse_ref = binding.attn_fwd(qd, kd, vd, mask=mask,
                                          key_lens=None if kl_host is None else kl_host.cuda())
    binding.check()
    assert torch.equal(o, o_ref.cpu())
    assert torch.equal(lse, lse_ref.cpu())


def test_fwd_host_matches_oracle_pageable_and_without_lse():
    B, h, n, d = 3, 2, 257, 64
    q, k, v = _host(B, h, n, n, d, seed=50, pin=False)   # pageable memory: correct, not async
    o, lse = binding.attn_fwd_host(q, k, v, mask=MASK_CAUSAL, with_lse=False)
    binding.check()
    assert lse is None
    o_ref, _ = oracle.attn_fwd(q, k, v, 0.125, MASK_CAUSAL, None)
    err = np.abs(o.float().numpy().astype(np.float64) - o_ref)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3


def test_fwd_host_back_to_back_calls_share_the_staging_buffer():
    """Two calls enqueued without a synchronisation in between, on a side stream,
    into one staging buffer: the second call's copies in wait for the first's
    copies out."""
    B, h, n, d = 12, 2, 320, 64
    a = _host(B, h, n, n, d, seed=60)
    b = _host(B, h, n, n, d, seed=70)
    buf = torch.empty(binding.host_buffer_bytes(B, h, n, n, d), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    oa, la = binding.attn_fwd_host(*a, buf=buf, stream=s)
    ob, lb = binding.attn_fwd_host(*b, buf=buf, stream=s)
    binding.check(s)
    for (q, k, v), o, lse in ((a, oa, la), (b, ob, lb)):
        o_ref, lse_ref = binding.attn_fwd(q.cuda(), k.cuda(), v.cuda())
        binding.check()
        assert torch.equal(o, o_ref.cpu()) and torch.equal(lse, lse_ref.cpu())

"""GPU parity of restricted self-attention (attn_fwd_window) against the
float64 oracle (oracle.attn_band), with the forward's bf16 tolerances:
max |O - O_ref| <= 2e-2, mean |O - O_ref| <= 2e-3, |LSE - LSE_ref| <= 1e-3.
Small cases compare every row; the full-size workload compares sampled rows
(the first and last rows of every 128-row tile band and random ones)."""
import numpy as np
import pytest
import torch

import oracle
from transformer_head_scaled_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, LSE_TOL = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from transformer_head_scaled_gb300.build import build
    build()
    oracle.build()
    return binding.load()


def _inputs(B, h, n_q, n_k, seed=0):
    q = inputs.gaussian((B, h, n_q, 64), seed).to(torch.bfloat16)
    k = inputs.gaussian((B, h, n_k, 64), seed + 1).to(torch.bfloat16)
    v = inputs.gaussian((B, h, n_k, 64), seed + 2).to(torch.bfloat16)
    return q, k, v


def _compare(o, lse, o_ref, l_ref):
    o = o.float().cpu().numpy().astype(np.float64).reshape(o_ref.shape)
    lse = lse.cpu().numpy().astype(np.float64).reshape(l_ref.shape)
    assert np.isfinite(o).all()
    err = np.abs(o - o_ref)
    assert err.max() <= BF16_MAX, f"max abs err {err.max():.3g}"
    assert err.mean() <= BF16_MEAN, f"mean abs err {err.mean():.3g}"
    assert np.array_equal(np.isneginf(lse), np.isneginf(l_ref))
    fin = np.isfinite(l_ref)
    if fin.any():
        assert np.abs(lse[fin] - l_ref[fin]).max() <= LSE_TOL


CASES = [
    # B, h, n_q, n_k, left, right
    (2, 2, 300, 300, 64, 64),     # centred window, ragged tail
    (1, 2, 512, 512, 128, 0),     # causal window
    (2, 1, 200, 333, 0, 50),      # forward-looking window
    (1, 2, 384, 384, 0, 0),       # each query sees itself only
    (1, 2, 130, 600, 200, 30),    # n_q < n_k
    (1, 1, 700, 100, 20, 20),     # queries past the last key: empty windows
    (1, 2, 1000, 1000, 127, 129), # window edges one off the tile size
    (2, 2, 640, 640, 300, 300),   # window wider than a tile pair
]


@pytest.mark.parametrize("B,h,n_q,n_k,left,right", CASES)
def test_window_matches_oracle(B, h, n_q, n_k, left, right):
    q, k, v = _inputs(B, h, n_q, n_k)
    o, lse = binding.attn_fwd_window(q.cuda(), k.cuda(), v.cuda(), left, right)
    binding.check()
    o_ref, l_ref = oracle.attn_band(q, k, v, 0.125, left, right)
    _compare(o, lse, o_ref, l_ref)


def test_unbounded_window_equals_the_unmasked_and_causal_kernels():
    """A window covering everything is the unmasked forward and (right = 0)
    the causal one: same tiles, same arithmetic, bit for bit."""
    q, k, v = (t.cuda() for t in _inputs(2, 2, 400, 400, seed=5))
    a = binding.attn_fwd_window(q, k, v, 10 ** 6, 10 ** 6)
    b = binding.attn_fwd(q, k, v)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    a = binding.attn_fwd_window(q, k, v, 10 ** 6, 0)
    b = binding.attn_fwd(q, k, v, mask=inputs.MASK_CAUSAL)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    binding.check()


def test_keys_outside_every_window_are_never_used():
    q, k, v = (t.cuda() for t in _inputs(1, 2, 256, 1024, seed=7))
    a = binding.attn_fwd_window(q, k, v, 10, 10)
    k2, v2 = k.clone(), v.clone()
    k2[:, :, 512:] = float("nan")   # beyond every window of the 256 queries
    v2[:, :, 512:] = float("nan")
    b = binding.attn_fwd_window(q, k2, v2, 10, 10)
    binding.check()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_full_size_window_workload_whole_tensor():
    """The benchmark's restricted-attention workload (2048 work items), every
    element against the band oracle."""
    w = inputs.WORKLOADS["big_window"]
    q, k, v, _ = inputs.make_inputs(w, device="cuda")
    o, lse = binding.attn_fwd_window(q, k, v, w.win_left, w.win_right)
    binding.check()
    o_ref, l_ref = oracle.attn_band(q, k, v, w.scale, w.win_left, w.win_right)
    _compare(o, lse, o_ref, l_ref)

"""GPU parity of the decoding step with restricted self-attention
(attn_decode_window) against the float64 oracle.

Restricted self-attention ("Attention Is All You Need", section 4 and
Table 1) lets a position attend only to a neighbourhood of itself; at the
newest position of a decoder that neighbourhood is the newest cached key and
the `window` keys before it.  By that definition the expected result for
batch entry b is plain attention of its queries over the cache slice
[max(0, L_b - 1 - window), L_b), which is what the oracle is given here (an
empty slice: O = 0, LSE = -inf).  Tolerances as for the other decode tests:
max |dO| <= 2e-2, mean |dO| <= 2e-3, |dLSE| <= 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from transformer_head_scaled_gb300 import binding, inputs
from transformer_head_scaled_gb300.inputs import MASK_KEY_PADDING, MASK_NONE, Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from transformer_head_scaled_gb300.build import build
    build()
    oracle.build()
    return binding.load()


def _expected(q, k, v, lens, window, scale):
    """Per batch entry: the oracle over the window's slice of the cache."""
    q, k, v = (t.float().cpu() for t in (q, k, v))
    B, H, n_q, d = q.shape
    L_max = k.shape[2]
    o = np.zeros((B, H, n_q, d))
    lse = np.full((B, H, n_q), -np.inf)
    for b in range(B):
        L = L_max if lens is None else min(max(int(lens[b]), 0), L_max)
        lo = max(0, L - 1 - window)
        if L > lo:
            o[b:b + 1], lse[b:b + 1] = oracle.attn_fwd(q[b:b + 1], k[b:b + 1, :, lo:L],
                                                       v[b:b + 1, :, lo:L], scale, MASK_NONE)
    return o, lse


def _check(o, lse, want):
    o_ref, l_ref = want
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    err = np.abs(o - o_ref)
    assert np.isfinite(o).all()
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
    assert np.array_equal(np.isneginf(lse), np.isneginf(l_ref))
    fin = np.isfinite(l_ref)
    if fin.any():
        assert np.abs(lse[fin] - l_ref[fin]).max() <= 1e-3


def _case(B, h, n_q, L_max, lens, seed=0, d=64):
    w = Workload("dec", B, h, n_q, L_max, d, MASK_KEY_PADDING, "bf16", kind="decode")
    q, k, v, _ = inputs.make_inputs(w, device="cuda", seeds=(seed, seed + 1, seed + 2, seed + 3))
    kl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    return w, q, k, v, kl


LENS = [0, 1, 2, 127, 128, 129, 300, 511, 600, 600]


@pytest.mark.parametrize("d", [64, 128, 32, 16])
@pytest.mark.parametrize("window", [0, 1, 100, 127, 128, 299, 5000])
def test_decode_window_matches_oracle(d, window):
    w, q, k, v, kl = _case(len(LENS), 2, 3, 600, LENS, seed=11, d=d)
    o, lse = binding.attn_decode(q, k, v, kl, scale=w.scale, window=window)
    binding.check()
    _check(o, lse, _expected(q, k, v, LENS, window, w.scale))


@pytest.mark.parametrize("n_q", [1, 2, 8])
def test_decode_window_query_counts(n_q):
    lens = [1000, 37, 513]
    w, q, k, v, kl = _case(3, 4, n_q, 1024, lens, seed=21)
    o, lse = binding.attn_decode(q, k, v, kl, scale=w.scale, window=200)
    binding.check()
    _check(o, lse, _expected(q, k, v, lens, 200, w.scale))


@pytest.mark.parametrize("d", [64, 128])
def test_decode_window_split_cache(d):
    # few heads and a long window: the window's keys are split across CTAs
    # and merged by the second kernel; a short window of the same cache is not
    assert binding.decode_workspace_bytes(1, 2, 1, 4096, d, window=3000) > 0
    assert (binding.decode_workspace_bytes(1, 2, 1, 4096, d, window=100)
            <= binding.decode_workspace_bytes(1, 2, 1, 4096, d))
    lens = [4096, 3500]
    for window in (3000, 100, 2000):
        w, q, k, v, kl = _case(2, 2, 1, 4096, lens, seed=31, d=d)
        o, lse = binding.attn_decode(q, k, v, kl, scale=w.scale, window=window)
        binding.check()
        _check(o, lse, _expected(q, k, v, lens, window, w.scale))


@pytest.mark.parametrize("d", [64, 32])
def test_decode_wide_window_equals_attn_decode(d):
    # a window reaching the start of every cache is attn_decode itself: the
    # same plan and the same kernels, so the same bits
    lens = [5, 700, 1024, 1]
    w, q, k, v, kl = _case(4, 3, 2, 1024, lens, seed=41, d=d)
    a = binding.attn_decode(q, k, v, kl, scale=w.scale)
    b = binding.attn_decode(q, k, v, kl, scale=w.scale, window=1023)
    c = binding.attn_decode(q, k, v, kl, scale=w.scale, window=10 ** 6)
    binding.check()
    for x in (b, c):
        assert torch.equal(a[0], x[0]) and torch.equal(a[1], x[1])


@pytest.mark.parametrize("d", [64, 128, 16])
def test_decode_window_never_reads_keys_before_the_window(d):
    lens = [600, 130, 64]
    window = 50
    w, q, k, v, kl = _case(3, 2, 1, 640, lens, seed=51, d=d)
    want = _expected(q, k, v, lens, window, w.scale)
    for b, L in enumerate(lens):  # NaN before each window
        lo = max(0, L - 1 - window)
        k[b, :, :lo] = float("nan")
        v[b, :, :lo] = float("nan")
    o, lse = binding.attn_decode(q, k, v, kl, scale=w.scale, window=window)
    binding.check()
    _check(o, lse, want)


def test_decode_window_long_workload_every_row():
    # the bench's restricted decoding workload (32 x 16 heads, caches of
    # 2048-4096 keys, the newest 1024 positions), every output row compared,
    # in the launch configuration the bench times
    w = inputs.WORKLOADS["decode_long_window"]
    q, k, v, kl = inputs.make_inputs(w, device="cuda")
    o, lse = binding.attn_decode(q, k, v, kl, scale=w.scale, window=inputs.decode_window(w))
    binding.check()
    _check(o, lse, _expected(q, k, v, kl.cpu().tolist(), inputs.decode_window(w), w.scale))

"""GPU parity of the decoding path (a few new queries against a key/value
cache) with the float64 oracle: the same operation as the fused forward with
key padding, so the oracle is called with the cache lengths as key lengths.
Tolerances as for the bf16 forward: max |dO| <= 2e-2, mean |dO| <= 2e-3,
|dLSE| <= 1e-3 (this path keeps P in float32, so it lands far inside them).
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


def _check(o, lse, q, k, v, lens, scale):
    mask = MASK_NONE if lens is None else MASK_KEY_PADDING
    o_ref, l_ref = oracle.attn_fwd(q, k, v, scale, mask, lens)
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


@pytest.mark.parametrize("n_q", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("shape", [(3, 2, 300), (2, 4, 1000), (1, 1, 1), (4, 3, 129), (1, 2, 4096)])
def test_decode_matches_oracle(n_q, shape):
    B, h, L = shape
    lens = [max(0, (L * (b + 1)) // B - b) for b in range(B)]
    w, q, k, v, kl = _case(B, h, n_q, L, lens)
    o, lse = binding.attn_decode(q, k, v, kl, scale=w.scale)
    binding.check()
    _check(o, lse, q, k, v, kl, w.scale)


def test_decode_tile_boundary_lengths_and_empty_cache():
    lens = [0, 1, 127, 128, 129, 255, 256, 257, 511, 512]
    w, q, k, v, kl = _case(len(lens), 2, 2, 512, lens)
    o, lse = binding.attn_decode(q, k, v, kl, scale=w.scale)
    binding.check()
    _check(o, lse, q, k, v, kl, w.scale)


def test_decode_split_and_unsplit_paths():
    # few heads and a long cache: chunks merged by the second kernel
    assert binding.decode_workspace_bytes(1, 2, 1, 4096) > 0
    # many heads: one unit per head, no workspace
    assert binding.decode_workspace_bytes(256, 8, 1, 512) == 0
    for B, h, L in ((1, 2, 4096), (256, 8, 512)):
        lens = list(np.random.default_rng(B).integers(1, L + 1, size=B))
        w, q, k, v, kl = _case(B, h, 1, L, lens, seed=5)
        o, lse = binding.attn_decode(q, k, v, kl, scale=w.scale)
        binding.check()
        _check(o, lse, q, k, v, kl, w.scale)


def test_decode_without_lengths_uses_whole_cache():
    w, q, k, v, _ = _case(2, 3, 2, 700, None)
    o, lse = binding.attn_decode(q, k, v, None, scale=w.scale)
    binding.check()
    _check(o, lse, q, k, v, None, w.scale)


def test_decode_ignores_cache_past_lengths():
    """Cache rows past the filled length may hold anything, NaN included."""
    lens = [5, 300, 0, 129]
    w, q, k, v, kl = _case(4, 2, 1, 512, lens)
    o_ref, l_ref = binding.attn_decode(q, k, v, kl, scale=w.scale)
    k2, v2 = k.clone(), v.clone()
    for b, L in enumerate(lens):
        k2[b, :, L:] = float("nan")
        v2[b, :, L:] = float("nan")
    o, lse = binding.attn_decode(q, k2, v2, kl, scale=w.scale)
    binding.check()
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_decode_rejects_short_workspace():
    w, q, k, v, kl = _case(1, 2, 1, 4096, [4096])
    need = binding.decode_workspace_bytes(1, 2, 1, 4096)
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    rc = binding.attn_decode_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), None,
                                 1, 2, 1, 4096, 64, w.scale, kl.data_ptr(), ws.data_ptr(),
                                 ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert rc == binding.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["decode_beam", "decode_long"])
def test_decode_workloads_full(name):
    """The decoding workloads the benchmark times, every output row."""
    w = inputs.WORKLOADS[name]
    q, k, v, kl = inputs.make_inputs(w, device="cuda")
    o, lse = binding.attn_decode(q, k, v, kl, scale=w.scale)
    binding.check()
    _check(o, lse, q, k, v, kl, w.scale)


@pytest.mark.parametrize("B,h,L_max", [
    (600, 4, 300),    # several units per CTA, ordered longest first
    (1100, 1, 64),    # more (batch entry, split) pairs than the ordering takes: index order
    (1000, 16, 32),   # more units per CTA than its schedule holds: index order
    (40, 2, 3000),    # split caches: (batch entry, split) pairs ordered by key count
])
def test_decode_many_units_every_row(B, h, L_max):
    """Every unit is processed exactly once whatever order the CTAs take them in:
    random lengths (zeros and full caches included), every output row checked."""
    rng = np.random.default_rng(B * 7 + h)
    lens = rng.integers(0, L_max + 1, size=B)
    lens[:3] = [0, L_max, 1]
    w, q, k, v, kl = _case(B, h, 1, L_max, lens.tolist(), seed=3)
    o, lse = binding.attn_decode(q, k, v, kl, scale=w.scale)
    binding.check()
    _check(o, lse, q, k, v, kl, w.scale)



@pytest.mark.parametrize("d", [16, 32, 128])
@pytest.mark.parametrize("n_q", [1, 3, 8])
@pytest.mark.parametrize("shape", [(3, 2, 300), (1, 2, 4096), (40, 4, 200)])
def test_decode_other_head_sizes_match_oracle(d, n_q, shape):
    """Head sizes 16, 32 and 128 (Table 3 of the paper): split and unsplit caches,
    lengths from empty to full, every output row checked."""
    B, h, L = shape
    rng = np.random.default_rng(B + 7 * n_q + d)
    lens = rng.integers(0, L + 1, size=B)
    lens[0] = L
    if B > 2:
        lens[1] = 0
    w, q, k, v, kl = _case(B, h, n_q, L, lens.tolist(), seed=5, d=d)
    o, lse = binding.attn_decode(q, k, v, kl, scale=w.scale)
    binding.check()
    _check(o, lse, q, k, v, kl, w.scale)


@pytest.mark.parametrize("d", [16, 128])
def test_decode_other_head_sizes_without_lengths_and_nan_tail(d):
    """No lengths: the whole cache; with lengths, NaN past them is never read."""
    w, q, k, v, _ = _case(2, 3, 2, 700, None, seed=6, d=d)
    o, lse = binding.attn_decode(q, k, v, None, scale=w.scale)
    binding.check()
    _check(o, lse, q, k, v, None, w.scale)
    lens = [5, 300]
    w, q, k, v, kl = _case(2, 2, 1, 512, lens, seed=7, d=d)
    k2, v2 = k.clone(), v.clone()
    for b, L in enumerate(lens):
        k2[b, :, L:] = float("nan")
        v2[b, :, L:] = float("nan")
    o, lse = binding.attn_decode(q, k2, v2, kl, scale=w.scale)
    binding.check()
    _check(o, lse, q, k, v, kl, w.scale)


@pytest.mark.parametrize("d", [64, 128, 16])
@pytest.mark.parametrize("B,h,n_q,L_max", [(6, 4, 2, 700), (1, 2, 1, 4096)])
def test_decode_strided_caches_equal_contiguous(d, B, h, n_q, L_max):
    """Caches kept [B, L_max, h, d] and outputs written into a [B, n_q, h, d]
    buffer: the same results as the contiguous call, bit for bit, and the oracle's."""
    rng = np.random.default_rng(d + B)
    lens = rng.integers(0, L_max + 1, size=B)
    lens[0] = L_max
    w, q, k, v, kl = _case(B, h, n_q, L_max, lens.tolist(), seed=8, d=d)
    ks, vs = (t.transpose(1, 2).contiguous().transpose(1, 2) for t in (k, v))  # [B, L, h, d]
    qs = q.transpose(1, 2).contiguous().transpose(1, 2)
    out = torch.full((B, n_q, h, d), float("nan"), dtype=torch.bfloat16,
                     device="cuda").transpose(1, 2)
    o, lse = binding.attn_decode_strided(qs, ks, vs, kl, scale=w.scale, out=out)
    o_ref, lse_ref = binding.attn_decode(q, k, v, kl, scale=w.scale)
    binding.check()
    assert torch.equal(o.contiguous(), o_ref) and torch.equal(lse, lse_ref)
    _check(o.contiguous(), lse, q, k, v, kl, w.scale)

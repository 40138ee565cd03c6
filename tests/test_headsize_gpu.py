"""GPU parity of the tensor-core forward at the other head sizes of "Attention
Is All You Need", Table 3, rows (A) and (B): d_k = d_v in {16, 32, 128}
(d = 64 is covered by test_parity_gpu.py), every mask, against the float64
oracle with the forward's bf16 tolerances: max |O - O_ref| <= 2e-2,
mean |O - O_ref| <= 2e-3, |LSE - LSE_ref| <= 1e-3."""
import math

import numpy as np
import pytest
import torch

import oracle
from transformer_head_scaled_gb300 import binding, inputs
from transformer_head_scaled_gb300.inputs import MASK_CAUSAL, MASK_KEY_PADDING, MASK_NONE

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


def _inputs(B, h, n_q, n_k, d, seed=0):
    q = inputs.gaussian((B, h, n_q, d), seed).to(torch.bfloat16)
    k = inputs.gaussian((B, h, n_k, d), seed + 1).to(torch.bfloat16)
    v = inputs.gaussian((B, h, n_k, d), seed + 2).to(torch.bfloat16)
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
    # B, h, n_q, n_k, mask, lens
    (2, 2, 300, 333, MASK_NONE, None),       # ragged tails of both tile kinds
    (1, 2, 512, 512, MASK_CAUSAL, None),
    (1, 1, 200, 456, MASK_CAUSAL, None),     # n_q < n_k
    (3, 2, 200, 300, MASK_KEY_PADDING, [77, 300, 0]),
    (1, 1, 1, 1, MASK_NONE, None),
]


@pytest.mark.parametrize("d", [16, 32, 128])
@pytest.mark.parametrize("B,h,n_q,n_k,mask,lens", CASES)
def test_head_size_matches_oracle(d, B, h, n_q, n_k, mask, lens):
    q, k, v = _inputs(B, h, n_q, n_k, d)
    kl = None if lens is None else torch.tensor(lens, dtype=torch.int32)
    scale = 1.0 / math.sqrt(d)
    o, lse = binding.attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, mask=mask,
                              key_lens=None if kl is None else kl.cuda())
    binding.check()
    o_ref, l_ref = oracle.attn_fwd(q, k, v, scale, mask, kl)
    _compare(o, lse, o_ref, l_ref)


@pytest.mark.parametrize("d", [16, 32, 128])
def test_head_size_window_matches_oracle(d):
    q, k, v = _inputs(1, 2, 400, 400, d, seed=3)
    scale = 1.0 / math.sqrt(d)
    o, lse = binding.attn_fwd_window(q.cuda(), k.cuda(), v.cuda(), 50, 70, scale=scale)
    binding.check()
    o_ref, l_ref = oracle.attn_band(q, k, v, scale, 50, 70)
    _compare(o, lse, o_ref, l_ref)


@pytest.mark.parametrize("name", ["base_h4_d128", "base_h16_d32", "base_h32_d16"])
def test_head_size_full_workload_whole_tensor(name):
    """The benchmark's head-size workloads, every element against the oracle."""
    w = inputs.WORKLOADS[name]
    q, k, v, kl = inputs.make_inputs(w, device="cuda")
    o, lse = binding.attn_fwd(q, k, v, scale=w.scale, mask=w.mask, key_lens=kl)
    binding.check()
    o_ref, l_ref = oracle.attn_fwd(q, k, v, w.scale, w.mask, kl)
    _compare(o, lse, o_ref, l_ref)


@pytest.mark.parametrize("d", [16, 32, 128])
def test_head_size_many_items_per_cta(d):
    """B=16, h=8, n=1024 under the causal mask: 512 work items, several per
    persistent CTA, each element compared."""
    q, k, v = _inputs(16, 8, 1024, 1024, d, seed=31)
    scale = 1.0 / math.sqrt(d)
    o, lse = binding.attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, mask=MASK_CAUSAL)
    binding.check()
    o_ref, l_ref = oracle.attn_fwd(q, k, v, scale, MASK_CAUSAL)
    _compare(o, lse, o_ref, l_ref)

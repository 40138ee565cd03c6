"""GPU parity of the strided backward (attn_bwd_strided) with the float64
oracle, on the layouts a projection to h heads produces: [B, n, h, d] views
and Q, K, V packed in one [B, n, 3, h, d] buffer, with the gradients written
into the same kinds of views.  The strided path runs the same kernels as
attn_bwd with other tensor maps and row offsets, so dK and dV (each
accumulated inside one CTA) must equal attn_bwd's bit for bit; dQ, whose key
tiles' contributions are added in arrival order, is compared with the oracle
under the backward's tolerances (relative l2 <= 5e-3, max <= 1.5e-2 of the
largest entry)."""
import math

import numpy as np
import pytest
import torch

import oracle
from transformer_head_scaled_gb300 import binding, inputs
from transformer_head_scaled_gb300.inputs import MASK_CAUSAL, MASK_KEY_PADDING, MASK_NONE

pytestmark = pytest.mark.gpu

REL_L2 = 5e-3
MAX_REL = 1.5e-2


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from transformer_head_scaled_gb300.build import build
    build()
    oracle.build()
    return binding.load()


def _bf16(shape, seed):
    return inputs.gaussian(shape, seed).to(torch.bfloat16)


def _compare(got, want):
    for name, a, b in zip(("dq", "dk", "dv"), got, want):
        a = a.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(a).all(), name
        if np.abs(b).max() == 0:
            assert np.abs(a).max() == 0, name
            continue
        rel = np.linalg.norm(a - b) / np.linalg.norm(b)
        mrel = np.abs(a - b).max() / np.abs(b).max()
        assert rel <= REL_L2 and mrel <= MAX_REL, (name, rel, mrel)


def _contig(t):
    return t.contiguous().cpu()


CASES = [
    # B, h, n_q, n_k, d, mask, lens, window
    (2, 3, 200, 200, 64, MASK_NONE, None, None),
    (1, 4, 300, 300, 64, MASK_CAUSAL, None, None),
    (3, 2, 100, 330, 64, MASK_KEY_PADDING, [128, 0, 301], None),
    (1, 2, 640, 640, 64, MASK_NONE, None, (127, 129)),
    (2, 2, 256, 256, 32, MASK_CAUSAL, None, None),
    (2, 2, 200, 200, 16, MASK_NONE, None, None),
]


@pytest.mark.parametrize("B,h,n_q,n_k,d,mask,lens,window", CASES)
def test_bwd_bshd_views_match_oracle_and_contiguous(B, h, n_q, n_k, d, mask, lens, window):
    """Inputs and gradients as [B, n, h, d] buffers seen through transposed views."""
    scale = 1 / math.sqrt(d)

    def bshd(n, seed):
        return _bf16((B, n, h, d), seed).cuda().transpose(1, 2)   # [B, h, n, d] view
    q, k, v, g = bshd(n_q, 20), bshd(n_k, 21), bshd(n_k, 22), bshd(n_q, 23)
    kl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    o = torch.empty((B, n_q, h, d), dtype=torch.bfloat16, device="cuda").transpose(1, 2)
    o, lse = binding.attn_fwd_strided(q, k, v, scale=scale, mask=mask, key_lens=kl, window=window,
                                      out=o)
    dq, dk, dv = (torch.full((B, n, h, d), float("nan"), dtype=torch.bfloat16,
                             device="cuda").transpose(1, 2) for n in (n_q, n_k, n_k))
    binding.attn_bwd_strided(q, k, v, o, lse, g, dq, dk, dv, scale=scale, mask=mask, key_lens=kl,
                             window=window)
    binding.check()
    qc, kc, vc, gc = (_contig(t) for t in (q, k, v, g))
    if window is not None:
        want = oracle.attn_bwd_band(qc, kc, vc, gc, scale, window[0], window[1])
    else:
        want = oracle.attn_bwd(qc, kc, vc, gc, scale, mask, None if lens is None else np.array(lens))
    _compare([dq, dk, dv], want)
    # the contiguous entry point on contiguous copies: dK and dV bit for bit
    ref = binding.attn_bwd(q.contiguous(), k.contiguous(), v.contiguous(), o.contiguous(), lse,
                           g.contiguous(), scale=scale, mask=mask, key_lens=kl, window=window)
    binding.check()
    assert torch.equal(dk.contiguous(), ref[1]) and torch.equal(dv.contiguous(), ref[2])


def test_bwd_packed_qkv_gradient_buffer():
    """Q, K, V as slices of one [B, n, 3, h, d] projection output; the gradients
    land in the matching slices of one packed buffer and nowhere else."""
    B, n, h, d = 2, 384, 4, 64
    scale = 1 / math.sqrt(d)
    qkv = _bf16((B, n, 3, h, d), 30).cuda()
    q, k, v = (qkv[:, :, i].transpose(1, 2) for i in range(3))
    g = _bf16((B, n, h, d), 31).cuda().transpose(1, 2)
    o, lse = binding.attn_fwd_strided(q, k, v, scale=scale, mask=MASK_CAUSAL)
    dqkv = torch.full((B, n, 3, h, d + 8), 7.0, dtype=torch.bfloat16, device="cuda")
    grads = [dqkv[:, :, i, :, :d].transpose(1, 2) for i in range(3)]
    binding.attn_bwd_strided(q, k, v, o, lse, g, *grads, scale=scale, mask=MASK_CAUSAL)
    binding.check()
    assert torch.all(dqkv[..., d:] == 7.0)   # the padding columns are untouched
    want = oracle.attn_bwd(*(_contig(t) for t in (q, k, v, g)), scale, MASK_CAUSAL, None)
    _compare(grads, want)

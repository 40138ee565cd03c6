"""GPU parity of the strided forward (attn_fwd_strided): tensors in the
[B, n, h, d] layout a projection to heads produces, and Q, K, V packed in one
[B, n, 3, h, d] buffer, read and written in place.  The result must equal
the contiguous forward bit for bit (same tiles, same arithmetic) and the
oracle within the forward's bf16 tolerances (max 2e-2, mean 2e-3, LSE 1e-3)."""
import math

import numpy as np
import pytest
import torch

import oracle
from transformer_head_scaled_gb300 import binding, inputs
from transformer_head_scaled_gb300.inputs import MASK_CAUSAL, MASK_KEY_PADDING, MASK_NONE

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from transformer_head_scaled_gb300.build import build
    build()
    oracle.build()
    return binding.load()


def _bshd(B, n, h, d, seed):
    """A [B, h, n, d] view of [B, n, h, d] storage."""
    return inputs.gaussian((B, n, h, d), seed).to(torch.bfloat16).cuda().transpose(1, 2)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("mask", [MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING])
def test_bshd_equals_contiguous_and_oracle(d, mask):
    B, h, n_q, n_k = 2, 3, 300, 300
    q, k, v = _bshd(B, n_q, h, d, 0), _bshd(B, n_k, h, d, 1), _bshd(B, n_k, h, d, 2)
    lens = torch.tensor([77, 300], dtype=torch.int32, device="cuda") if mask == MASK_KEY_PADDING else None
    out_store = torch.empty((B, n_q, h, d), dtype=torch.bfloat16, device="cuda")
    o, lse = binding.attn_fwd_strided(q, k, v, mask=mask, key_lens=lens, out=out_store.transpose(1, 2))
    ref_o, ref_lse = binding.attn_fwd(q.contiguous(), k.contiguous(), v.contiguous(), mask=mask,
                                      key_lens=lens)
    binding.check()
    assert torch.equal(out_store.transpose(1, 2), ref_o) and torch.equal(lse, ref_lse)
    o64, l64 = oracle.attn_fwd(q, k, v, 1 / math.sqrt(d), mask, lens)
    err = np.abs(o.float().cpu().numpy() - o64)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3
    fin = np.isfinite(l64)
    assert np.abs(lse.cpu().numpy()[fin] - l64[fin]).max() <= 1e-3


def test_packed_qkv_buffer_and_window():
    B, n, h, d = 2, 513, 4, 64
    buf = inputs.gaussian((B, n, 3, h, d), 5).to(torch.bfloat16).cuda()
    q, k, v = (buf[:, :, i].transpose(1, 2) for i in range(3))
    for window in (None, (40, 0), (64, 64)):
        o, lse = binding.attn_fwd_strided(q, k, v, window=window)
        if window is None:
            ref = binding.attn_fwd(q.contiguous(), k.contiguous(), v.contiguous())
        else:
            ref = binding.attn_fwd_window(q.contiguous(), k.contiguous(), v.contiguous(), *window)
        binding.check()
        assert torch.equal(o, ref[0]) and torch.equal(lse, ref[1])
    o64, _ = oracle.attn_band(q, k, v, 0.125, 64, 64)
    assert np.abs(o.float().cpu().numpy() - o64).max() <= 2e-2


def test_full_size_bshd_base_encoder_whole_tensor():
    """The base encoder workload (1024 work items) read from and written to
    [B, n, h, d] storage, every element against the oracle."""
    w = inputs.WORKLOADS["base_enc"]
    q, k, v = (_bshd(w.B, w.n_q, w.h, w.d, s) for s in (0, 1, 2))
    o, lse = binding.attn_fwd_strided(q, k, v)
    binding.check()
    o64, l64 = oracle.attn_fwd(q, k, v, w.scale)
    err = np.abs(o.float().cpu().numpy() - o64)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3
    assert np.abs(lse.cpu().numpy() - l64).max() <= 1e-3

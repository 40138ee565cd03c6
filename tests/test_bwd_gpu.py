"""GPU parity of the backward (attn_bwd) against the float64 oracle.

The inputs q, k, v, dO are bf16 (the oracle sees the same bf16 values widened
to float64); o and lse come from attn_fwd on the GPU, as in training.  Each
gradient G in {dQ, dK, dV} is compared with the oracle's G_ref by

    ||G - G_ref||_2 / ||G_ref||_2 <= REL_L2    and    max|G - G_ref| <= MAX_REL * max|G_ref|

Where the bounds come from: four independent bf16 roundings reach each
gradient (P before dV, dS before dK and dQ, the forward's O inside D, and the
output itself), each a relative error uniform within +-2^-9, i.e. an rms of
2^-9/sqrt(3) = 1.1e-3; together about 2.2e-3 relative l2.  REL_L2 allows a
little over twice that; MAX_REL bounds the largest single deviation, which for
these Gaussian inputs stays within a few rms of the largest entry.  Small cases
and every full-size workload compare every element; the sampled-head cases
kept beside them compare whole heads, each head's gradients depending only on
that head's data.
"""
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


def _problem(B, h, n_q, n_k, seed=0, d=64):
    q = _bf16((B, h, n_q, d), seed)
    k = _bf16((B, h, n_k, d), seed + 1)
    v = _bf16((B, h, n_k, d), seed + 2)
    g = _bf16((B, h, n_q, d), seed + 3)
    return q, k, v, g


def _gpu_grads(q, k, v, g, mask, lens, scale):
    qc, kc, vc, gc = (t.cuda() for t in (q, k, v, g))
    lc = None if lens is None else torch.as_tensor(lens, dtype=torch.int32).cuda()
    o, lse = binding.attn_fwd(qc, kc, vc, scale=scale, mask=mask, key_lens=lc)
    dq, dk, dv = binding.attn_bwd(qc, kc, vc, o, lse, gc, scale=scale, mask=mask, key_lens=lc)
    binding.check()
    return [t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv)]


def _compare(got, want, names=("dq", "dk", "dv")):
    stats = {}
    for name, a, b in zip(names, got, want):
        assert np.isfinite(a).all(), name
        scale_l2 = np.linalg.norm(b)
        scale_max = np.abs(b).max()
        err = np.abs(a - b)
        if scale_max == 0:
            assert err.max() == 0, f"{name}: expected exact zeros, max {err.max():.3g}"
            stats[name] = (0.0, 0.0)
            continue
        rel = np.linalg.norm(a - b) / scale_l2
        mrel = err.max() / scale_max
        stats[name] = (rel, mrel)
        assert rel <= REL_L2, f"{name}: relative l2 error {rel:.3g}"
        assert mrel <= MAX_REL, f"{name}: max error {mrel:.3g} of max |ref|"
    print(" ".join(f"{n}: l2 {r:.2e} max {m:.2e}" for n, (r, m) in stats.items()))
    return stats


CASES = [
    # (B, h, n_q, n_k, mask, lens)
    (1, 2, 128, 128, MASK_NONE, None),
    (2, 3, 200, 328, MASK_NONE, None),
    (2, 1, 5, 700, MASK_NONE, None),
    (1, 2, 512, 512, MASK_CAUSAL, None),
    (2, 2, 300, 300, MASK_CAUSAL, None),
    (1, 2, 256, 384, MASK_CAUSAL, None),
    (1, 1, 384, 200, MASK_CAUSAL, None),
    (4, 2, 256, 384, MASK_KEY_PADDING, [0, 1, 129, 384]),
    (3, 2, 100, 130, MASK_KEY_PADDING, [128, 5, 130]),
]


@pytest.mark.parametrize("B,h,n_q,n_k,mask,lens", CASES)
def test_bwd_matches_oracle(B, h, n_q, n_k, mask, lens):
    q, k, v, g = _problem(B, h, n_q, n_k)
    scale = 1 / math.sqrt(64)
    got = _gpu_grads(q, k, v, g, mask, lens, scale)
    want = oracle.attn_bwd(q, k, v, g, scale, mask, None if lens is None else np.array(lens))
    _compare(got, want)


def test_bwd_single_key_and_query():
    """One key: P = 1, dV = dO and the score gradients vanish (up to fp32 rounding)."""
    q, k, v, g = _problem(1, 1, 1, 1, seed=5)
    dq, dk, dv = _gpu_grads(q, k, v, g, MASK_NONE, None, 0.125)
    np.testing.assert_allclose(dv, g.double().numpy(), rtol=2 ** -8)
    assert np.abs(dq).max() < 1e-3 and np.abs(dk).max() < 1e-3


def test_bwd_masked_keys_and_empty_sequences_are_exact_zeros():
    q, k, v, g = _problem(3, 2, 160, 300, seed=9)
    lens = [0, 77, 300]
    dq, dk, dv = _gpu_grads(q, k, v, g, MASK_KEY_PADDING, lens, 0.125)
    assert np.all(dq[0] == 0) and np.all(dk[0] == 0) and np.all(dv[0] == 0)
    assert np.all(dk[1, :, 77:] == 0) and np.all(dv[1, :, 77:] == 0)
    # under the causal mask keys no query reaches (j >= n_q) get zeros
    q, k, v, g = _problem(1, 2, 130, 400, seed=4)
    _, dk, dv = _gpu_grads(q, k, v, g, MASK_CAUSAL, None, 0.125)
    assert np.all(dk[:, :, 130:] == 0) and np.all(dv[:, :, 130:] == 0)


def test_bwd_workspace_contents_do_not_matter_and_dk_dv_repeat():
    """dK and dV are accumulated inside one CTA each: bitwise repeatable.  dQ
    sums the key tiles' contributions in whatever order they land, so it is
    compared to the oracle rather than bitwise."""
    q, k, v, g = (t.cuda() for t in _problem(2, 2, 256, 256, seed=3))
    o, lse = binding.attn_fwd(q, k, v)
    need = binding.bwd_workspace_bytes(2, 2, 256)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN patterns
    a = binding.attn_bwd(q, k, v, o, lse, g, workspace=ws)
    binding.check()
    ws.fill_(0x7F)
    b = binding.attn_bwd(q, k, v, o, lse, g, workspace=ws)
    binding.check()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    want = oracle.attn_bwd(q, k, v, g, 0.125)
    _compare([t.float().cpu().numpy().astype(np.float64) for t in b], want)


def test_bwd_launch_count():
    q, k, v, g = (t.cuda() for t in _problem(1, 1, 128, 128))
    o, lse = binding.attn_fwd(q, k, v)
    before = binding.launch_count()
    binding.attn_bwd(q, k, v, o, lse, g)
    binding.check()
    assert binding.launch_count() - before == 3


@pytest.mark.parametrize("name", ["base_enc", "base_dec", "encdec", "big", "base_h16_d32",
                                  "base_h32_d16"])
def test_bwd_full_size_sampled_heads(name):
    """Full-size workloads in the launch configuration the benchmark times;
    the oracle recomputes a few whole heads (first, last and random ones)."""
    w = inputs.WORKLOADS[name]
    q, k, v, lens = inputs.make_inputs(w, device="cuda")
    g = inputs.gaussian((w.B, w.h, w.n_q, w.d), 4).to(torch.bfloat16).cuda()
    o, lse = binding.attn_fwd(q, k, v, scale=w.scale, mask=w.mask, key_lens=lens)
    dq, dk, dv = binding.attn_bwd(q, k, v, o, lse, g, scale=w.scale, mask=w.mask, key_lens=lens)
    binding.check()
    BH = w.B * w.h
    rng = np.random.default_rng(0)
    n_heads = 2 if w.n_q >= 4096 else 6
    sel = sorted({0, BH - 1, *rng.integers(0, BH, size=n_heads - 2).tolist()})
    b_idx = [s // w.h for s in sel]
    h_idx = [s % w.h for s in sel]

    def pick(t):
        return t[b_idx, h_idx].unsqueeze(1).cpu()

    sub_lens = None
    if lens is not None:
        sub_lens = lens.cpu().numpy()[b_idx].astype(np.int32)
    want = oracle.attn_bwd(pick(q), pick(k), pick(v), pick(g), w.scale, w.mask, sub_lens)
    got = [pick(t).float().numpy().astype(np.float64) for t in (dq, dk, dv)]
    _compare(got, want)
    # a property over every head: each row set's key gradients sum to zero
    if w.mask == MASK_NONE:
        dks = dk.float().sum(dim=2)
        assert dks.abs().max().item() <= 0.05 * dk.float().abs().max().item() * math.sqrt(w.n_k)


@pytest.mark.parametrize("name", ["base_enc", "base_dec", "encdec", "base_h16_d32",
                                  "base_h32_d16", "big", "big_causal"])
def test_bwd_full_size_whole_tensor(name):
    """Full-size workloads in the launch configuration the benchmark times,
    every element of dQ, dK and dV against the oracle (every head: every
    work item of every persistent CTA)."""
    w = inputs.WORKLOADS[name]
    q, k, v, lens = inputs.make_inputs(w, device="cuda")
    g = inputs.gaussian((w.B, w.h, w.n_q, w.d), 4).to(torch.bfloat16).cuda()
    o, lse = binding.attn_fwd(q, k, v, scale=w.scale, mask=w.mask, key_lens=lens)
    dq, dk, dv = binding.attn_bwd(q, k, v, o, lse, g, scale=w.scale, mask=w.mask, key_lens=lens)
    binding.check()
    want = oracle.attn_bwd(q.cpu(), k.cpu(), v.cpu(), g.cpu(), w.scale, w.mask,
                           None if lens is None else lens.cpu().numpy().astype(np.int32))
    got = [t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv)]
    _compare(got, want)


# ---------------------------------------------------------------- restricted window

WINDOW_CASES = [
    # B, h, n_q, n_k, left, right
    (1, 2, 300, 300, 64, 64),
    (1, 2, 512, 512, 128, 0),     # causal window
    (2, 1, 200, 333, 0, 50),
    (1, 1, 700, 100, 20, 20),     # queries past the last key: empty windows
    (1, 2, 640, 640, 127, 129),   # window edges one off the tile size
]


@pytest.mark.parametrize("B,h,n_q,n_k,left,right", WINDOW_CASES)
def test_bwd_window_matches_oracle(B, h, n_q, n_k, left, right):
    q, k, v, g = _problem(B, h, n_q, n_k, seed=2)
    qc, kc, vc, gc = (t.cuda() for t in (q, k, v, g))
    o, lse = binding.attn_fwd_window(qc, kc, vc, left, right)
    grads = binding.attn_bwd(qc, kc, vc, o, lse, gc, window=(left, right))
    binding.check()
    want = oracle.attn_bwd_band(q, k, v, g, 0.125, left, right)
    _compare([t.float().cpu().numpy().astype(np.float64) for t in grads], want)


def test_bwd_window_wide_equals_unmasked_bit_for_bit():
    q, k, v, g = (t.cuda() for t in _problem(1, 2, 384, 384, seed=6))
    o, lse = binding.attn_fwd(q, k, v)
    a = binding.attn_bwd(q, k, v, o, lse, g, window=(10 ** 6, 10 ** 6))
    b = binding.attn_bwd(q, k, v, o, lse, g)
    binding.check()
    # dK and dV accumulate inside one CTA each in the same order
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def test_bwd_window_full_size_sampled_heads():
    w = inputs.WORKLOADS["big_window"]
    q, k, v, _ = inputs.make_inputs(w, device="cuda")
    g = inputs.gaussian((w.B, w.h, w.n_q, w.d), 4).to(torch.bfloat16).cuda()
    o, lse = binding.attn_fwd_window(q, k, v, w.win_left, w.win_right)
    dq, dk, dv = binding.attn_bwd(q, k, v, o, lse, g, window=(w.win_left, w.win_right))
    binding.check()
    sel = [0, w.B * w.h - 1]
    b_idx, h_idx = [s // w.h for s in sel], [s % w.h for s in sel]

    def pick(t):
        return t[b_idx, h_idx].unsqueeze(1).cpu()

    want = oracle.attn_bwd_band(pick(q), pick(k), pick(v), pick(g), w.scale, w.win_left,
                                w.win_right)
    _compare([pick(t).float().numpy().astype(np.float64) for t in (dq, dk, dv)], want)


def test_bwd_window_full_size_whole_tensor():
    """The restricted-window workload (big model, window of 513 positions),
    every element of the three gradients against the band oracle."""
    w = inputs.WORKLOADS["big_window"]
    q, k, v, _ = inputs.make_inputs(w, device="cuda")
    g = inputs.gaussian((w.B, w.h, w.n_q, w.d), 4).to(torch.bfloat16).cuda()
    o, lse = binding.attn_fwd_window(q, k, v, w.win_left, w.win_right)
    dq, dk, dv = binding.attn_bwd(q, k, v, o, lse, g, window=(w.win_left, w.win_right))
    binding.check()
    want = oracle.attn_bwd_band(q.cpu(), k.cpu(), v.cpu(), g.cpu(), w.scale, w.win_left,
                                w.win_right)
    _compare([t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv)], want)


# ---------------------------------------------------------------- other head sizes

HEAD_SIZE_CASES = [
    # B, h, n_q, n_k, mask, lens
    (1, 2, 128, 128, MASK_NONE, None),
    (2, 3, 200, 328, MASK_NONE, None),
    (2, 2, 300, 300, MASK_CAUSAL, None),
    (1, 1, 384, 200, MASK_CAUSAL, None),
    (3, 2, 100, 330, MASK_KEY_PADDING, [128, 0, 301]),
]


@pytest.mark.parametrize("d", [16, 32])
@pytest.mark.parametrize("B,h,n_q,n_k,mask,lens", HEAD_SIZE_CASES)
def test_bwd_head_sizes_match_oracle(d, B, h, n_q, n_k, mask, lens):
    q, k, v, g = _problem(B, h, n_q, n_k, seed=11, d=d)
    scale = 1 / math.sqrt(d)
    got = _gpu_grads(q, k, v, g, mask, lens, scale)
    want = oracle.attn_bwd(q, k, v, g, scale, mask, None if lens is None else np.array(lens))
    _compare(got, want)


@pytest.mark.parametrize("d", [16, 32])
def test_bwd_head_sizes_window_matches_oracle(d):
    q, k, v, g = _problem(1, 2, 640, 640, seed=12, d=d)
    scale = 1 / math.sqrt(d)
    qc, kc, vc, gc = (t.cuda() for t in (q, k, v, g))
    o, lse = binding.attn_fwd_window(qc, kc, vc, 127, 129, scale=scale)
    grads = binding.attn_bwd(qc, kc, vc, o, lse, gc, scale=scale, window=(127, 129))
    binding.check()
    want = oracle.attn_bwd_band(q, k, v, g, scale, 127, 129)
    _compare([t.float().cpu().numpy().astype(np.float64) for t in grads], want)

"""Pins for the float64 backward oracle (oracle.attn_bwd).

The backward is the gradient of eq. (1) of "Attention Is All You Need"
(section 3.2.1) with the masks of section 3.2.3.  None of the pages writes it
out, so every pin here ties it to something other than itself:

* finite differences of the forward oracle, which its own pins tie to the
  pages (central differences on inputs chosen so that every perturbed value
  is exact in float32, with Richardson extrapolation);
* automatic differentiation by PyTorch of the plain float64 expression
  (a library routine, independent of the oracle's C loops);
* closed forms and invariants that hold for any inputs: one key, constant
  values, zero queries, the key-shift invariance of the softmax, the
  homogeneity of the scores in q and k, masked keys, linearity in dO, and
  dV = P^T dO with P read off the forward oracle through V = I.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _grid(shape, seed, step=1.0 / 16, lim=2.0):
    """Values on a coarse binary grid, so that x +- small powers of two stay exact in float32."""
    rng = np.random.default_rng(seed)
    return (np.round(rng.uniform(-lim, lim, size=shape) / step) * step).astype(np.float32)


def _inputs(B=2, H=2, n_q=5, n_k=6, d_k=4, d_v=3, seed=0):
    q = _grid((B, H, n_q, d_k), seed)
    k = _grid((B, H, n_k, d_k), seed + 1)
    v = _grid((B, H, n_k, d_v), seed + 2)
    g = _grid((B, H, n_q, d_v), seed + 3)
    return q, k, v, g


def _loss(q, k, v, g, scale, mask, lens):
    o, _ = oracle.attn_fwd(q, k, v, scale, mask, lens)
    return float((o * g.astype(np.float64)).sum())


CASES = [
    (oracle.MASK_NONE, None),
    (oracle.MASK_CAUSAL, None),
    (oracle.MASK_KEY_PADDING, np.array([3, 6], dtype=np.int32)),
]


@pytest.mark.parametrize("mask,lens", CASES)
def test_finite_differences_of_the_forward(mask, lens):
    q, k, v, g = _inputs()
    scale = 0.5
    dq, dk, dv = oracle.attn_bwd(q, k, v, g, scale, mask, lens)
    rng = np.random.default_rng(11)
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in x.shape)

            def central(h):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = {"q": q, "k": k, "v": v}
                args_m = dict(args_p)
                args_p[name], args_m[name] = xp, xm
                lp = _loss(args_p["q"], args_p["k"], args_p["v"], g, scale, mask, lens)
                lm = _loss(args_m["q"], args_m["k"], args_m["v"], g, scale, mask, lens)
                return (lp - lm) / (2 * h)

            h = 2.0 ** -9
            est = (4 * central(h / 2) - central(h)) / 3  # error O(h^4)
            assert abs(est - grad[idx]) <= 1e-7 + 1e-6 * abs(grad[idx]), (name, idx)


def _torch_grads(q, k, v, g, scale, mask, lens):
    Q, K, V = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    n_q, n_k = q.shape[2], k.shape[2]
    allowed = torch.ones(q.shape[0], 1, n_q, n_k, dtype=torch.bool)
    if mask == oracle.MASK_CAUSAL:
        allowed &= torch.ones(n_q, n_k).tril().bool()
    if mask == oracle.MASK_KEY_PADDING:
        keys = torch.arange(n_k)
        allowed &= (keys[None, :] < torch.tensor(lens)[:, None])[:, None, None, :]
    any_row = allowed.any(-1, keepdim=True)
    s = scale * Q @ K.transpose(-1, -2)
    s = torch.where(allowed, s, torch.tensor(-math.inf, dtype=torch.float64))
    s = torch.where(any_row, s, torch.zeros((), dtype=torch.float64))
    p = torch.softmax(s, dim=-1) * any_row
    o = p @ V
    (o * torch.tensor(g, dtype=torch.float64)).sum().backward()
    return Q.grad.numpy(), K.grad.numpy(), V.grad.numpy()


@pytest.mark.parametrize("mask,lens", CASES + [(oracle.MASK_KEY_PADDING, np.array([0, 2], np.int32))])
@pytest.mark.parametrize("shape", [(2, 3, 7, 9, 5, 6), (1, 2, 9, 4, 8, 8), (2, 1, 1, 1, 3, 2)])
def test_matches_autograd_of_the_plain_expression(mask, lens, shape):
    B, H, n_q, n_k, d_k, d_v = shape
    if lens is not None:
        lens = np.minimum(lens[:B], n_k).astype(np.int32)
        if lens.shape[0] < B:
            lens = np.full(B, n_k, np.int32)
    rng = np.random.default_rng(5)
    q = rng.standard_normal((B, H, n_q, d_k)).astype(np.float32)
    k = rng.standard_normal((B, H, n_k, d_k)).astype(np.float32)
    v = rng.standard_normal((B, H, n_k, d_v)).astype(np.float32)
    g = rng.standard_normal((B, H, n_q, d_v)).astype(np.float32)
    scale = 1 / math.sqrt(d_k)
    got = oracle.attn_bwd(q, k, v, g, scale, mask, lens)
    want = _torch_grads(q, k, v, g, scale, mask, lens)
    for a, b in zip(got, want):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


def test_single_key():
    """One key: P = 1, so dV = sum_i dO_i and the scores get no gradient."""
    q, k, v, g = _inputs(n_k=1)
    dq, dk, dv = oracle.attn_bwd(q, k, v, g, 0.5)
    assert np.all(dq == 0) and np.all(dk == 0)
    np.testing.assert_allclose(dv[:, :, 0, :], g.astype(np.float64).sum(axis=2), rtol=1e-14)


def test_constant_values_give_no_score_gradient():
    q, k, v, g = _inputs()
    v[...] = v[:, :, :1, :]
    dq, dk, _ = oracle.attn_bwd(q, k, v, g, 0.5)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13


def test_zero_queries_uniform_weights():
    """q = 0: every weight is 1/n_k, dV_j = mean of dO over queries' sum / n_k, dK = 0."""
    q, k, v, g = _inputs(n_k=4)
    q[...] = 0
    dq, dk, dv = oracle.attn_bwd(q, k, v, g, 0.5)
    assert np.abs(dk).max() < 1e-14
    want = g.astype(np.float64).sum(axis=2, keepdims=True) / 4
    np.testing.assert_allclose(dv, np.broadcast_to(want, dv.shape), rtol=1e-14)
    # dQ_i = scale * sum_j (dP_ij - mean_j dP_ij) k_j / n_k with dP_ij = dO_i . v_j
    dp = np.einsum("bhic,bhjc->bhij", g.astype(np.float64), v.astype(np.float64))
    ds = (dp - dp.mean(-1, keepdims=True)) / 4
    np.testing.assert_allclose(dq, 0.5 * np.einsum("bhij,bhjt->bhit", ds, k.astype(np.float64)),
                               rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("mask,lens", CASES)
def test_key_shift_invariance(mask, lens):
    """Adding one vector to every visible key leaves each row's softmax unchanged, so
    the key gradients of each row-set sum to zero (for causal: per key column set)."""
    q, k, v, g = _inputs(n_q=6, n_k=6)
    dq, dk, dv = oracle.attn_bwd(q, k, v, g, 0.5, mask, lens)
    if mask == oracle.MASK_CAUSAL:
        return  # each query sees a different key set; covered by the homogeneity pin
    np.testing.assert_allclose(dk.sum(axis=2), 0, atol=1e-12)


@pytest.mark.parametrize("mask,lens", CASES)
def test_homogeneity_of_scores(mask, lens):
    """Scores are bilinear in q and k: scaling q or k by a is the same change, so
    sum q.dQ = sum k.dK (a transposed operand or misplaced scale breaks it)."""
    q, k, v, g = _inputs(n_q=6, n_k=7)
    dq, dk, _ = oracle.attn_bwd(q, k, v, g, 0.7, mask, lens)
    a = (q.astype(np.float64) * dq).sum(axis=(2, 3))
    b = (k.astype(np.float64) * dk).sum(axis=(2, 3))
    np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-13)


def test_value_gradient_sums_to_output_gradient():
    q, k, v, g = _inputs()
    _, _, dv = oracle.attn_bwd(q, k, v, g, 0.5)
    np.testing.assert_allclose(dv.sum(axis=2), g.astype(np.float64).sum(axis=2), rtol=1e-12)


def test_value_gradient_is_weights_transposed_times_dout():
    """With V = I (n_k = d_v) the forward's output is the weight matrix P itself."""
    q, k, _, _ = _inputs(n_q=5, n_k=6, d_v=6)
    g = _grid((2, 2, 5, 6), 9)
    eye = np.broadcast_to(np.eye(6, dtype=np.float32), (2, 2, 6, 6)).copy()
    for mask, lens in CASES:
        p, _ = oracle.attn_fwd(q, k, eye, 0.5, mask, lens)
        _, _, dv = oracle.attn_bwd(q, k, eye, g, 0.5, mask, lens)
        np.testing.assert_allclose(dv, np.einsum("bhij,bhic->bhjc", p, g.astype(np.float64)),
                                   rtol=1e-13, atol=1e-15)


def test_masked_keys_get_no_gradient():
    q, k, v, g = _inputs(n_k=8)
    lens = np.array([3, 0], dtype=np.int32)
    dq, dk, dv = oracle.attn_bwd(q, k, v, g, 0.5, oracle.MASK_KEY_PADDING, lens)
    assert np.all(dk[0, :, 3:] == 0) and np.all(dv[0, :, 3:] == 0)
    assert np.all(dk[1] == 0) and np.all(dv[1] == 0) and np.all(dq[1] == 0)
    # padding values never matter
    k2, v2 = k.copy(), v.copy()
    k2[0, :, 3:] = 7.0
    v2[0, :, 3:] = -5.0
    again = oracle.attn_bwd(q, k2, v2, g, 0.5, oracle.MASK_KEY_PADDING, lens)
    np.testing.assert_array_equal(again[0], dq)
    np.testing.assert_array_equal(again[1][:, :, :3], dk[:, :, :3])


def test_causal_key_sees_only_later_queries():
    """Under the causal mask key j receives gradient only from queries i >= j."""
    q, k, v, g = _inputs(n_q=6, n_k=6)
    _, dk, dv = oracle.attn_bwd(q, k, v, g, 0.5, oracle.MASK_CAUSAL)
    g2 = g.copy()
    g2[:, :, :3] = _grid(g2[:, :, :3].shape, 99)   # change dO of queries 0..2
    _, dk2, dv2 = oracle.attn_bwd(q, k, v, g2, 0.5, oracle.MASK_CAUSAL)
    np.testing.assert_array_equal(dk[:, :, 3:], dk2[:, :, 3:])
    np.testing.assert_array_equal(dv[:, :, 3:], dv2[:, :, 3:])
    # the last key is seen by the last query only: dV_last = P_last,last dO_last
    o, _ = oracle.attn_fwd(q, k, np.broadcast_to(np.eye(6, dtype=np.float32), (2, 2, 6, 6)).copy(),
                           0.5, oracle.MASK_CAUSAL)
    np.testing.assert_allclose(dv[:, :, 5], o[:, :, 5, 5, None] * g[:, :, 5].astype(np.float64),
                               rtol=1e-13)


def test_linear_in_output_gradient():
    q, k, v, g = _inputs()
    g2 = _grid(g.shape, 42)
    a = oracle.attn_bwd(q, k, v, g, 0.5)
    b = oracle.attn_bwd(q, k, v, g2, 0.5)
    c = oracle.attn_bwd(q, k, v, g + g2, 0.5)
    for x, y, z in zip(a, b, c):
        np.testing.assert_allclose(x + y, z, rtol=1e-12, atol=1e-13)


def test_bad_arguments():
    q, k, v, g = _inputs()
    with pytest.raises(ValueError):
        oracle.attn_bwd(q, k, v, g[:, :, :2], 0.5)
    with pytest.raises(ValueError):
        oracle.attn_bwd(q, k, v, g, 0.5, oracle.MASK_KEY_PADDING, None)


# ---------------------------------------------------------------- restricted window

def _torch_band_grads(q, k, v, g, scale, left, right):
    Q, K, V = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    i = torch.arange(q.shape[2])[:, None]
    j = torch.arange(k.shape[2])[None, :]
    allowed = ((j >= i - left) & (j <= i + right))[None, None]
    any_row = allowed.any(-1, keepdim=True)
    s = scale * Q @ K.transpose(-1, -2)
    s = torch.where(allowed, s, torch.tensor(-math.inf, dtype=torch.float64))
    s = torch.where(any_row, s, torch.zeros((), dtype=torch.float64))
    p = torch.softmax(s, dim=-1) * any_row
    (p @ V * torch.tensor(g, dtype=torch.float64)).sum().backward()
    return Q.grad.numpy(), K.grad.numpy(), V.grad.numpy()


@pytest.mark.parametrize("left,right", [(2, 2), (4, 0), (0, 3), (1, 6), (0, 0)])
def test_band_matches_autograd(left, right):
    rng = np.random.default_rng(21)
    q = rng.standard_normal((2, 2, 11, 5)).astype(np.float32)
    k = rng.standard_normal((2, 2, 9, 5)).astype(np.float32)   # queries 9, 10 see few or no keys
    v = rng.standard_normal((2, 2, 9, 4)).astype(np.float32)
    g = rng.standard_normal((2, 2, 11, 4)).astype(np.float32)
    got = oracle.attn_bwd_band(q, k, v, g, 0.45, left, right)
    want = _torch_band_grads(q, k, v, g, 0.45, left, right)
    for a, b in zip(got, want):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


def test_band_finite_differences_of_the_band_forward():
    q, k, v, g = _inputs(n_q=6, n_k=7)
    left, right = 2, 1
    grads = oracle.attn_bwd_band(q, k, v, g, 0.5, left, right)
    rng = np.random.default_rng(8)
    for name, x, grad in zip(("q", "k", "v"), (q, k, v), grads):
        for _ in range(5):
            idx = tuple(int(rng.integers(0, n)) for n in x.shape)

            def loss(h):
                xs = {"q": q, "k": k, "v": v}
                y = x.copy()
                y[idx] += h
                xs[name] = y
                o, _ = oracle.attn_band(xs["q"], xs["k"], xs["v"], 0.5, left, right)
                return float((o * g.astype(np.float64)).sum())

            def central(h):
                return (loss(h) - loss(-h)) / (2 * h)

            h = 2.0 ** -9
            est = (4 * central(h / 2) - central(h)) / 3
            assert abs(est - grad[idx]) <= 1e-7 + 1e-6 * abs(grad[idx]), (name, idx)


def test_band_limits_are_the_unmasked_and_causal_backward():
    q, k, v, g = _inputs(n_q=6, n_k=6)
    a = oracle.attn_bwd_band(q, k, v, g, 0.5, 100, 100)
    b = oracle.attn_bwd(q, k, v, g, 0.5)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    a = oracle.attn_bwd_band(q, k, v, g, 0.5, 100, 0)
    b = oracle.attn_bwd(q, k, v, g, 0.5, oracle.MASK_CAUSAL)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_band_keys_outside_every_window_get_no_gradient():
    q, k, v, g = _inputs(n_q=5, n_k=12)
    dq, dk, dv = oracle.attn_bwd_band(q, k, v, g, 0.5, 1, 2)   # queries 0..4 reach keys <= 6
    assert np.all(dk[:, :, 7:] == 0) and np.all(dv[:, :, 7:] == 0)
    k2 = k.copy()
    k2[:, :, 7:] = 9.0
    again = oracle.attn_bwd_band(q, k2, v, g, 0.5, 1, 2)
    np.testing.assert_array_equal(again[0], dq)

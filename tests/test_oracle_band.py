"""Pins for the restricted (banded) self-attention oracle (oracle.attn_band).

Restricted self-attention is named on "Lire << Attention Is All You Need >>"
(section 4, Table 1: each output position attends to a neighbourhood of size
r around it, O(r.n.d) work, O(n/r) path length) and on the slide deck's
Table 1; the pages give no formula beyond that.  Reading: query i sees keys
i - left <= j <= i + right.  Pins tie it to the pinned full oracle and to
counts that a wrong window bound (off by one, swapped sides) breaks.
"""
import math

import numpy as np
import pytest

import oracle


def _qkv(B=2, H=2, n_q=37, n_k=41, d=8, seed=0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, n_q, d)).astype(np.float32)
    k = rng.standard_normal((B, H, n_k, d)).astype(np.float32)
    v = rng.standard_normal((B, H, n_k, d)).astype(np.float32)
    return q, k, v


def test_wide_window_is_no_mask():
    q, k, v = _qkv()
    o, l = oracle.attn_band(q, k, v, 0.3, 100, 100)
    o2, l2 = oracle.attn_fwd(q, k, v, 0.3, oracle.MASK_NONE)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(l, l2)


def test_no_right_side_is_causal():
    q, k, v = _qkv(n_q=41)
    o, l = oracle.attn_band(q, k, v, 0.3, 1000, 0)
    o2, l2 = oracle.attn_fwd(q, k, v, 0.3, oracle.MASK_CAUSAL)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(l, l2)


def test_zero_window_sees_itself_only():
    q, k, v = _qkv(n_q=45, n_k=41)
    o, l = oracle.attn_band(q, k, v, 0.3, 0, 0)
    np.testing.assert_allclose(o[:, :, :41], v.astype(np.float64), rtol=0, atol=1e-15)
    s_ii = 0.3 * np.einsum("bhid,bhid->bhi", q[:, :, :41].astype(np.float64), k.astype(np.float64))
    np.testing.assert_allclose(l[:, :, :41], s_ii, rtol=1e-14)
    # queries past the last key have an empty window
    assert np.all(o[:, :, 41:] == 0) and np.all(np.isneginf(l[:, :, 41:]))


@pytest.mark.parametrize("left,right", [(3, 3), (5, 0), (0, 4), (2, 7), (40, 1)])
def test_window_counts_with_equal_scores(left, right):
    """Identical keys: every visible key has the same score s, so LSE_i = s + ln(#window_i)
    and O_i is the mean of the visible values."""
    q, k, v = _qkv(n_q=30, n_k=26)
    k[...] = k[:, :, :1]
    o, l = oracle.attn_band(q, k, v, 0.5, left, right)
    s = 0.5 * np.einsum("bhid,bhd->bhi", q.astype(np.float64), k[:, :, 0].astype(np.float64))
    for i in range(30):
        lo, hi = max(0, i - left), min(25, i + right)
        if lo > hi:
            assert np.all(np.isneginf(l[:, :, i]))
            continue
        np.testing.assert_allclose(l[:, :, i], s[:, :, i] + math.log(hi - lo + 1), rtol=1e-13)
        np.testing.assert_allclose(o[:, :, i], v[:, :, lo:hi + 1].astype(np.float64).mean(axis=2),
                                   rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("left,right", [(4, 4), (9, 0), (0, 6), (13, 2)])
def test_each_row_is_the_full_oracle_on_its_window(left, right):
    """Row i equals the (pinned) unmasked oracle run on the keys and values of its window only."""
    q, k, v = _qkv(B=1, H=2, n_q=33, n_k=35)
    o, l = oracle.attn_band(q, k, v, 0.4, left, right)
    for i in range(33):
        lo, hi = max(0, i - left), min(34, i + right)
        if lo > hi:
            continue
        oi, li = oracle.attn_fwd(q[:, :, i:i + 1], k[:, :, lo:hi + 1], v[:, :, lo:hi + 1], 0.4)
        np.testing.assert_array_equal(o[:, :, i], oi[:, :, 0])
        np.testing.assert_array_equal(l[:, :, i], li[:, :, 0])


def test_numpy_explicit_band_mask():
    q, k, v = _qkv(n_q=50, n_k=47)
    left, right = 6, 3
    o, l = oracle.attn_band(q, k, v, 0.25, left, right)
    i = np.arange(50)[:, None]
    j = np.arange(47)[None, :]
    allowed = (j >= i - left) & (j <= i + right)
    s = 0.25 * np.einsum("bhid,bhjd->bhij", q.astype(np.float64), k.astype(np.float64))
    s = np.where(allowed, s, -np.inf)
    m = s.max(-1, keepdims=True)
    w = np.exp(s - m)
    np.testing.assert_allclose(o, (w @ v.astype(np.float64)) / w.sum(-1, keepdims=True),
                               rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l, (m[..., 0] + np.log(w.sum(-1))), rtol=1e-13)


def test_keys_outside_the_window_never_matter():
    q, k, v = _qkv(n_q=40, n_k=40)
    o, l = oracle.attn_band(q, k, v, 0.3, 3, 2)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, 30:] = 50.0    # far from rows 0..24
    v2[:, :, 30:] = np.nan
    o2, l2 = oracle.attn_band(q, k2, v2, 0.3, 3, 2)
    np.testing.assert_array_equal(o[:, :, :25], o2[:, :, :25])
    np.testing.assert_array_equal(l[:, :, :25], l2[:, :, :25])


def test_rows_entry_point_matches():
    q, k, v = _qkv()
    o, l = oracle.attn_band(q, k, v, 0.3, 5, 2)
    rows = np.array([0, 7, 36, 37, 80, 147], dtype=np.int64)
    orow, lrow = oracle.attn_band(q, k, v, 0.3, 5, 2, rows=rows)
    np.testing.assert_array_equal(orow, o.reshape(-1, o.shape[-1])[rows])
    np.testing.assert_array_equal(lrow, l.reshape(-1)[rows])


def test_bad_window():
    q, k, v = _qkv()
    with pytest.raises(ValueError):
        oracle.attn_band(q, k, v, 0.3, -1, 2)

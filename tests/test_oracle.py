"""Pins for the float64 CPU oracle (no GPU).

Each test ties the oracle to something other than itself: numbers printed on
the pages, closed forms, invariants the definition implies, or a NumPy float64
evaluation of the textbook formula.  Together they are chosen so that a
plausible slip anywhere in the oracle (a transposed operand, a missing
1/sqrt(d_k), an off-by-one in the causal or key-padding boundary, a dropped
max-subtraction, a wrong LSE base) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

from transformer_head_scaled_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NONE, CAUSAL, PAD = 0, 1, 2


def _printed_tol(s: str) -> float:
    """Half a unit in the last printed digit."""
    dec = len(s.split(".")[1]) if "." in s else 0
    return 0.5 * 10.0 ** (-dec) + 1e-12


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)


# ---------------------------------------------------------------- printed pins

def test_sentence_example_scores_and_weights(oracle_mod):
    """Worked example of section 3.2.1 on "Lire << Attention Is All You Need >>"
    (figure "L'attention dans une phrase"): q = [2.2, 0]
    against seven 2-D keys, scores divided by sqrt(2).  With V = I_7 the output
    row is the weight vector itself; with a single key the log-sum-exp is that
    key's scaled score."""
    ex = json.load(open(os.path.join(GOLDEN, "sentence_example.json")))
    q = np.array(ex["query"], dtype=np.float32).reshape(1, 1, 1, 2)
    keys = np.array([e["k"] for e in ex["keys"]], dtype=np.float32)
    n = len(keys)
    scale = 1.0 / math.sqrt(ex["d_k"])
    k = keys.reshape(1, 1, n, 2)
    v = np.eye(n, dtype=np.float32).reshape(1, 1, n, n)
    o, lse = oracle_mod.attn_fwd(q, k, v, scale, NONE)
    for j, e in enumerate(ex["keys"]):
        pct = 100.0 * o[0, 0, 0, j]
        assert abs(pct - float(e["weight_percent"])) <= _printed_tol(e["weight_percent"]), e
        # score of key j alone: lse over one key = its scaled score
        _, l1 = oracle_mod.attn_fwd(q, keys[j].reshape(1, 1, 1, 2),
                                    np.ones((1, 1, 1, 1), np.float32), scale, NONE)
        assert abs(l1[0, 0, 0] - float(e["score"])) <= _printed_tol(e["score"]), e
    # the most compatible key ("chat") dominates
    assert int(np.argmax(o[0, 0, 0])) == 1
    assert abs(o.sum() - 1.0) < 1e-12


def test_two_key_softmax_example(oracle_mod):
    """Section 3.2.1 on "Lire << Attention Is All You Need >>": scores (8, 0) give weight ~0.9997 and
    p(1-p) ~0.0003; scaled by 1/8 to (1, 0) they give 0.73/0.27 and p(1-p) ~0.20."""
    ex = json.load(open(os.path.join(GOLDEN, "two_key_softmax.json")))
    for case in ex["cases"]:
        s = case["scores"]
        # q = [1], keys = [[s0], [s1]], scale 1: the scores are s exactly.
        q = np.ones((1, 1, 1, 1), np.float32)
        k = np.array(s, np.float32).reshape(1, 1, 2, 1)
        v = np.eye(2, dtype=np.float32).reshape(1, 1, 2, 2)
        o, _ = oracle_mod.attn_fwd(q, k, v, 1.0, NONE)
        p = o[0, 0, 0]
        for got, want in zip(p, case["weights"]):
            if want is not None:
                assert abs(got - float(want)) <= _printed_tol(want)
        d = p[0] * (1 - p[0])
        assert abs(d - float(case["derivative"])) <= _printed_tol(case["derivative"])
    # and the scaled case is the unscaled one divided by sqrt(d_k)=8
    q = np.ones((1, 1, 1, 1), np.float32)
    k = np.array([8.0, 0.0], np.float32).reshape(1, 1, 2, 1)
    v = np.eye(2, dtype=np.float32).reshape(1, 1, 2, 2)
    o8, _ = oracle_mod.attn_fwd(q, k, v, 1.0 / 8.0, NONE)
    assert abs(o8[0, 0, 0, 0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-12


def test_score_variance_footnote(oracle_mod):
    """Section 3.2.1 footnote: for independent unit-variance q, k the dot
    product has mean 0 and variance d_k; divided by sqrt(d_k) the variance is 1.
    With one key per query the log-sum-exp equals the scaled score."""
    d, n = 64, 100_000
    q = _rand((n, 1, 1, d), 11)
    k = _rand((n, 1, 1, d), 12)
    v = np.zeros((n, 1, 1, 1), np.float32)
    _, raw = oracle_mod.attn_fwd(q, k, v, 1.0, NONE)
    _, scaled = oracle_mod.attn_fwd(q, k, v, 1.0 / math.sqrt(d), NONE)
    raw, scaled = raw.ravel(), scaled.ravel()
    # sampling error of a variance estimate over 1e5 draws is ~0.6%
    assert abs(raw.var() / d - 1.0) < 0.05
    assert abs(scaled.var() - 1.0) < 0.05
    assert abs(raw.mean()) < 0.1
    np.testing.assert_allclose(scaled * math.sqrt(d), raw, rtol=1e-12, atol=1e-9)


def test_ten_token_shapes(oracle_mod):
    """Section 3.2.2 on "Lire << Attention Is All You Need >>": 10 tokens, 8 heads of 64 -> each head gives a
    10x64 output (from 10x10 weights)."""
    q, k, v = (_rand((1, 8, 10, 64), s) for s in (1, 2, 3))
    o, lse = oracle_mod.attn_fwd(q, k, v, 0.125, NONE)
    assert o.shape == (1, 8, 10, 64) and lse.shape == (1, 8, 10)


# ---------------------------------------------------------------- closed forms

def test_two_keys_closed_form(oracle_mod):
    """Two keys: the weight of key 0 is the logistic function of the score
    difference, and lse = log(e^s0 + e^s1)."""
    rng = np.random.default_rng(5)
    for _ in range(20):
        d = int(rng.integers(1, 9))
        q = rng.standard_normal((1, 1, 1, d)).astype(np.float32)
        k = rng.standard_normal((1, 1, 2, d)).astype(np.float32)
        v = rng.standard_normal((1, 1, 2, 3)).astype(np.float32)
        sc = float(rng.uniform(0.1, 2.0))
        o, lse = oracle_mod.attn_fwd(q, k, v, sc, NONE)
        s = [sc * float(np.dot(q[0, 0, 0].astype(np.float64), k[0, 0, j].astype(np.float64)))
             for j in range(2)]
        w0 = 1.0 / (1.0 + math.exp(s[1] - s[0]))
        want = w0 * v[0, 0, 0].astype(np.float64) + (1 - w0) * v[0, 0, 1].astype(np.float64)
        np.testing.assert_allclose(o[0, 0, 0], want, rtol=1e-12, atol=1e-12)
        assert abs(lse[0, 0, 0] - math.log(math.exp(s[0]) + math.exp(s[1]))) < 1e-12


def test_equal_scores_give_mean_of_values(oracle_mod):
    """Identical keys give uniform weights: unmasked O = mean of all V rows,
    causal row i = mean of V[0..i] (i inclusive), key padding = mean of the
    first L rows; lse = s + ln(number of visible keys)."""
    n, d = 9, 4
    q = _rand((2, 1, n, d), 21)
    k = np.broadcast_to(_rand((1, 1, 1, d), 22), (2, 1, n, d)).copy()
    v = _rand((2, 1, n, 5), 23)
    sc = 0.5
    s = sc * (q.astype(np.float64) @ k[0, 0, 0].astype(np.float64))  # [2,1,n]
    o, lse = oracle_mod.attn_fwd(q, k, v, sc, NONE)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True, dtype=np.float64), o.shape), atol=1e-12)
    np.testing.assert_allclose(lse, s + math.log(n), atol=1e-12)
    o, lse = oracle_mod.attn_fwd(q, k, v, sc, CAUSAL)
    for i in range(n):
        np.testing.assert_allclose(o[:, :, i], v[:, :, : i + 1].astype(np.float64).mean(axis=2), atol=1e-12)
        np.testing.assert_allclose(lse[:, :, i], s[:, :, i] + math.log(i + 1), atol=1e-12)
    lens = np.array([3, 7], np.int32)
    o, lse = oracle_mod.attn_fwd(q, k, v, sc, PAD, lens)
    for b in range(2):
        np.testing.assert_allclose(o[b, 0], np.broadcast_to(v[b, 0, : lens[b]].astype(np.float64).mean(axis=0), (n, 5)), atol=1e-12)
        np.testing.assert_allclose(lse[b, 0], s[b, 0] + math.log(lens[b]), atol=1e-12)


# ---------------------------------------------------------------- invariants

def test_rows_sum_to_one(oracle_mod):
    """Each row is its own softmax summing to 100% (figure of section 3.2.1 on
    "Lire << Attention Is All You Need >>"; the comment of the PyTorch listing
    on "32 Transformer"): V = 1 gives O = 1 under every mask."""
    q, k = _rand((2, 3, 17, 8), 31), _rand((2, 3, 19, 8), 32)
    v = np.ones((2, 3, 19, 1), np.float32)
    for mask, lens in ((NONE, None), (CAUSAL, None), (PAD, np.array([5, 19], np.int32))):
        o, _ = oracle_mod.attn_fwd(q, k, v, 0.3, mask, lens)
        np.testing.assert_allclose(o, 1.0, atol=1e-13)


def test_constant_values(oracle_mod):
    """A convex combination of identical rows is that row."""
    q, k = _rand((1, 2, 11, 8), 41), _rand((1, 2, 13, 8), 42)
    row = _rand((1, 1, 1, 6), 43)
    v = np.broadcast_to(row, (1, 2, 13, 6)).copy()
    o, _ = oracle_mod.attn_fwd(q, k, v, 0.35, NONE)
    np.testing.assert_allclose(o, np.broadcast_to(row.astype(np.float64), o.shape), atol=1e-12)


def test_causal_row_zero_is_first_value(oracle_mod):
    """Causal: position 0 sees only itself, so O[0] = V[0] and lse = s_00."""
    q, k, v = _rand((2, 2, 7, 8), 51), _rand((2, 2, 7, 8), 52), _rand((2, 2, 7, 8), 53)
    o, lse = oracle_mod.attn_fwd(q, k, v, 0.125, CAUSAL)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0].astype(np.float64), atol=1e-15)
    s00 = 0.125 * np.einsum("bhd,bhd->bh", q[:, :, 0].astype(np.float64), k[:, :, 0].astype(np.float64))
    np.testing.assert_allclose(lse[:, :, 0], s00, atol=1e-13)


def test_causal_equals_prefix_key_padding(oracle_mod):
    """Causal row i equals attention of that row over the first i+1 keys."""
    n = 12
    q, k, v = _rand((1, 1, n, 8), 61), _rand((1, 1, n, 8), 62), _rand((1, 1, n, 4), 63)
    oc, lc = oracle_mod.attn_fwd(q, k, v, 0.2, CAUSAL)
    for i in range(n):
        op, lp = oracle_mod.attn_fwd(q[:, :, i : i + 1], k, v, 0.2, PAD, np.array([i + 1], np.int32))
        np.testing.assert_allclose(oc[0, 0, i], op[0, 0, 0], atol=1e-14)
        assert abs(lc[0, 0, i] - lp[0, 0, 0]) < 1e-13


def test_one_hot_dominant_key(oracle_mod):
    """A key far more compatible than the rest takes essentially all the
    weight (the saturation discussed in section 3.2.1): O ~= its value."""
    d, n = 16, 10
    q = np.zeros((1, 1, 1, d), np.float32); q[..., 0] = 1.0
    k = _rand((1, 1, n, d), 71) * 0.1
    k[0, 0, 6, 0] = 100.0
    v = _rand((1, 1, n, 3), 72)
    o, _ = oracle_mod.attn_fwd(q, k, v, 1.0, NONE)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 6], atol=1e-30 + 1e-12)


def test_key_padding_special_cases(oracle_mod):
    """key_len = n_k is no mask; key_len = 1 gives O = V[0]; key_len = 0
    leaves no visible key (O = 0, lse = -inf); keys past the length are never
    read (changing them changes nothing)."""
    B, H, n, d = 4, 2, 10, 8
    q, k, v = _rand((B, H, 6, d), 81), _rand((B, H, n, d), 82), _rand((B, H, n, d), 83)
    o0, l0 = oracle_mod.attn_fwd(q, k, v, 0.125, NONE)
    lens = np.array([n, 1, 0, 4], np.int32)
    o, lse = oracle_mod.attn_fwd(q, k, v, 0.125, PAD, lens)
    np.testing.assert_array_equal(o[0], o0[0])
    np.testing.assert_array_equal(lse[0], l0[0])
    np.testing.assert_allclose(o[1], np.broadcast_to(v[1, :, :1].astype(np.float64), o[1].shape), atol=1e-15)
    assert np.all(o[2] == 0.0) and np.all(np.isneginf(lse[2]))
    k2, v2 = k.copy(), v.copy()
    k2[3, :, 4:] = 1e3
    v2[3, :, 4:] = -7.0
    o2, l2 = oracle_mod.attn_fwd(q, k2, v2, 0.125, PAD, lens)
    np.testing.assert_array_equal(o2, o)
    np.testing.assert_array_equal(l2, lse)


def test_key_permutation_invariance(oracle_mod):
    """Unmasked attention does not depend on the order of the key/value pairs
    (it is a weighted sum over a set)."""
    q, k, v = _rand((1, 2, 5, 8), 91), _rand((1, 2, 23, 8), 92), _rand((1, 2, 23, 8), 93)
    perm = np.random.default_rng(94).permutation(23)
    o, lse = oracle_mod.attn_fwd(q, k, v, 0.125, NONE)
    op, lp = oracle_mod.attn_fwd(q, k[:, :, perm], v[:, :, perm], 0.125, NONE)
    np.testing.assert_allclose(op, o, atol=1e-13)
    np.testing.assert_allclose(lp, lse, atol=1e-13)


def test_heads_are_independent(oracle_mod):
    """Multi-head attention runs h independent attentions (section 3.2.2)."""
    q, k, v = _rand((2, 4, 9, 8), 101), _rand((2, 4, 11, 8), 102), _rand((2, 4, 11, 8), 103)
    lens = np.array([7, 11], np.int32)
    for mask in (NONE, CAUSAL, PAD):
        o, lse = oracle_mod.attn_fwd(q, k, v, 0.125, mask, lens if mask == PAD else None)
        for b in range(2):
            for h in range(4):
                oh, lh = oracle_mod.attn_fwd(q[b:b+1, h:h+1], k[b:b+1, h:h+1], v[b:b+1, h:h+1], 0.125,
                                             mask, lens[b:b+1] if mask == PAD else None)
                np.testing.assert_array_equal(oh[0, 0], o[b, h])
                np.testing.assert_array_equal(lh[0, 0], lse[b, h])


def test_max_shift_invariance_large_scores(oracle_mod):
    """Adding a constant to every score of a row changes neither the weights
    nor O (softmax is shift-invariant); the oracle must not overflow when the
    scores are large (it subtracts the row max)."""
    q = np.ones((1, 1, 1, 2), np.float32)
    k = np.zeros((1, 1, 6, 2), np.float32)
    k[..., 0] = _rand((1, 1, 6), 111)
    v = _rand((1, 1, 6, 3), 112)
    o, lse = oracle_mod.attn_fwd(q, k, v, 1.0, NONE)
    k_shift = k.copy(); k_shift[..., 1] = 800.0   # every score +800; exp(800) overflows float64
    o2, lse2 = oracle_mod.attn_fwd(q, k_shift, v, 1.0, NONE)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    assert abs(lse2[0, 0, 0] - (lse[0, 0, 0] + 800.0)) < 1e-9


# ---------------------------------------------------------------- library cross-check

def _numpy_attention(q, k, v, scale, mask=None):
    """softmax(Q K^T * scale) V with NumPy float64 matmul and exp (the
    textbook formula that the PyTorch listing on "32 Transformer" evaluates),
    independent of the C loops."""
    q, k, v = (x.astype(np.float64) for x in (q, k, v))
    s = (q @ np.swapaxes(k, -1, -2)) * scale
    if mask is not None:
        s = np.where(mask, -np.inf, s)
    mx = s.max(axis=-1, keepdims=True)
    w = np.exp(s - mx)
    z = w.sum(axis=-1, keepdims=True)
    return (w / z) @ v, (mx + np.log(z))[..., 0]


@pytest.mark.parametrize("mask", [NONE, CAUSAL, PAD])
def test_matches_numpy_formula(oracle_mod, mask):
    B, H, nq, nk, d = 2, 3, 33, 33 if mask == CAUSAL else 40, 16
    q, k, v = _rand((B, H, nq, d), 121), _rand((B, H, nk, d), 122), _rand((B, H, nk, d), 123)
    lens = np.array([17, 40], np.int32)
    m = None
    if mask == CAUSAL:
        m = np.triu(np.ones((nq, nk), bool), 1)[None, None]
    elif mask == PAD:
        m = (np.arange(nk)[None, :] >= lens[:, None])[:, None, None, :]
    o_ref, l_ref = _numpy_attention(q, k, v, 0.25, m)
    o, lse = oracle_mod.attn_fwd(q, k, v, 0.25, mask, lens if mask == PAD else None)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, l_ref, rtol=1e-12, atol=1e-12)


def test_rows_entry_point_matches_full(oracle_mod):
    w = inputs.Workload("t", 2, 3, 50, 70, 16, PAD, "bf16")
    q, k, v, lens = inputs.make_inputs(w)
    o, lse = oracle_mod.attn_fwd(q, k, v, w.scale, PAD, lens)
    rows = np.array([0, 7, 49, 50, 123, 299])
    orow, lrow = oracle_mod.attn_rows(q, k, v, rows, w.scale, PAD, lens)
    np.testing.assert_array_equal(orow, o.reshape(-1, 16)[rows])
    np.testing.assert_array_equal(lrow, lse.reshape(-1)[rows])


def test_bad_arguments_rejected(oracle_mod):
    q = np.zeros((1, 1, 2, 4), np.float32)
    with pytest.raises(ValueError):
        oracle_mod.attn_fwd(q, q, q, 1.0, PAD)          # key padding without lengths
    with pytest.raises(ValueError):
        oracle_mod.attn_fwd(q, q, q, 1.0, 7)
    with pytest.raises(RuntimeError):
        oracle_mod.attn_rows(q, q, q, [5], 1.0, NONE)   # row out of range


def test_input_generator_recipe():
    """The shared generator draws N(0,1), rounds to bf16, and is seeded."""
    w = inputs.WORKLOADS["encdec"]
    small = inputs.Workload("s", 4, 2, 32, 48, 64, PAD, "bf16")
    q1, k1, v1, l1 = inputs.make_inputs(small)
    q2, _, _, l2 = inputs.make_inputs(small)
    assert (q1 == q2).all() and (l1 == l2).all()
    assert q1.dtype == inputs.torch.bfloat16 and l1.dtype == inputs.torch.int32
    assert int(l1.min()) >= 64 or int(l1.min()) >= min(64, small.n_k)
    assert int(l1.max()) <= small.n_k
    g = inputs.gaussian((200_000,), 0).double()
    assert abs(g.mean().item()) < 0.01 and abs(g.var().item() - 1) < 0.02
    lens = inputs.key_lengths(w.B, 64, 512)
    assert lens.min() >= 64 and lens.max() <= 512

"""The largest sizes the method allows, checked by properties that hold at
any size (the oracle cannot afford them): with every key zero the scores are
all 0, the softmax is uniform, O is the mean of the visible value rows and
LSE = ln(number of visible keys), exactly in the pages' definition.  The
sizes put more than 2^31 elements in one tensor (every offset must be 64-bit)
and one head's keys far beyond the benchmark's.  A many-heads case is checked
against the oracle on sampled heads."""
import math

import numpy as np
import pytest
import torch

import oracle
from transformer_head_scaled_gb300 import binding, inputs
from transformer_head_scaled_gb300.inputs import MASK_NONE

pytestmark = pytest.mark.gpu

BIG_N = (1 << 25) + 77   # keys of one head: K and V hold 2^31 + 4928 elements each
SPIKE = BIG_N - 5        # a key whose elements lie past element 2^31 of K and V


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from transformer_head_scaled_gb300.build import build
    build()
    oracle.build()
    return binding.load()


def _big_kv(seed):
    """K = 0 and V ~ N(0, 1) (bf16, seeded on the device) for one head of BIG_N keys."""
    gen = torch.Generator(device="cuda").manual_seed(seed)
    k = torch.zeros((1, 1, BIG_N, 64), dtype=torch.bfloat16, device="cuda")
    v = torch.randn((1, 1, BIG_N, 64), generator=gen, device="cuda", dtype=torch.float32)
    return k, v.to(torch.bfloat16)


def _mean_rows(v, n):
    """float64 mean of the first n rows of v, in chunks."""
    acc = torch.zeros(v.shape[1], dtype=torch.float64, device=v.device)
    for s in range(0, n, 1 << 22):
        acc += v[s: min(n, s + (1 << 22))].double().sum(dim=0)
    return acc / n


def _check_uniform_then_spike(call, k, v, n_visible, n_q):
    """All scores 0: every visible key counts once, so LSE = ln(n_visible)
    (exact: the running sum adds whole tiles of ones) and O is the mean of the
    visible value rows.  Zero-mean values keep the fp32 accumulator small; a
    uniform softmax over 2^25 keys of values with a large mean would grow it to
    ~10^7, where the tensor core's accumulation drops the low bits of each
    16-key partial sum.  Then one key past element 2^31 gets a score of 32 for
    every query: O must be that key's value row and LSE 32 (+ n e^-32)."""
    o, lse = call()
    binding.check()
    assert torch.allclose(lse, torch.full_like(lse, math.log(n_visible)), atol=1e-3, rtol=0)
    want = _mean_rows(v[0, 0], n_visible).float()
    assert (o[0, 0].float() - want).abs().max().item() <= 2e-3
    k[0, 0, SPIKE] = 4.0     # q = 1 everywhere: score 64 * 4 / 8 = 32
    o, lse = call()
    binding.check()
    spike = math.log(math.exp(32.0) + n_visible - 1)
    assert torch.allclose(lse, torch.full_like(lse, spike), atol=1e-3, rtol=0)
    row = v[0, 0, SPIKE].float().expand(n_q, 64)
    assert torch.allclose(o[0, 0].float(), row, atol=1e-3, rtol=8e-3)


def test_forward_one_head_beyond_2e31_elements():
    n_q = 130
    q = torch.ones((1, 1, n_q, 64), dtype=torch.bfloat16, device="cuda")
    k, v = _big_kv(11)
    _check_uniform_then_spike(lambda: binding.attn_fwd(q, k, v), k, v, BIG_N, n_q)


def test_decode_cache_beyond_2e31_elements():
    n_q, L = 2, BIG_N - 3
    q = torch.ones((1, 1, n_q, 64), dtype=torch.bfloat16, device="cuda")
    k, v = _big_kv(12)
    lens = torch.tensor([L], dtype=torch.int32, device="cuda")
    _check_uniform_then_spike(lambda: binding.attn_decode(q, k, v, lens), k, v, L, n_q)


def test_backward_long_keys_uniform_softmax():
    """K = 0: P = 1/n_k everywhere, so dV_j = mean_i dO_i ... summed over queries
    (sum_i P_ij dO_i), dQ = scale * dS K = 0, and dK = scale * dS^T Q with
    dS_ij = (dO_i . V_j - D_i) / n_k, D_i = mean_j dO_i . V_j, all in float64."""
    d, n_q, n_k = 64, 256, 1 << 18
    scale = 0.125
    q = inputs.gaussian((1, 1, n_q, d), 3).to(torch.bfloat16).cuda()
    k = torch.zeros((1, 1, n_k, d), dtype=torch.bfloat16, device="cuda")
    v = inputs.gaussian((1, 1, n_k, d), 4).to(torch.bfloat16).cuda()
    g = inputs.gaussian((1, 1, n_q, d), 5).to(torch.bfloat16).cuda()
    o, lse = binding.attn_fwd(q, k, v)
    dq, dk, dv = binding.attn_bwd(q, k, v, o, lse, g)
    binding.check()
    q64, v64, g64 = (t[0, 0].double() for t in (q, v, g))
    dv_want = g64.sum(dim=0) / n_k                       # every row the same
    dp = g64 @ v64.T                                     # [n_q, n_k]
    ds = (dp - dp.mean(dim=1, keepdim=True)) / n_k
    dk_want = scale * ds.T @ q64
    assert torch.count_nonzero(dq) == 0
    err_v = (dv[0, 0].double() - dv_want).abs().max().item()
    assert err_v <= 2e-2 * dv_want.abs().max().item() + 1e-6, err_v
    rel_k = ((dk[0, 0].double() - dk_want).norm() / dk_want.norm()).item()
    assert rel_k <= 5e-3, rel_k


def test_many_heads_against_oracle():
    """131072 (b, h) pairs of short sequences: the item index space, head and
    batch coordinates at their largest in the benchmark's range and beyond;
    every element compared, the oracle run over slices of 1024 batch entries."""
    B, h, n, d = 8192, 16, 40, 64
    w = inputs.Workload("heads", B, h, n, n, d, MASK_NONE, "bf16")
    q, k, v, _ = inputs.make_inputs(w, device="cuda")
    o, lse = binding.attn_fwd(q, k, v)
    binding.check()
    err_sum, err_max, count = 0.0, 0.0, 0
    for b0 in range(0, B, 1024):
        sub = [t[b0: b0 + 1024] for t in (q, k, v)]
        o_ref, l_ref = oracle.attn_fwd(*sub, 0.125, MASK_NONE, None)
        err = np.abs(o[b0: b0 + 1024].float().cpu().numpy() - o_ref)
        err_sum += float(err.sum())
        err_max = max(err_max, float(err.max()))
        count += err.size
        assert np.abs(lse[b0: b0 + 1024].cpu().numpy() - l_ref).max() <= 1e-3
    assert err_max <= 2e-2 and err_sum / count <= 2e-3

"""Host-side accounting of the workloads (no GPU): the FLOP and HBM-byte
counts the bench divides by, checked against closed forms written out here
from the definitions (Table 1 of "Attention Is All You Need": O(n^2 d) work
per head, O(r n d) for a window of r positions).
"""
import numpy as np

from transformer_head_scaled_gb300 import inputs
from transformer_head_scaled_gb300.inputs import WORKLOADS


def test_base_encoder_counts():
    w = WORKLOADS["base_enc"]
    # two products of 2 * n_q * n_k * d FLOPs per head
    assert inputs.flops(w) == 4 * 64 * 8 * 512 * 512 * 64
    # Q, K, V read and O written once (bf16), LSE written once (float32)
    assert inputs.hbm_bytes(w) == 4 * 64 * 8 * 512 * 64 * 2 + 64 * 8 * 512 * 4


def test_causal_halves_the_nominal_count_and_counts_the_triangle():
    w = WORKLOADS["base_dec"]
    assert inputs.flops(w) == 0.5 * inputs.flops(WORKLOADS["base_enc"])
    n = 512
    assert inputs.algorithmic_flops(w) == 4 * 64 * 8 * (n * (n + 1) // 2) * 64


def test_key_padding_counts_the_visible_keys():
    w = WORKLOADS["encdec"]
    lens = np.array([0, 1, 511, 512, 600] + [64] * 59)
    want = 4 * w.h * w.n_q * 64 * (0 + 1 + 511 + 512 + 512 + 64 * 59)
    assert inputs.algorithmic_flops(w, lens) == want


def test_window_counts_the_band():
    w = WORKLOADS["big_window"]
    n, r = 4096, 256
    # row i sees keys max(0, i - r) .. min(n - 1, i + r)
    pairs = sum(min(n - 1, i + r) - max(0, i - r) + 1 for i in range(n))
    assert inputs.flops(w) == 4 * w.B * w.h * pairs * 64


def test_decode_reads_only_the_filled_cache():
    w = WORKLOADS["decode_long"]
    lens = np.array([4096, 2048, 0] + [3000] * 29)
    kv = 2 * w.h * int(lens.sum()) * 64 * 2
    qo = 2 * w.B * w.h * 1 * 64 * 2
    assert inputs.hbm_bytes(w, lens) == kv + qo + 4 * w.B * w.h


def test_decode_window_reads_only_the_window():
    w = WORKLOADS["decode_long_window"]
    assert inputs.decode_window(w) == 1023
    assert inputs.decode_window(WORKLOADS["decode_long"]) is None
    lens = np.array([4096, 1024, 1025, 100, 0] + [2500] * 27)
    seen = np.minimum(lens, 1024)
    assert list(inputs.seen_keys(w, lens)) == list(seen)
    kv = 2 * w.h * int(seen.sum()) * 64 * 2
    assert inputs.hbm_bytes(w, lens) == kv + 2 * w.B * w.h * 64 * 2 + 4 * w.B * w.h
    assert inputs.algorithmic_flops(w, lens) == 4 * w.h * 1 * int(seen.sum()) * 64
    # the nominal count takes window + 1 keys per query
    assert inputs.flops(w) == 4 * w.B * w.h * 1 * 1024 * 64


def test_backward_counts_two_and_a_half_forwards():
    assert inputs.flops(WORKLOADS["base_enc_bwd"]) == 2.5 * inputs.flops(WORKLOADS["base_enc"])

"""Seeded synthetic inputs for multi-head scaled dot-product attention.

This module is shared by the tests, the benchmark and the smoke check, and by
both sides of every parity comparison (the CUDA path and the CPU oracle).  It
holds no step of the attention arithmetic: it only draws numbers and rounds
them to the storage type.

Recipe (the pages' own data, WMT14 batches of about 25K source and 25K target
tokens bucketed by length, section 5.1 of "Attention Is All You Need", are not
available here; these tensors stand in for them):

* Q, K, V entries are i.i.d. N(0, 1), drawn as float32 with NumPy's PCG64
  generator seeded 0 (Q), 1 (K), 2 (V), then rounded to bfloat16 with
  round-to-nearest-even (the float32 workload keeps the float32 draws).
  Unit-variance q and k are the premise of the scaling argument in section
  3.2.1 (footnote: q.k then has mean 0 and variance d_k).
* Per-sequence key lengths for encoder-decoder attention are integers uniform
  on [64, n_k] inclusive, PCG64 seeded 3 (decoding workloads: the filled part
  of each key/value cache, uniform on [lens_lo, n_k]).
* For the backward, the output gradient dO is i.i.d. N(0, 1), PCG64 seeded 4,
  rounded to bfloat16 (O and LSE come from the forward on the same inputs).
* Layout is [B, h, n, d] contiguous (heads split as (h, seq, d)).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_KEY_PADDING = 2
MASK_BAND = 3  # restricted self-attention: query i sees keys i - win_left .. i + win_right

SEED_Q, SEED_K, SEED_V, SEED_LENS, SEED_DOUT = 0, 1, 2, 3, 4


@dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, mask and storage type."""

    name: str
    B: int
    h: int
    n_q: int
    n_k: int
    d: int
    mask: int
    dtype: str  # "bf16" or "f32"
    lens_lo: int = 64
    kind: str = "fwd"  # "fwd": fused forward; "decode": few queries against a cache;
    #                    "bwd": gradients of the forward
    win_left: int = 0   # MASK_BAND; for kind "decode", > 0: attn_decode_window's window
    win_right: int = 0
    note: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        """1/sqrt(d_k), the scaling of eq. (1)."""
        return 1.0 / math.sqrt(self.d)


# The workloads: the base model (d_model=512, h=8, d_k=d_v=64) and the big
# model (d_model=1024, h=16, d_k=d_v=64) of "Attention Is All You Need",
# Table 3, used the three ways section 3.2.3 lists.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 8, 64, 64, 64, MASK_NONE, "f32",
                     note="tiny encoder self-attention, float32"),
    "base_enc": Workload("base_enc", 64, 8, 512, 512, 64, MASK_NONE, "bf16",
                         note="base encoder self-attention"),
    "base_dec": Workload("base_dec", 64, 8, 512, 512, 64, MASK_CAUSAL, "bf16",
                         note="base decoder masked self-attention"),
    "encdec": Workload("encdec", 64, 8, 384, 512, 64, MASK_KEY_PADDING, "bf16",
                       note="base encoder-decoder attention, key padding"),
    "big": Workload("big", 8, 16, 4096, 4096, 64, MASK_NONE, "bf16",
                    note="big model, long sequence, unmasked"),
    "big_causal": Workload("big_causal", 8, 16, 4096, 4096, 64, MASK_CAUSAL,
                           "bf16", note="big model, long sequence, causal"),
    # Decoding steps (section 6.1 on "Lire << Attention Is All You Need >>":
    # beam search of width 4): one new query per hypothesis against its
    # key/value cache; n_k is the cache capacity, the key lengths the filled
    # part.
    "decode_beam": Workload("decode_beam", 256, 8, 1, 512, 64, MASK_KEY_PADDING, "bf16",
                            lens_lo=64, kind="decode",
                            note="base model, 64 sentences x beam 4, cache up to 512"),
    "decode_long": Workload("decode_long", 32, 16, 1, 4096, 64, MASK_KEY_PADDING, "bf16",
                            lens_lo=2048, kind="decode",
                            note="big model, 8 sentences x beam 4, cache up to 4096"),
    # The decoding step of the base model split into other head counts
    # ("Attention Is All You Need", Table 3, rows (A)): the same cache bytes.
    "decode_long_window": Workload("decode_long_window", 32, 16, 1, 4096, 64, MASK_KEY_PADDING,
                                   "bf16", lens_lo=2048, kind="decode", win_left=1023,
                                   note="decode_long, restricted to the newest 1024 positions"),
    "decode_beam_h4_d128": Workload("decode_beam_h4_d128", 256, 4, 1, 512, 128, MASK_KEY_PADDING,
                                    "bf16", kind="decode",
                                    note="decode_beam with 4 heads of 128"),
    "decode_beam_h16_d32": Workload("decode_beam_h16_d32", 256, 16, 1, 512, 32, MASK_KEY_PADDING,
                                    "bf16", kind="decode",
                                    note="decode_beam with 16 heads of 32"),
    # Other splits of the base model's d_model = 512 into heads ("Attention
    # Is All You Need", Table 3, rows (A)): h x d_k = 4 x 128, 16 x 32, 32 x 16.
    "base_h4_d128": Workload("base_h4_d128", 64, 4, 512, 512, 128, MASK_NONE, "bf16",
                             note="base encoder self-attention, 4 heads of 128"),
    "base_h16_d32": Workload("base_h16_d32", 64, 16, 512, 512, 32, MASK_NONE, "bf16",
                             note="base encoder self-attention, 16 heads of 32"),
    "base_h32_d16": Workload("base_h32_d16", 64, 32, 512, 512, 16, MASK_NONE, "bf16",
                             note="base encoder self-attention, 32 heads of 16"),
    # Restricted self-attention for long sequences ("Lire << Attention Is All
    # You Need >>", section 4 and Table 1): a window of 2*256 + 1 positions
    # centred on each output position of the big model's long sequences.
    "big_window": Workload("big_window", 8, 16, 4096, 4096, 64, MASK_BAND, "bf16",
                           win_left=256, win_right=256,
                           note="big model, long sequence, window of 513 centred positions"),
    # Training needs the gradient of every attention layer (section 5 of
    # "Attention Is All You Need"): the backward on the same problems.
    "base_enc_bwd": Workload("base_enc_bwd", 64, 8, 512, 512, 64, MASK_NONE, "bf16", kind="bwd",
                             note="backward of base encoder self-attention"),
    "base_dec_bwd": Workload("base_dec_bwd", 64, 8, 512, 512, 64, MASK_CAUSAL, "bf16", kind="bwd",
                             note="backward of base decoder masked self-attention"),
    "encdec_bwd": Workload("encdec_bwd", 64, 8, 384, 512, 64, MASK_KEY_PADDING, "bf16", kind="bwd",
                           note="backward of base encoder-decoder attention"),
    "big_bwd": Workload("big_bwd", 8, 16, 4096, 4096, 64, MASK_NONE, "bf16", kind="bwd",
                        note="backward, big model, long sequence"),
    "big_causal_bwd": Workload("big_causal_bwd", 8, 16, 4096, 4096, 64, MASK_CAUSAL, "bf16",
                               kind="bwd", note="backward, big model, long sequence, causal"),
    "big_window_bwd": Workload("big_window_bwd", 8, 16, 4096, 4096, 64, MASK_BAND, "bf16",
                               win_left=256, win_right=256, kind="bwd",
                               note="backward of restricted self-attention, window of 513"),
    "base_h16_d32_bwd": Workload("base_h16_d32_bwd", 64, 16, 512, 512, 32, MASK_NONE, "bf16",
                                 kind="bwd", note="backward, base encoder, 16 heads of 32"),
    "base_h32_d16_bwd": Workload("base_h32_d16_bwd", 64, 32, 512, 512, 16, MASK_NONE, "bf16",
                                 kind="bwd", note="backward, base encoder, 32 heads of 16"),
}


def gaussian(shape, seed: int) -> torch.Tensor:
    """i.i.d. N(0,1) float32 on the CPU from PCG64(seed)."""
    rng = np.random.default_rng(seed)
    return torch.from_numpy(rng.standard_normal(size=tuple(shape), dtype=np.float32))


def key_lengths(B: int, lo: int, hi: int, seed: int = SEED_LENS) -> torch.Tensor:
    """B integers uniform on [lo, hi] inclusive, int32 on the CPU."""
    rng = np.random.default_rng(seed)
    return torch.from_numpy(rng.integers(lo, hi, size=B, endpoint=True).astype(np.int32))


def make_inputs(w: Workload, device="cpu", seeds=(SEED_Q, SEED_K, SEED_V, SEED_LENS)):
    """(q, k, v, key_lens) for a workload.

    q, k, v are bfloat16 (or float32) tensors on ``device``; key_lens is an
    int32 tensor on ``device`` for key padding, else None.
    """
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    q = gaussian((w.B, w.h, w.n_q, w.d), seeds[0]).to(dt)
    k = gaussian((w.B, w.h, w.n_k, w.d), seeds[1]).to(dt)
    v = gaussian((w.B, w.h, w.n_k, w.d), seeds[2]).to(dt)
    lens = None
    if w.mask == MASK_KEY_PADDING:
        lens = key_lengths(w.B, min(w.lens_lo, w.n_k), w.n_k, seeds[3])
    if device != "cpu":
        q, k, v = q.to(device), k.to(device), v.to(device)
        lens = None if lens is None else lens.to(device)
    return q, k, v, lens


def make_dout(w: Workload, device="cpu", seed: int = SEED_DOUT) -> torch.Tensor:
    """The output gradient dO [B, h, n_q, d] for a backward workload."""
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    g = gaussian((w.B, w.h, w.n_q, w.d), seed).to(dt)
    return g if device == "cpu" else g.to(device)


def products(w: Workload) -> float:
    """Tile products per pass, in units of one n_q x n_k x d contraction:
    2 for the forward (Q K^T and P V), 5 for the backward (Q K^T recomputed,
    dO V^T, P^T dO, dS^T Q, dS K)."""
    return 5.0 if w.kind == "bwd" else 2.0


def decode_window(w: Workload):
    """The window of a restricted decoding step (keys len-1-window .. len-1),
    or None for attention over the whole cache."""
    return w.win_left if w.kind == "decode" and w.win_left > 0 else None


def seen_keys(w: Workload, lens):
    """Keys each batch entry's queries see in a decoding step: the filled
    cache, or its newest window + 1 positions."""
    seen = np.minimum(np.asarray(lens), w.n_k)
    win = decode_window(w)
    return seen if win is None else np.minimum(seen, win + 1)


def flops(w: Workload, key_lens=None) -> float:
    """Nominal FLOPs of one pass: 2*n_q*n_k*d per contraction and head
    (forward 4*B*h*n_q*n_k*d, backward 2.5 times that), halved for the causal
    mask; a restricted decoding step counts window + 1 keys."""
    n_k = w.n_k if decode_window(w) is None else min(w.n_k, decode_window(w) + 1)
    f = 2.0 * products(w) * w.B * w.h * w.n_q * n_k * w.d
    if w.mask == MASK_CAUSAL:
        f *= 0.5
    if w.mask == MASK_BAND:
        # the work the window leaves: O(r n d) instead of O(n^2 d)
        f = 2.0 * products(w) * w.B * w.h * band_pairs(w.n_q, w.n_k, w.win_left,
                                                       w.win_right) * w.d
    return f


def band_pairs(n_q: int, n_k: int, left: int, right: int) -> float:
    """Number of (query, key) pairs inside the window i-left <= j <= i+right."""
    i = np.arange(n_q, dtype=np.int64)
    cnt = np.minimum(n_k - 1, i + right) - np.maximum(0, i - left) + 1
    return float(np.maximum(cnt, 0).sum())


def algorithmic_flops(w: Workload, key_lens=None) -> float:
    """FLOPs over the connections the mask allows: causal counts the exact
    triangle, key padding counts sum_b L_b keys per query, the band counts
    the pairs inside each query's window."""
    if w.mask == MASK_BAND:
        return 2.0 * products(w) * w.B * w.h * band_pairs(w.n_q, w.n_k, w.win_left,
                                                          w.win_right) * w.d
    if w.mask == MASK_CAUSAL:
        n = min(w.n_q, w.n_k)
        pairs = n * (n + 1) / 2 + max(0, w.n_q - n) * w.n_k
        return 2.0 * products(w) * w.B * w.h * pairs * w.d
    if w.mask == MASK_KEY_PADDING:
        lens = np.asarray(key_lens.cpu() if hasattr(key_lens, "cpu") else key_lens)
        return 2.0 * products(w) * w.h * w.n_q * float(seen_keys(w, lens).sum()) * w.d
    return flops(w)


def hbm_bytes(w: Workload, key_lens=None) -> float:
    """Compulsory HBM bytes of one forward pass: Q, K, V read once, O written
    once, LSE (float32) written once; the n_q x n_k scores never leave the chip.
    For a decoding step only the filled part of the caches is read (of a
    restricted step, only its window).  The
    backward reads Q, K, V, O, dO and LSE and writes dQ, dK, dV."""
    es = 2 if w.dtype == "bf16" else 4
    if w.kind == "bwd":
        return float(4 * w.B * w.h * w.n_q * w.d * es + 4 * w.B * w.h * w.n_k * w.d * es
                     + 4 * w.B * w.h * w.n_q)
    qo = 2 * w.B * w.h * w.n_q * w.d * es
    if w.kind == "decode" and key_lens is not None:
        lens = np.asarray(key_lens.cpu() if hasattr(key_lens, "cpu") else key_lens)
        kv = 2 * w.h * float(seen_keys(w, lens).sum()) * w.d * es
    else:
        kv = 2 * w.B * w.h * w.n_k * w.d * es
    return float(qo + kv + 4 * w.B * w.h * w.n_q)

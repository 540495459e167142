"""Seeded synthetic inputs for the attention forward pass.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's
tests. It holds no attention arithmetic: it only draws random numbers, rounds
them to bf16 and (for the base encoder workload) applies the bias-free Q/K/V
projections that produce the heads, which sit *before* the attention path.

Shapes follow the head-split layout of "Transformer 详解" §4.2 (multi-head:
``view(batch, seq, h, d_k).transpose(1, 2)`` -> ``[B, H, L, d_k]``) and of
"从 RNN 到 Transformer（二）" §4.9 (``Q: (B, h, L_q, d_k)``, ``K: (B, h, L_k,
d_k)``, ``V: (B, h, L_k, d_v)``). Key padding is a valid prefix per batch
entry, which is what tail padding to the batch maximum produces
("Transformer 详解" §3.3-§3.4).

All draws use ``torch.Generator('cpu').manual_seed(seed)`` in a fixed order, in
fp32, then round to bf16 (round-to-nearest-even, torch's ``.to``).
"""

from __future__ import annotations

import dataclasses
import math

import torch

MASK_NONE = "none"
MASK_CAUSAL = "causal"
MASK_KEY_PADDING = "key_padding"
MASK_CAUSAL_KEY_PADDING = "causal_key_padding"
MASK_CAUSAL_CACHE = "causal_cache"     # causal, the queries being the last n of each entry's key_lengths[b]
MASK_KINDS = (MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING, MASK_CAUSAL_KEY_PADDING, MASK_CAUSAL_CACHE)
LENGTH_MASKS = (MASK_KEY_PADDING, MASK_CAUSAL_KEY_PADDING, MASK_CAUSAL_CACHE)
CAUSAL_MASKS = (MASK_CAUSAL, MASK_CAUSAL_KEY_PADDING, MASK_CAUSAL_CACHE)


def nominal_pairs(n: int, m: int, mask: str) -> float:
    """(query, key) pairs a FLOP count charges: n*m, or under a causal mask the
    visible part with the masked triangle counted as half its square (n*m - n*n/2
    for n <= m, m*m/2 for n > m), the usual convention that charges a square
    causal mask n*m/2."""
    if mask not in CAUSAL_MASKS:
        return float(n) * m
    if n <= m:
        return float(n) * m - float(n) * n / 2
    return float(m) * m / 2


@dataclasses.dataclass(frozen=True)
class Workload:
    """One seeded attention workload: shapes, mask, value recipe and seed."""

    name: str
    B: int
    H: int
    n: int
    m: int
    d_k: int
    d_v: int
    mask: str
    seed: int
    recipe: str = "normal"          # "normal" | "projection"
    value_scale: float = 1.0        # multiplies the N(0,1) draws (normal recipe)
    len_lo: int = 0                 # key-padding valid length range, inclusive
    len_hi: int = 0
    d_model: int = 0                # projection recipe only
    path: str = "fwd"               # "fwd": attn_fwd; "decode": the few-row attn_decode
    alibi: bool = False             # linear distance bias with the slopes of alibi_slopes(H)

    def flops(self) -> float:
        """Nominal forward FLOPs: 2*d_k (scores) + 2*d_v (weighted sum) per visible
        (query, key) pair (``nominal_pairs``; half of n*m for a square causal mask)."""
        return 2.0 * self.B * self.H * (self.d_k + self.d_v) * nominal_pairs(self.n, self.m, self.mask)

    def decode_bytes(self, key_lengths=None) -> float:
        """Algorithmic HBM bytes of a few-row pass: the visible K and V rows once (per
        batch entry min(length, m) rows under the key-padding masks), Q, O and LSE."""
        if key_lengths is not None and self.mask in LENGTH_MASKS:
            rows = float(key_lengths.clamp(0, self.m).sum()) * self.H
        else:
            rows = float(self.B) * self.H * self.m
        bh = self.B * self.H
        return rows * 2 * (self.d_k + self.d_v) + bh * self.n * (2 * self.d_k + 2 * self.d_v + 4)

    def io_bytes(self) -> int:
        """Algorithmic HBM bytes: Q, K, V read once (bf16); O (bf16) and LSE (fp32) written once."""
        bh = self.B * self.H
        return bh * (2 * self.n * self.d_k + 2 * self.m * self.d_k + 2 * self.m * self.d_v
                     + 2 * self.n * self.d_v + 4 * self.n)


# The five seeded workloads: tiny encoder self-attention; base encoder
# self-attention (d_model 512, h 8) with key padding; big decoder causal
# self-attention (d_model 1024, h 16); decoder->encoder cross-attention with
# encoder key padding; long-context causal self-attention at d 128.
WORKLOADS = {
    "tiny_encoder": Workload("tiny_encoder", 1, 8, 32, 32, 64, 64, MASK_NONE, seed=0),
    "base_encoder_keypad": Workload("base_encoder_keypad", 32, 8, 512, 512, 64, 64,
                                    MASK_KEY_PADDING, seed=1, recipe="projection",
                                    len_lo=256, len_hi=512, d_model=512),
    "big_decoder_causal": Workload("big_decoder_causal", 16, 16, 1024, 1024, 64, 64,
                                   MASK_CAUSAL, seed=2),
    "cross_keypad": Workload("cross_keypad", 32, 16, 256, 1024, 64, 64, MASK_KEY_PADDING,
                             seed=3, len_lo=512, len_hi=1024),
    "long_causal": Workload("long_causal", 4, 16, 8192, 8192, 128, 128, MASK_CAUSAL, seed=4,
                            value_scale=0.5),
}
WORKLOAD_ORDER = ["tiny_encoder", "base_encoder_keypad", "big_decoder_causal",
                  "cross_keypad", "long_causal"]

# Mask and shape variants at the sizes of the workloads above: the decoder target
# mask (causal and key padding, "Transformer 详解" §5.3) at big-decoder sizes with
# key lengths in [512, 1024]; 1024 new query rows against 8192 keys under the
# causal mask (bottom-right) at d 128; value heads twice as wide as the key heads.
WORKLOADS.update({
    "decoder_target_mask": Workload("decoder_target_mask", 16, 16, 1024, 1024, 64, 64,
                                    MASK_CAUSAL_KEY_PADDING, seed=5, len_lo=512, len_hi=1024),
    "prefill_continuation": Workload("prefill_continuation", 4, 16, 1024, 8192, 128, 128,
                                     MASK_CAUSAL, seed=6, value_scale=0.5),
    "wide_values": Workload("wide_values", 16, 16, 1024, 1024, 64, 128, MASK_NONE, seed=7),
})
VARIANT_ORDER = ["decoder_target_mask", "prefill_continuation", "wide_values"]

# Decoding steps against a key/value cache (the few-row attn_decode): a served batch
# of 64 sequences x 16 heads with cache lengths in [4096, 8192] of 8192 slots, and
# one long-context pair of sequences with 32768 cached positions. d 128, one query.
WORKLOADS.update({
    "decode_kv_cache": Workload("decode_kv_cache", 64, 16, 1, 8192, 128, 128, MASK_KEY_PADDING, seed=8,
                                len_lo=4096, len_hi=8192, path="decode"),
    "decode_long_context": Workload("decode_long_context", 2, 16, 1, 32768, 128, 128, MASK_NONE, seed=9,
                                    path="decode"),
})
# A speculative-decoding check: 4 draft tokens per sequence verified against a
# cache of 8192 slots filled to [4096, 8192] positions (the causal mask inside each
# entry's filled cache), 64 sequences x 16 heads, d 128.
WORKLOADS["spec_decode_cache"] = Workload("spec_decode_cache", 64, 16, 4, 8192, 128, 128, MASK_CAUSAL_CACHE,
                                          seed=12, len_lo=4096, len_hi=8192, path="decode")
DECODE_ORDER = ["decode_kv_cache", "decode_long_context", "spec_decode_cache"]

# The linear distance bias ("第2章：完整的 Transformer 架构" §5.3) on the big-decoder
# and the long-context causal self-attention.
WORKLOADS.update({
    "alibi_decoder_causal": Workload("alibi_decoder_causal", 16, 16, 1024, 1024, 64, 64, MASK_CAUSAL,
                                     seed=10, alibi=True),
    "alibi_long_causal": Workload("alibi_long_causal", 4, 16, 8192, 8192, 128, 128, MASK_CAUSAL,
                                  seed=11, value_scale=0.5, alibi=True),
})
ALIBI_ORDER = ["alibi_decoder_causal", "alibi_long_causal"]


def alibi_slopes(H: int) -> torch.Tensor:
    """Distance-bias slopes, one per head: the geometric sequence 2^(-8 h / H),
    h = 1..H, of the linear-bias method's paper. fp32 CPU tensor [H]."""
    return torch.tensor([2.0 ** (-8.0 * h / H) for h in range(1, H + 1)], dtype=torch.float32)


@dataclasses.dataclass
class Inputs:
    """bf16 CPU tensors Q [B,H,n,d_k], K [B,H,m,d_k], V [B,H,m,d_v]; int32 key_lengths [B] or None."""

    Q: torch.Tensor
    K: torch.Tensor
    V: torch.Tensor
    key_lengths: torch.Tensor | None
    mask: str
    scale: float


def _normal(g, shape, value_scale):
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if value_scale != 1.0:
        x = x * value_scale
    return x.to(torch.bfloat16)


def make_inputs(B, H, n, m, d_k, d_v, mask=MASK_NONE, seed=0, *, value_scale=1.0,
                len_lo=None, len_hi=None, key_lengths=None, scale=None) -> Inputs:
    """Draw i.i.d. N(0,1)*value_scale Q, K, V (in that order), then key lengths.

    For the key-padding masks the valid lengths are ``randint(len_lo, len_hi+1)``
    unless ``key_lengths`` is given explicitly (a list/tensor of B ints).
    ``scale`` defaults to ``1/sqrt(d_k)``.
    """
    if mask not in MASK_KINDS:
        raise ValueError(f"unknown mask kind {mask!r}")
    g = torch.Generator("cpu").manual_seed(seed)
    Q = _normal(g, (B, H, n, d_k), value_scale)
    K = _normal(g, (B, H, m, d_k), value_scale)
    V = _normal(g, (B, H, m, d_v), value_scale)
    lens = _lengths(g, B, m, mask, len_lo, len_hi, key_lengths)
    return Inputs(Q, K, V, lens, mask, 1.0 / math.sqrt(d_k) if scale is None else float(scale))


def _lengths(g, B, m, mask, len_lo, len_hi, key_lengths):
    if mask not in LENGTH_MASKS:
        return None
    if key_lengths is not None:
        return torch.as_tensor(key_lengths, dtype=torch.int32).reshape(B).clone()
    lo = 1 if len_lo is None else len_lo
    hi = m if len_hi is None else len_hi
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)


def make_grad_output(B, H, n, d_v, seed, value_scale=1.0) -> torch.Tensor:
    """Upstream gradient dO [B,H,n,d_v] for the backward: i.i.d. N(0,1)*value_scale,
    rounded to bf16, from its own seeded generator."""
    g = torch.Generator("cpu").manual_seed(seed)
    return _normal(g, (B, H, n, d_v), value_scale)


def make_linear(out_features, in_features, seed, bias=False):
    """bf16 nn.Linear-layout weight [out, in], Xavier-uniform (bound sqrt(6/(in+out))), and
    if asked a bias [out] drawn U(-1/sqrt(in), 1/sqrt(in)) (nn.Linear's default bias range)."""
    g = torch.Generator("cpu").manual_seed(seed)
    bound = math.sqrt(6.0 / (in_features + out_features))
    W = ((torch.rand(out_features, in_features, generator=g, dtype=torch.float32) * 2.0 - 1.0) * bound)
    b = None
    if bias:
        bb = 1.0 / math.sqrt(in_features)
        b = ((torch.rand(out_features, generator=g, dtype=torch.float32) * 2.0 - 1.0) * bb).to(torch.bfloat16)
    return W.to(torch.bfloat16), b


def make_projection_inputs(B, H, n, d_model, mask, seed, len_lo, len_hi) -> Inputs:
    """Base-encoder recipe: X ~ N(0,1) [B,n,d_model]; W_Q, W_K, W_V Xavier-uniform
    [d_model, d_model] with bound sqrt(6/(2*d_model)), no bias ("Transformer 详解"
    §4.1 uses bias-free projections); Q = (X @ W_Q).view(B,n,H,d).transpose(1,2),
    likewise K and V ("Transformer 详解" §4.2). Draw order: X, W_Q, W_K, W_V,
    then lengths. The projections run in fp32 on the CPU, then round to bf16."""
    d = d_model // H
    g = torch.Generator("cpu").manual_seed(seed)
    X = torch.randn(B, n, d_model, generator=g, dtype=torch.float32)
    bound = math.sqrt(6.0 / (d_model + d_model))
    Ws = [(torch.rand(d_model, d_model, generator=g, dtype=torch.float32) * 2.0 - 1.0) * bound
          for _ in range(3)]
    heads = [(X @ W).view(B, n, H, d).transpose(1, 2).contiguous().to(torch.bfloat16) for W in Ws]
    lens = _lengths(g, B, n, mask, len_lo, len_hi, None)
    return Inputs(heads[0], heads[1], heads[2], lens, mask, 1.0 / math.sqrt(d))


def workload_inputs(w: Workload | str) -> Inputs:
    """The seeded inputs of one named workload."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    if w.recipe == "projection":
        return make_projection_inputs(w.B, w.H, w.n, w.d_model, w.mask, w.seed, w.len_lo, w.len_hi)
    return make_inputs(w.B, w.H, w.n, w.m, w.d_k, w.d_v, w.mask, w.seed,
                       value_scale=w.value_scale,
                       len_lo=w.len_lo if w.mask in LENGTH_MASKS else None,
                       len_hi=w.len_hi if w.mask in LENGTH_MASKS else None)


def sample_rows(B, H, n, count, seed):
    """A seeded sample of ``count`` distinct flat query-row indices into [B*H*n],
    always including the first and last row of the tensor."""
    total = B * H * n
    if count >= total:
        return torch.arange(total, dtype=torch.int64)
    g = torch.Generator("cpu").manual_seed(seed)
    idx = torch.randperm(total, generator=g)[: max(count - 2, 0)]
    idx = torch.unique(torch.cat([idx, torch.tensor([0, total - 1])]))
    return idx.to(torch.int64)

"""Pins of the oracle's causal mask inside a partly filled key/value cache.

The wiki page's KV cache ("实现要点": a cache of fixed size allocated up front,
each step adding the new tokens' K and V, batches supported) holds len_b valid
positions of m slots per batch entry; the n new queries are the last n of those
len_b positions, so query i sees the keys j < len_b with j <= i + (len_b - n).
This is the causal mask of reading 4 applied to each entry's filled length
instead of to m. Each pin raises AssertionError on a mismatch; a planted copy that
aligns the diagonal to m instead of len_b must fail at least one.
"""

import numpy as np
import pytest
import torch

from oracle import oracle


def rnd(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64).numpy()


def pin_cache_is_causal_on_the_filled_part(plant=0):
    """Entry b equals the causal oracle on its first len_b keys (pinned for n <= m by the
    causal suffix pin); the cache slots past len_b do not matter."""
    B, H, n, m, d = 3, 2, 4, 12, 8
    Q, K, V = rnd((B, H, n, d), 1), rnd((B, H, m, d), 2), rnd((B, H, m, 5), 3)
    lens = [12, 7, 4]
    O, L = oracle.attn_fwd(Q, K, V, "causal_cache", key_lengths=lens, plant=plant)
    for b, ln in enumerate(lens):
        Oc, Lc = oracle.attn_fwd(Q[b:b + 1], K[b:b + 1, :, :ln], V[b:b + 1, :, :ln], "causal", plant=plant)
        np.testing.assert_allclose(O[b:b + 1], Oc, atol=1e-12)
        np.testing.assert_allclose(L[b:b + 1], Lc, atol=1e-12)


def pin_cache_full_is_causal(plant=0):
    """A cache filled to m is the causal mask itself."""
    B, H, n, m, d = 2, 2, 5, 9, 8
    Q, K, V = rnd((B, H, n, d), 4), rnd((B, H, m, d), 5), rnd((B, H, m, 3), 6)
    O, L = oracle.attn_fwd(Q, K, V, "causal_cache", key_lengths=[m, m], plant=plant)
    Oc, Lc = oracle.attn_fwd(Q, K, V, "causal", plant=plant)
    np.testing.assert_array_equal(O, Oc)
    np.testing.assert_array_equal(L, Lc)


def pin_cache_library(plant=0):
    """Against torch fp64 scaled_dot_product_attention with the boolean mask
    (j < len_b) & (j <= i + len_b - n) and torch.logsumexp (rows that see a key)."""
    B, H, n, m, d = 3, 2, 6, 16, 8
    Q, K, V = rnd((B, H, n, d), 7), rnd((B, H, m, d), 8), rnd((B, H, m, 4), 9)
    lens = [16, 9, 6]
    O, L = oracle.attn_fwd(Q, K, V, "causal_cache", key_lengths=lens, plant=plant)
    i = torch.arange(n)[:, None]
    j = torch.arange(m)[None, :]
    ln = torch.tensor(lens).view(B, 1, 1, 1)
    allowed = (j < ln) & (j <= i + ln - n)
    q, k, v = map(torch.from_numpy, (Q, K, V))
    Ot = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=allowed, scale=1 / 8 ** 0.5)
    Lt = torch.logsumexp((q @ k.transpose(-1, -2) / 8 ** 0.5).masked_fill(~allowed, float("-inf")), -1)
    np.testing.assert_allclose(O, Ot.numpy(), atol=1e-12)
    np.testing.assert_allclose(L, Lt.numpy(), atol=1e-12)


PINS = [pin_cache_is_causal_on_the_filled_part, pin_cache_full_is_causal, pin_cache_library]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(0)


def test_planted_alignment_is_caught():
    caught = []
    for pin in PINS:
        try:
            pin(18)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, "the diagonal aligned to m passed every pin"


def test_rows_before_the_cache_start_see_nothing():
    """n > len_b: the first n - len_b queries precede the filled part (reading 2)."""
    Q, K, V = rnd((1, 1, 5, 4), 10), rnd((1, 1, 8, 4), 11), rnd((1, 1, 8, 2), 12)
    O, L = oracle.attn_fwd(Q, K, V, "causal_cache", key_lengths=[3])
    assert np.all(np.isneginf(L[0, 0, :2])) and np.all(O[0, 0, :2] == 0)
    assert np.all(np.isfinite(L[0, 0, 2:]))


def test_backward_matches_truncated_causal():
    """The backward under the cache mask equals the causal backward on the filled part,
    and the cache slots past len_b get zero gradient."""
    B, H, n, m, d = 2, 1, 3, 7, 4
    Q, K, V, G = rnd((B, H, n, d), 13), rnd((B, H, m, d), 14), rnd((B, H, m, 3), 15), rnd((B, H, n, 3), 16)
    lens = [7, 5]
    dQ, dK, dV = oracle.attn_bwd(Q, K, V, G, "causal_cache", lens)
    for b, ln in enumerate(lens):
        rq, rk, rv = oracle.attn_bwd(Q[b:b + 1], K[b:b + 1, :, :ln], V[b:b + 1, :, :ln], G[b:b + 1], "causal")
        np.testing.assert_allclose(dQ[b:b + 1], rq, atol=1e-12)
        np.testing.assert_allclose(dK[b:b + 1, :, :ln], rk, atol=1e-12)
        np.testing.assert_allclose(dV[b:b + 1, :, :ln], rv, atol=1e-12)
        assert np.all(dK[b, :, ln:] == 0) and np.all(dV[b, :, ln:] == 0)

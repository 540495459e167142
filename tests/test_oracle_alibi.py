"""Pins of the oracle's linear distance bias ("第2章：完整的 Transformer 架构" §5.3,
ALiBi): softmax(Q Kᵀ / sqrt(d_k) - m_h D) V with D_ij = |i' - j| and a slope m_h per
head, i' = i + (m - n) the query's position among the keys.

Each pin raises AssertionError on a mismatch; the tests run them on the shipped
oracle and on copies with a planted mistake (bias added instead of subtracted,
query position not aligned for n != m, slope taken per batch entry instead of per
head, the bias dropped in the backward), each of which at least one pin must catch.
"""

import math

import numpy as np
import pytest
import torch

from oracle import oracle

MASKS = ("none", "causal", "key_padding", "causal_key_padding")


def rnd(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g, dtype=torch.float64) * scale).numpy()


def pin_alibi_zero_slope(plant=0):
    """Slope 0 is no bias: the result equals the unbiased oracle exactly, every mask."""
    B, H, n, m, d = 2, 3, 7, 11, 8
    Q, K, V = rnd((B, H, n, d), 1), rnd((B, H, m, d), 2), rnd((B, H, m, 5), 3)
    lens = [11, 6]
    for mask in MASKS:
        O, L = oracle.attn_fwd(Q, K, V, mask, key_lengths=lens, slopes=np.zeros(H), plant=plant)
        O0, L0 = oracle.attn_fwd(Q, K, V, mask, key_lengths=lens, plant=plant)
        assert np.array_equal(O, O0) and np.array_equal(L, L0)


def _geometric(r, N):
    """Sum_{k=0}^{N} r^k and sum_{k=0}^{N} k r^k in closed form (0 < r < 1)."""
    s0 = (1.0 - r ** (N + 1)) / (1.0 - r)
    s1 = r * (1.0 - (N + 1) * r ** N + N * r ** (N + 1)) / (1.0 - r) ** 2
    return s0, s1


def pin_alibi_geometric(plant=0):
    """Equal raw scores (Q = 0) under the causal mask: query position i' sees keys
    0..i' with weights r^(i'-j) / Z, r = e^-m_h, so Z = (1 - r^(i'+1)) / (1 - r) (a
    geometric series), LSE = ln Z, and with v_j = (j, 1) the output is
    (i' - sum_k k r^k / Z, 1). Checked for n = m and for n < m (i' = i + m - n), with a
    different slope in every head of two batch entries."""
    slopes = np.array([0.25, 0.7, 1.3])
    B, H, d = 2, 3, 4
    for n, m in ((6, 6), (3, 9)):
        Q = np.zeros((B, H, n, d))
        K = rnd((B, H, m, d), 4)
        V = np.zeros((B, H, m, 2))
        V[..., 0] = np.arange(m)[None, None, :]
        V[..., 1] = 1.0
        O, L = oracle.attn_fwd(Q, K, V, "causal", slopes=slopes, plant=plant)
        for b in range(B):
            for h in range(H):
                r = math.exp(-slopes[h])
                for i in range(n):
                    ip = i + m - n
                    s0, s1 = _geometric(r, ip)
                    assert abs(L[b, h, i] - math.log(s0)) < 1e-12
                    assert abs(O[b, h, i, 0] - (ip - s1 / s0)) < 1e-11
                    assert abs(O[b, h, i, 1] - 1.0) < 1e-12


def pin_alibi_nearest_key(plant=0):
    """A very large slope leaves only the visible key nearest to the query position:
    v_{i'} without a mask or under the causal mask, v_{len-1} once i' >= len under key
    padding (the nearest visible key), within e^-40."""
    B, H, n, m, d = 2, 2, 5, 9, 8
    Q, K = rnd((B, H, n, d), 5, 0.1), rnd((B, H, m, d), 6, 0.1)
    V = rnd((B, H, m, 3), 7)
    slopes = np.full(H, 40.0)
    lens = [9, 6]
    for mask in MASKS:
        O, _ = oracle.attn_fwd(Q, K, V, mask, key_lengths=lens, slopes=slopes, plant=plant)
        for b in range(B):
            for i in range(n):
                ip = i + m - n
                j = min(ip, lens[b] - 1) if mask in ("key_padding", "causal_key_padding") else ip
                np.testing.assert_allclose(O[b, :, i], V[b, :, j], atol=1e-12)


def _torch_bias_ref(Q, K, V, mask, lens, scale, slopes):
    """Library reference: torch fp64 scaled_dot_product_attention with a float additive
    mask (the bias, -inf where masked) and torch.logsumexp."""
    q, k, v = map(torch.from_numpy, (Q, K, V))
    B, H, n, _ = q.shape
    m = k.shape[2]
    dist = (torch.arange(n)[:, None] + (m - n) - torch.arange(m)[None, :]).abs().double()
    bias = -torch.from_numpy(np.asarray(slopes, dtype=np.float64)).view(1, H, 1, 1) * dist
    allowed = torch.ones(1, 1, n, m, dtype=torch.bool)
    if mask in ("causal", "causal_key_padding"):
        allowed = allowed & torch.ones(n, m, dtype=torch.bool).tril(diagonal=m - n)
    if mask in ("key_padding", "causal_key_padding"):
        allowed = allowed & (torch.arange(m)[None, :] < torch.tensor(lens)[:, None]).view(B, 1, 1, m)
    add = bias.expand(B, H, n, m).masked_fill(~allowed, float("-inf"))
    O = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=add, scale=scale)
    L = torch.logsumexp(torch.matmul(q, k.transpose(-1, -2)) * scale + add, dim=-1)
    return O.numpy(), L.numpy()


def pin_alibi_library(plant=0):
    """Tiny shapes, every mask, n = m and n != m, against the library reference."""
    cases = [(2, 3, 8, 8, 16, 8, [8, 5]), (1, 2, 4, 13, 8, 8, [13]), (2, 2, 12, 5, 8, 4, [5, 2])]
    for t, (B, H, n, m, dk, dv, lens) in enumerate(cases):
        Q, K, V = rnd((B, H, n, dk), 10 + t), rnd((B, H, m, dk), 20 + t), rnd((B, H, m, dv), 30 + t)
        slopes = 2.0 ** (-8.0 * np.arange(1, H + 1) / H)
        for mask in MASKS:
            if mask in ("causal", "causal_key_padding") and n > m:
                continue                      # rows without a visible key: reading, not library
            O, L = oracle.attn_fwd(Q, K, V, mask, key_lengths=lens, slopes=slopes, plant=plant)
            Ot, Lt = _torch_bias_ref(Q, K, V, mask, lens, 1.0 / math.sqrt(dk), slopes)
            np.testing.assert_allclose(O, Ot, atol=1e-12)
            np.testing.assert_allclose(L, Lt, atol=1e-12)


def pin_alibi_bwd_finite_differences(plant=0):
    """The backward of the biased forward: for L = sum(O * G) every entry of dQ, dK, dV
    equals the central difference of the (pinned) biased forward oracle, h = 1e-6."""
    h = 1e-6
    cases = [(1, 2, 4, 4, 2, 2, "causal", None), (1, 2, 3, 5, 2, 3, "none", None),
             (2, 1, 3, 6, 2, 2, "causal_key_padding", [6, 4])]
    for t, (B, H, n, m, dk, dv, mask, lens) in enumerate(cases):
        Q, K, V = rnd((B, H, n, dk), 50 + t), rnd((B, H, m, dk), 60 + t), rnd((B, H, m, dv), 70 + t)
        G = rnd((B, H, n, dv), 80 + t)
        slopes = np.array([0.6, 0.15][:H])
        grads = oracle.attn_bwd(Q, K, V, G, mask, lens, 0.8, slopes=slopes, threads=1, plant=plant)

        def loss():
            O, _ = oracle.attn_fwd(Q, K, V, mask, lens, 0.8, slopes=slopes, threads=1, plant=plant)
            return float(np.sum(O * G))

        for x, gx in zip((Q, K, V), grads):
            fd = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                old = x[idx]
                x[idx] = old + h
                lp = loss()
                x[idx] = old - h
                lm = loss()
                x[idx] = old
                fd[idx] = (lp - lm) / (2 * h)
            np.testing.assert_allclose(gx, fd, atol=1e-7, err_msg=f"case {t} ({mask})")


PINS = [pin_alibi_zero_slope, pin_alibi_geometric, pin_alibi_nearest_key, pin_alibi_library,
        pin_alibi_bwd_finite_differences]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(0)


@pytest.mark.parametrize("plant", [14, 15, 16, 17])
def test_planted_mistake_is_caught(plant):
    caught = []
    for pin in PINS:
        try:
            pin(plant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {plant} passed every pin"


def test_rows_match_full():
    """The sampled-row entry point gives the full forward's rows."""
    B, H, n, m, d = 2, 2, 6, 10, 8
    Q, K, V = rnd((B, H, n, d), 40), rnd((B, H, m, d), 41), rnd((B, H, m, 4), 42)
    slopes = np.array([0.5, 0.125])
    O, L = oracle.attn_fwd(Q, K, V, "causal_key_padding", key_lengths=[10, 7], slopes=slopes)
    rows = np.array([0, 5, 13, 23])
    Or, Lr = oracle.attn_rows(Q, K, V, rows, "causal_key_padding", key_lengths=[10, 7], slopes=slopes)
    np.testing.assert_array_equal(Or, O.reshape(-1, 4)[rows])
    np.testing.assert_array_equal(Lr, L.reshape(-1)[rows])


def test_slopes_shape_checked():
    Q = np.zeros((1, 2, 3, 4))
    with pytest.raises(ValueError):
        oracle.attn_fwd(Q, Q, Q, "none", slopes=[1.0, 2.0, 3.0])

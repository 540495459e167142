"""Pins of the oracle's attention backward (dQ, dK, dV for an upstream gradient dO).

The pages print the forward only; the backward is the chain rule through it, so
it is pinned to the forward (finite differences of the pinned forward oracle),
to a library's automatic differentiation, and to identities the softmax forces.
Each planted backward mistake (a dropped D_i term, a dropped scale in dK, O in
place of dO in dV) must fail at least one pin.
"""

import numpy as np
import pytest
import torch

from oracle import oracle


def rnd(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g, dtype=torch.float64) * scale).numpy()


# (B, H, n, m, dk, dv, mask, key lengths)
FD_CASES = [
    (1, 2, 3, 5, 3, 2, "none", None),
    (1, 1, 4, 4, 2, 3, "causal", None),
    (1, 1, 3, 6, 2, 2, "causal", None),        # bottom-right: row i sees j <= i + 3
    (2, 1, 3, 5, 2, 2, "key_padding", [2, 5]),
    (2, 1, 4, 4, 2, 2, "causal_key_padding", [3, 1]),
]


def _loss(Q, K, V, G, mask, lens, scale, plant):
    O, _ = oracle.attn_fwd(Q, K, V, mask, lens, scale, threads=1, plant=plant)
    return float(np.sum(O * G))


def pin_bwd_finite_differences(plant=0):
    """For L = sum(O * G), every entry of dQ, dK, dV equals the central difference
    (L(x + h) - L(x - h)) / 2h of the forward oracle, h = 1e-6 (truncation ~h^2,
    cancellation ~1e-16/h: both far below the 1e-7 tolerance)."""
    h = 1e-6
    for t, (B, H, n, m, dk, dv, mask, lens) in enumerate(FD_CASES):
        Q, K, V = rnd((B, H, n, dk), 40 + t), rnd((B, H, m, dk), 50 + t), rnd((B, H, m, dv), 60 + t)
        G = rnd((B, H, n, dv), 70 + t)
        sc = 0.8
        grads = oracle.attn_bwd(Q, K, V, G, mask, lens, sc, threads=1, plant=plant)
        for x, gx in zip((Q, K, V), grads):
            fd = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                old = x[idx]
                x[idx] = old + h
                lp = _loss(Q, K, V, G, mask, lens, sc, plant)
                x[idx] = old - h
                lm = _loss(Q, K, V, G, mask, lens, sc, plant)
                x[idx] = old
                fd[idx] = (lp - lm) / (2 * h)
            np.testing.assert_allclose(gx, fd, atol=1e-7, err_msg=f"case {t} ({mask})")


def _torch_grads(Q, K, V, G, mask, lens, scale):
    q, k, v = (torch.from_numpy(a.copy()).requires_grad_(True) for a in (Q, K, V))
    B, H, n, _ = q.shape
    m = k.shape[2]
    allowed = torch.ones(1, 1, n, m, dtype=torch.bool)
    if mask in ("causal", "causal_key_padding"):
        allowed = allowed & torch.ones(n, m, dtype=torch.bool).tril(diagonal=m - n)
    if mask in ("key_padding", "causal_key_padding"):
        allowed = allowed & (torch.arange(m)[None, :] < torch.tensor(lens)[:, None]).view(B, 1, 1, m)
    O = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=allowed, scale=scale)
    (O * torch.from_numpy(G)).sum().backward()
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


def pin_bwd_library_autograd(plant=0):
    """torch fp64 autograd through scaled_dot_product_attention with a boolean mask
    (every row keeps at least one key), within 1e-12."""
    cases = [
        (2, 2, 9, 9, 16, 16, "none", None),
        (1, 3, 17, 17, 8, 4, "causal", None),
        (2, 1, 5, 13, 8, 8, "causal", None),
        (3, 2, 7, 12, 8, 16, "key_padding", [12, 1, 7]),
        (2, 2, 10, 10, 16, 8, "causal_key_padding", [10, 4]),
    ]
    for t, (B, H, n, m, dk, dv, mask, lens) in enumerate(cases):
        Q, K, V = rnd((B, H, n, dk), 80 + t), rnd((B, H, m, dk), 90 + t), rnd((B, H, m, dv), 100 + t)
        G = rnd((B, H, n, dv), 110 + t)
        sc = 1.0 / np.sqrt(dk)
        ours = oracle.attn_bwd(Q, K, V, G, mask, lens, sc, plant=plant)
        ref = _torch_grads(Q, K, V, G, mask, lens, sc)
        for a, b, name in zip(ours, ref, ("dQ", "dK", "dV")):
            np.testing.assert_allclose(a, b, atol=1e-12, err_msg=f"{name} case {t} ({mask})")


def pin_bwd_identities(plant=0):
    """Softmax identities, for every mask: the weights of a row sum to one, so the keys'
    gradients dK sum to zero over the keys of a head and dV sums to the dO of the rows
    that see a key; masked keys get exactly zero gradient; with all keys equal the
    scores do not depend on Q, so dQ = 0."""
    B, H, n, m, d = 3, 2, 6, 9, 4
    Q, K, V = rnd((B, H, n, d), 120), rnd((B, H, m, d), 121), rnd((B, H, m, d), 122)
    G = rnd((B, H, n, d), 123)
    lens = [9, 4, 0]
    for mask in ("none", "causal", "key_padding", "causal_key_padding"):
        L = lens if mask in ("key_padding", "causal_key_padding") else None
        dQ, dK, dV = oracle.attn_bwd(Q, K, V, G, mask, L, 0.7, plant=plant)
        np.testing.assert_allclose(dK.sum(axis=2), 0.0, atol=1e-12)
        _, lse = oracle.attn_fwd(Q, K, V, mask, L, 0.7, plant=plant)
        seen = np.isfinite(lse)[..., None]
        np.testing.assert_allclose(dV.sum(axis=2), (G * seen).sum(axis=2), atol=1e-12)
        if L is not None:
            for b, ln in enumerate(L):
                assert np.all(dK[b, :, ln:] == 0.0) and np.all(dV[b, :, ln:] == 0.0)
                if ln == 0:
                    assert np.all(dQ[b] == 0.0)
    Ke = np.broadcast_to(K[:, :, :1], K.shape).copy()
    dQ, _, _ = oracle.attn_bwd(Q, Ke, V, G, "none", None, 0.7, plant=plant)
    np.testing.assert_allclose(dQ, 0.0, atol=1e-12)


PINS = [pin_bwd_finite_differences, pin_bwd_library_autograd, pin_bwd_identities]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(0)


@pytest.mark.parametrize("plant", [9, 10, 11])
def test_planted_backward_mistake_is_caught(plant):
    caught = []
    for pin in PINS:
        try:
            pin(plant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {plant} passed every pin"


def test_bwd_rejects_bad_shapes():
    Q = rnd((1, 1, 3, 4), 1)
    with pytest.raises(ValueError):
        oracle.attn_bwd(Q, Q, Q, rnd((1, 1, 3, 5), 2))

"""Pins of the oracle's projections around the attention (the QKV projection with
its head split, and the head merge with W_O), against the pages' view/transpose
semantics written out element by element and against identities. Two planted
mistakes (head split with the (head, dim) order swapped; an untransposed weight)
must each fail a pin."""

import numpy as np
import pytest
import torch

from oracle import oracle


def rnd(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64).numpy()


def pin_loops(plant=0):
    """Pure-Python loops from the definitions: y[b,i,c] = sum_k x[b,i,k] W[c,k] + bias[c];
    head t's tensor at [b,h,i,j] is y[b,i, t*d_model + h*d + j] (view(B, n, h, d) then
    transpose(1, 2)); the merge puts head h's column j at h*d + j of the row."""
    B, n, dm, H, num = 2, 3, 6, 3, 3
    d = dm // H
    X, W, bias = rnd((B, n, dm), 1), rnd((num * dm, dm), 2), rnd((num * dm,), 3)
    outs = oracle.proj_heads(X, W, bias, H, num, plant=plant)
    for t in range(num):
        for b in range(B):
            for h in range(H):
                for i in range(n):
                    for j in range(d):
                        c = t * dm + h * d + j
                        ref = sum(X[b, i, k] * W[c, k] for k in range(dm)) + bias[c]
                        assert abs(outs[t][b, h, i, j] - ref) < 1e-12
    O, Wo, bo = rnd((B, H, n, d), 4), rnd((5, dm), 5), rnd((5,), 6)
    Y = oracle.merge_proj(O, Wo, bo, plant=plant)
    for b in range(B):
        for i in range(n):
            for c in range(5):
                ref = sum(O[b, h, i, j] * Wo[c, h * d + j] for h in range(H) for j in range(d)) + bo[c]
                assert abs(Y[b, i, c] - ref) < 1e-12


def pin_round_trip(plant=0):
    """With identity weights and no bias, merging the split heads gives the input back,
    for every head count; a one-hot input row picks one weight column."""
    B, n, dm = 2, 5, 12
    X = rnd((B, n, dm), 7)
    for H in (1, 2, 3, 4, 6):
        (Qh,) = oracle.proj_heads(X, np.eye(dm), None, H, 1, plant=plant)
        assert Qh.shape == (B, H, n, dm // H)
        Y = oracle.merge_proj(Qh, np.eye(dm), None, plant=plant)
        np.testing.assert_allclose(Y, X, atol=1e-12)
    W = rnd((dm, dm), 8)
    Xo = np.zeros((1, 1, dm))
    Xo[0, 0, 5] = 1.0
    (Qo,) = oracle.proj_heads(Xo, W, None, 3, 1, plant=plant)
    np.testing.assert_allclose(Qo.transpose(0, 2, 1, 3).reshape(dm), W[:, 5], atol=1e-12)


def pin_bias_and_linearity(plant=0):
    """The bias shifts every row by the same vector; the projection is linear in X."""
    B, n, dm, H = 2, 4, 8, 2
    X1, X2, W, bias = rnd((B, n, dm), 9), rnd((B, n, dm), 10), rnd((2 * dm, dm), 11), rnd((2 * dm,), 12)
    a = oracle.proj_heads(X1, W, bias, H, 2, plant=plant)
    z = oracle.proj_heads(X1, W, None, H, 2, plant=plant)
    for t in range(2):
        shift = bias[t * dm:(t + 1) * dm].reshape(H, 1, dm // H)
        np.testing.assert_allclose(a[t] - z[t], np.broadcast_to(shift, a[t].shape[1:])[None].repeat(B, 0),
                                   atol=1e-12)
    s = oracle.proj_heads(2.0 * X1 - 3.0 * X2, W, None, H, 2, plant=plant)
    p1 = oracle.proj_heads(X1, W, None, H, 2, plant=plant)
    p2 = oracle.proj_heads(X2, W, None, H, 2, plant=plant)
    for t in range(2):
        np.testing.assert_allclose(s[t], 2.0 * p1[t] - 3.0 * p2[t], atol=1e-11)


def pin_multihead_attention(plant=0):
    """The whole multi-head self-attention of "第2章：完整的 Transformer 架构" §7.5
    (nn.MultiheadAttention): the oracle's QKV projection and head split, attention and
    head merge with W_O against torch's fp64 nn.MultiheadAttention with the same
    weights (in_proj_weight is the stacked W_Q, W_K, W_V), with no mask, the causal
    mask (attn_mask, True = masked) and key padding (key_padding_mask)."""
    B, n, E, H = 2, 7, 12, 3
    X = rnd((B, n, E), 20)
    mha = torch.nn.MultiheadAttention(E, H, bias=True, batch_first=True, dtype=torch.float64)
    with torch.no_grad():
        for prm, seed in ((mha.in_proj_weight, 21), (mha.in_proj_bias, 22), (mha.out_proj.weight, 23),
                          (mha.out_proj.bias, 24)):
            prm.copy_(torch.from_numpy(rnd(tuple(prm.shape), seed)))
    Xt = torch.from_numpy(X)
    lens = [7, 4]
    cases = {
        "none": dict(),
        "causal": dict(attn_mask=torch.ones(n, n, dtype=torch.bool).triu(1)),
        "key_padding": dict(key_padding_mask=torch.arange(n)[None, :] >= torch.tensor(lens)[:, None]),
    }
    for mask, kw in cases.items():
        with torch.no_grad():
            ref, _ = mha(Xt, Xt, Xt, need_weights=False, **kw)
        Q, K, V = oracle.proj_heads(X, mha.in_proj_weight.detach(), mha.in_proj_bias.detach(), H, 3, plant=plant)
        O, _ = oracle.attn_fwd(Q, K, V, mask, key_lengths=lens if mask == "key_padding" else None)
        Y = oracle.merge_proj(O, mha.out_proj.weight.detach(), mha.out_proj.bias.detach(), plant=plant)
        np.testing.assert_allclose(Y, ref.numpy(), atol=1e-12, err_msg=mask)


PINS = [pin_loops, pin_round_trip, pin_bias_and_linearity, pin_multihead_attention]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(0)


@pytest.mark.parametrize("plant", [12, 13])
def test_planted_projection_mistake_is_caught(plant):
    caught = []
    for pin in PINS:
        try:
            pin(plant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {plant} passed every pin"

"""GPU parity with K and V past 2^31 bytes each: B = 2, H = 68, m = 131,277 keys
(a ragged last key tile), d = 64, so 2.29 GB per tensor and every byte offset of
the last (b, h) pair above 2^31. A kernel that formed any of its global offsets in
32 bits would wrap there.

The last pair holds a seeded random input checked against the fp64 oracle. Every
other pair holds K = 0 and V = -3: all its scores are 0, so the weights are
uniform, O = -3 exactly, LSE = ln m, and the gradients are dQ = dK = 0 (dP equals
D for every key) and dV_j = (1/m) sum_i dO_i for every key j. A read or write at a
wrapped offset in the last pair meets these constants, or lands on them.
Tolerances are those of test_parity (forward, decode) and test_bwd_parity
(backward).
"""

import math

import numpy as np
import pytest
import torch

from oracle import oracle
from transformer_scaled_dot_03_gb300 import attn, build, inputs

from test_bwd_parity import U, bounds
from test_parity import compare

pytestmark = pytest.mark.gpu

B, H, M, D = 2, 68, 131_277, 64
V_CONST = -3.0


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return attn.load()


def test_sizes_cross_2_31_bytes():
    """The premise, on the host: the last pair starts past 2^31 bytes."""
    assert (B * H - 1) * M * D * 2 > 2 ** 31


def big_kv(x):
    """K, V [B, H, M, D] on the device: the constant pairs and the seeded last pair."""
    K = torch.zeros(B, H, M, D, dtype=torch.bfloat16, device="cuda")
    V = torch.full((B, H, M, D), V_CONST, dtype=torch.bfloat16, device="cuda")
    K[-1, -1] = x.K[0, 0].cuda()
    V[-1, -1] = x.V[0, 0].cuda()
    return K, V


def spread(t):
    """A [1, 1, r, c] tensor repeated to every (b, h) pair, on the device."""
    return t.cuda().expand(B, H, t.shape[2], t.shape[3]).contiguous()


def check_constant_pairs(O, L, label):
    """O = -3 exactly and LSE = ln m on every pair but the last."""
    Oc = O.view(B * H, -1)[:-1]
    Lc = L.view(B * H, -1)[:-1]
    assert torch.all(Oc == V_CONST), f"{label}: constant pairs' O differs from {V_CONST}"
    lerr = (Lc.double() - math.log(M)).abs().max().item()
    assert lerr <= 1e-5, f"{label}: constant pairs' LSE off ln m by {lerr:.3e}"


def test_forward_past_2_31_bytes():
    n = 130
    x = inputs.make_inputs(1, 1, n, M, D, D, "none", seed=9100)
    K, V = big_kv(x)
    O, L = attn.attn_fwd(spread(x.Q), K, V, "none", None, x.scale)
    rc, detail = attn.device_status()
    assert rc == attn.ATTN_OK, (rc, detail)
    check_constant_pairs(O, L, "forward")
    Or, Lr = oracle.attn_fwd(x.Q, x.K, x.V, "none", None, x.scale)
    compare(O[-1:, -1:].float().cpu().numpy(), L[-1:, -1:].cpu().numpy(), Or, Lr, "forward, last pair")


def test_decode_past_2_31_bytes():
    x = inputs.make_inputs(1, 1, 1, M, D, D, "none", seed=9200)
    K, V = big_kv(x)
    O, L = attn.attn_decode(spread(x.Q), K, V, "none", None, x.scale)
    rc, detail = attn.device_status()
    assert rc == attn.ATTN_OK, (rc, detail)
    check_constant_pairs(O, L, "decode")
    Or, Lr = oracle.attn_fwd(x.Q, x.K, x.V, "none", None, x.scale)
    compare(O[-1:, -1:].float().cpu().numpy(), L[-1:, -1:].cpu().numpy(), Or, Lr, "decode, last pair")


def test_backward_past_2_31_bytes():
    n = 130
    x = inputs.make_inputs(1, 1, n, M, D, D, "none", seed=9300)
    dO = inputs.make_grad_output(1, 1, n, D, seed=9301)
    K, V = big_kv(x)
    Q, G = spread(x.Q), spread(dO)
    O, L = attn.attn_fwd(Q, K, V, "none", None, x.scale)
    dQ, dK, dV = attn.attn_bwd(Q, K, V, O, L, G, "none", None, x.scale)
    rc, detail = attn.device_status()
    assert rc == attn.ATTN_OK, (rc, detail)
    del K, V, O, L

    # constant pairs: dQ = 0 exactly, dK = 0 up to the rounding of dP - D, dV_j = mean of dO rows
    e = (dO[0, 0].double().sum(0) / M).cuda()
    dQc, dKc, dVc = (t.view(B * H, -1, D)[:-1] for t in (dQ, dK, dV))
    assert torch.all(dQc == 0), "constant pairs' dQ is not zero"
    for p0 in range(0, B * H - 1, 16):
        kerr = dKc[p0:p0 + 16].float().abs().max().item()
        assert kerr <= 1e-6, f"constant pairs {p0}..: |dK| reaches {kerr:.3e}"
        verr = ((dVc[p0:p0 + 16].double() - e).abs() - (2 * U * e.abs() + 1e-6)).max().item()
        assert verr <= 0, f"constant pairs {p0}..: dV exceeds its bound by {verr:.3e}"

    # the last pair against the oracle, with the bounds of the backward parity tests
    got = tuple(t[-1:, -1:].float().cpu().numpy() for t in (dQ, dK, dV))
    refs = oracle.attn_bwd(x.Q, x.K, x.V, dO, "none", None, x.scale)
    for name, Gd, R, bd in zip(("dQ", "dK", "dV"), got, refs, bounds(x, dO, refs)):
        assert np.all(np.isfinite(Gd)), f"last pair: non-finite {name}"
        excess = np.abs(Gd - R) - (2 * bd + 1e-6)
        assert excess.max() <= 0, f"last pair: {name} exceeds its bound by {excess.max():.3e}"

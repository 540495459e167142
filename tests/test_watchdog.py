"""Device-side watchdog: every wait in the kernel is bounded. A debug flag makes
the softmax warps wait on a barrier that nothing completes; the kernel must give
up after its short limit, report ATTN_ERR_TIMEOUT through the status word,
release its tensor memory and leave the context usable (no trap, no fault)."""

import numpy as np
import pytest
import torch

from oracle import oracle
from transformer_scaled_dot_03_gb300 import attn, build, inputs

pytestmark = pytest.mark.gpu

FORCED_BIT = 8   # status bit of the forced wait


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return attn.load()


def _run(x):
    lens = x.key_lengths.cuda() if x.key_lengths is not None else None
    return attn.attn_fwd(x.Q.cuda(), x.K.cuda(), x.V.cuda(), x.mask, lens, x.scale)


@pytest.mark.parametrize("mask,d", [("none", 64), ("causal", 128), ("key_padding", 64)])
def test_forced_timeout_reports_and_recovers(mask, d):
    x = inputs.make_inputs(1, 2, 300, 300, d, d, mask, seed=5000, len_lo=200, len_hi=300)
    assert attn.device_status() == (attn.ATTN_OK, 0)
    attn.set_watchdog(0, 1)
    try:
        _run(x)
        rc, detail = attn.device_status()
    finally:
        attn.set_watchdog(0, 0)
    assert rc == attn.ATTN_ERR_TIMEOUT
    assert detail & FORCED_BIT
    # the status word was cleared, and a normal call afterwards is correct
    O, L = _run(x)
    assert attn.device_status() == (attn.ATTN_OK, 0)
    Or, Lr = oracle.attn_fwd(x.Q, x.K, x.V, x.mask, x.key_lengths, x.scale)
    assert np.abs(O.float().cpu().numpy() - Or).max() <= 1e-2
    assert np.abs(L.cpu().numpy() - Lr).max() <= 1e-3


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128)])
def test_forced_timeout_in_the_backward(dk, dv):
    """The same for the backward kernels (the persistent 128-query-tile kernel at
    d = 64, the 64-query-step kernel with two MMA issuers and a read-out warpgroup at
    d = 128, the one-tile-per-CTA kernel for d_k != d_v): the forced wait gives up,
    the status reports it, every role leaves, and a normal backward afterwards
    matches the oracle."""
    x = inputs.make_inputs(2, 2, 260, 260, dk, dv, "causal", seed=5100 + dk + dv)
    dO = inputs.make_grad_output(2, 2, 260, dv, seed=5101 + dk + dv)
    Q, K, V, g = x.Q.cuda(), x.K.cuda(), x.V.cuda(), dO.cuda()
    O, L = attn.attn_fwd(Q, K, V, x.mask, None, x.scale)
    assert attn.device_status() == (attn.ATTN_OK, 0)
    attn.set_watchdog(0, 1)
    try:
        attn.attn_bwd(Q, K, V, O, L, g, x.mask, None, x.scale)
        rc, detail = attn.device_status()
    finally:
        attn.set_watchdog(0, 0)
    assert rc == attn.ATTN_ERR_TIMEOUT
    assert detail & FORCED_BIT
    dQ, dK, dV = attn.attn_bwd(Q, K, V, O, L, g, x.mask, None, x.scale)
    assert attn.device_status() == (attn.ATTN_OK, 0)
    rq, rk, rv = oracle.attn_bwd(x.Q, x.K, x.V, dO, x.mask, None, x.scale)
    for G, R in ((dQ, rq), (dK, rk), (dV, rv)):
        G = G.float().cpu().numpy()
        assert np.all(np.isfinite(G))
        assert np.abs(G - R).max() <= 0.05 * max(1.0, np.abs(R).max())


def test_forced_timeout_in_the_decode_path():
    """The few-row kernel split over key chunks (and the chunk merge after it): the
    forced wait in its consumer warps gives up, the status reports it, and a normal
    call afterwards matches the oracle."""
    x = inputs.make_inputs(1, 2, 1, 4096, 128, 128, "none", seed=5200)
    Q, K, V = x.Q.cuda(), x.K.cuda(), x.V.cuda()
    assert attn.device_status() == (attn.ATTN_OK, 0)
    attn.set_watchdog(0, 1)
    try:
        attn.attn_decode(Q, K, V, "none", None, x.scale)
        rc, detail = attn.device_status()
    finally:
        attn.set_watchdog(0, 0)
    assert rc == attn.ATTN_ERR_TIMEOUT
    assert detail & FORCED_BIT
    O, L = attn.attn_decode(Q, K, V, "none", None, x.scale)
    assert attn.device_status() == (attn.ATTN_OK, 0)
    Or, Lr = oracle.attn_fwd(x.Q, x.K, x.V, "none", None, x.scale)
    assert np.abs(O.float().cpu().numpy() - Or).max() <= 1e-2
    assert np.abs(L.cpu().numpy() - Lr).max() <= 1e-3


def test_forced_timeout_in_the_projections():
    """The projection kernel: the forced wait in its epilogue warps gives up, the MMA
    warp drains what it issued before the tensor memory is released, the status
    reports it, and a normal call afterwards matches the oracle."""
    X = inputs.make_inputs(2, 1, 160, 1, 512, 512, seed=5300).Q[:, 0].contiguous()
    W, bias = inputs.make_linear(3 * 512, 512, seed=5301, bias=True)
    Xd, Wd, bd = X.cuda(), W.cuda(), bias.cuda()
    assert attn.device_status() == (attn.ATTN_OK, 0)
    attn.set_watchdog(0, 1)
    try:
        attn.proj_heads(Xd, Wd, 8, bd, 3)
        rc, detail = attn.device_status()
    finally:
        attn.set_watchdog(0, 0)
    assert rc == attn.ATTN_ERR_TIMEOUT
    assert detail & FORCED_BIT
    outs = attn.proj_heads(Xd, Wd, 8, bd, 3)
    assert attn.device_status() == (attn.ATTN_OK, 0)
    refs = oracle.proj_heads(X, W, bias, 8, 3)
    for got, ref in zip(outs, refs):
        assert np.abs(got.float().cpu().numpy() - ref).max() <= 2e-2 * max(1.0, np.abs(ref).max())

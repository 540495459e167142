"""GPU parity of the forward with the linear distance bias ("第2章：完整的 Transformer
架构" §5.3, ALiBi) against the fp64 oracle, element by element, on seeded bf16
inputs, through the C entry points attn_fwd_alibi, attn_decode_alibi (the
few-row decoding form) and attn_bwd_alibi (its gradients).

The bias makes the nearby keys dominate a row, so rows are sharper than without
it and |O| approaches the largest |v_j|. The comparison therefore uses the
format-aware bound of the forward's stress cases: |O - O_ref| <= 1e-2 + 2^-8
(|O_ref| + A) elementwise, A = sum_j w_j |v_j| from the oracle run on |V| (2^-8 is
the unit roundoff of bf16, which rounds both the weights P and the output), the
mean error <= 1e-3 + 2^-8 mean(|O_ref| + A); LSE max-abs <= 1e-3. Outputs land in
buffers with guard bands that must come back untouched.
"""

import ctypes

import numpy as np
import pytest
import torch

from oracle import oracle
from transformer_scaled_dot_03_gb300 import attn, build, inputs

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3
BF16_U = 2.0 ** -8
GUARD = 2048
SENTINEL = -12345.0


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return attn.load()


def run_gpu(x, slopes):
    Q, K, V = x.Q.cuda(), x.K.cuda(), x.V.cuda()
    lens = x.key_lengths.cuda() if x.key_lengths is not None else None
    B, H, n, _ = Q.shape
    dv = V.shape[3]
    ob = torch.full((B * H * n * dv + 2 * GUARD,), SENTINEL, dtype=torch.bfloat16, device="cuda")
    lb = torch.full((B * H * n + 2 * GUARD,), SENTINEL, dtype=torch.float32, device="cuda")
    O = ob[GUARD:GUARD + B * H * n * dv].view(B, H, n, dv)
    L = lb[GUARD:GUARD + B * H * n].view(B, H, n)
    attn.attn_fwd_alibi(Q, K, V, slopes.cuda(), x.mask, lens, x.scale, O=O, LSE=L)
    rc, detail = attn.device_status()
    assert rc == attn.ATTN_OK, (rc, detail)
    obc, lbc = ob.cpu(), lb.cpu()
    for buf in (obc, lbc):
        assert torch.all(buf[:GUARD] == SENTINEL) and torch.all(buf[-GUARD:] == SENTINEL), "guard band overwritten"
    return O.float().cpu().numpy(), L.cpu().numpy()


def compare(O, L, Or, Lr, A, label):
    O = O.reshape(Or.shape)
    L = L.reshape(Lr.shape)
    assert np.all(np.isfinite(O)), f"{label}: non-finite O"
    err = np.abs(O - Or)
    excess = err - (O_MAX + BF16_U * (np.abs(Or) + A))
    assert excess.max() <= 0, f"{label}: O error over the bound by {excess.max():.3e}"
    assert err.mean() <= O_MEAN + BF16_U * (np.abs(Or) + A).mean(), f"{label}: O mean-abs {err.mean():.3e}"
    empty = np.isneginf(Lr)
    assert np.array_equal(np.isneginf(L), empty), f"{label}: -inf LSE pattern differs"
    if (~empty).any():
        assert np.all(np.isfinite(L[~empty])), f"{label}: non-finite LSE"
        lerr = np.abs(L[~empty] - Lr[~empty]).max()
        assert lerr <= LSE_MAX, f"{label}: LSE max-abs {lerr:.3e}"


def check_full(x, slopes, label):
    O, L = run_gpu(x, slopes)
    Or, Lr = oracle.attn_fwd(x.Q, x.K, x.V, x.mask, x.key_lengths, x.scale, slopes=slopes)
    A, _ = oracle.attn_fwd(x.Q, x.K, x.V.abs(), x.mask, x.key_lengths, x.scale, slopes=slopes)
    compare(O, L, Or, Lr, A, label)


# ------------------------------------------------------------------ seeded workloads

@pytest.mark.parametrize("name", ["alibi_decoder_causal", "alibi_long_causal"])
def test_workload_every_row(name):
    """Full-size workload in the benchmark's launch configuration, compared with the
    oracle on every row (the oracle runs on all host cores)."""
    w = inputs.WORKLOADS[name]
    x = inputs.workload_inputs(w)
    slopes = inputs.alibi_slopes(w.H)
    O, L = run_gpu(x, slopes)
    t = oracle.default_threads()
    Or, Lr = oracle.attn_fwd(x.Q, x.K, x.V, x.mask, x.key_lengths, x.scale, slopes=slopes, threads=t)
    A, _ = oracle.attn_fwd(x.Q, x.K, x.V.abs(), x.mask, x.key_lengths, x.scale, slopes=slopes, threads=t)
    compare(O, L, Or, Lr, A, name)


# ------------------------------------------------------------------ shapes, masks, slopes

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mask,n,m", [("none", 200, 200), ("none", 100, 333), ("none", 257, 64),
                                      ("causal", 300, 300), ("causal", 129, 400), ("causal", 300, 130),
                                      ("key_padding", 150, 300), ("causal_key_padding", 260, 260)])
def test_shapes_and_masks(d, mask, n, m):
    lens = [m, max(1, m // 3), 1] if mask in inputs.LENGTH_MASKS else None
    B = 3 if lens else 2
    x = inputs.make_inputs(B, 4, n, m, d, d, mask, seed=5000 + n + m + d, key_lengths=lens)
    check_full(x, inputs.alibi_slopes(4), f"{mask} n={n} m={m} d={d}")


def test_slope_range():
    """Zero, tiny, steep and negative slopes in one call (one per head)."""
    x = inputs.make_inputs(2, 5, 300, 300, 64, 64, "none", seed=5100)
    slopes = torch.tensor([0.0, 1e-4, 2.0, -0.03, 0.5], dtype=torch.float32)
    check_full(x, slopes, "slope range")


@pytest.mark.parametrize("dk,dv", [(64, 128), (128, 64)])
def test_mixed_head_dims(dk, dv):
    x = inputs.make_inputs(3, 4, 200, 330, dk, dv, "causal_key_padding", seed=5600 + dk, key_lengths=[330, 200, 9])
    check_full(x, inputs.alibi_slopes(4), f"bias d_k={dk} d_v={dv}")
    # its decoding form and its backward
    xd = inputs.make_inputs(2, 4, 3, 2000, dk, dv, "causal", seed=5601 + dk)
    slopes = inputs.alibi_slopes(4)
    O, L = run_decode(xd, slopes)
    Or, Lr = oracle.attn_fwd(xd.Q, xd.K, xd.V, xd.mask, None, xd.scale, slopes=slopes)
    A, _ = oracle.attn_fwd(xd.Q, xd.K, xd.V.abs(), xd.mask, None, xd.scale, slopes=slopes)
    compare(O, L, Or, Lr, A, f"bias decode d_k={dk} d_v={dv}")
    check_bwd(x, slopes, f"bias backward d_k={dk} d_v={dv}")


def test_zero_slopes_match_attn_fwd():
    x = inputs.make_inputs(2, 3, 200, 200, 128, 128, "causal", seed=5200)
    O, L = run_gpu(x, torch.zeros(3))
    O0, L0 = attn.attn_fwd(x.Q.cuda(), x.K.cuda(), x.V.cuda(), "causal", None, x.scale)
    assert np.abs(O - O0.float().cpu().numpy()).max() <= 1e-2
    assert np.abs(L - L0.cpu().numpy()).max() <= 1e-4


def test_rejected_arguments():
    lib = attn.load()
    q = torch.zeros(1, 2, 4, 64, dtype=torch.bfloat16, device="cuda")
    q2 = torch.zeros(1, 2, 4, 128, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(q2)
    sl = torch.zeros(2, device="cuda")
    vp = ctypes.c_void_p
    stream = vp(torch.cuda.current_stream().cuda_stream)
    # no slopes
    rc = lib.attn_fwd_alibi(vp(q.data_ptr()), vp(q.data_ptr()), vp(q.data_ptr()), 1, 2, 4, 4, 64, 64, 0, None, None,
                            ctypes.c_float(-1.0), vp(o.data_ptr()), None, stream)
    assert rc == attn.ATTN_ERR_INVALID_ARG
    # a head dim outside {64, 128}
    rc = lib.attn_fwd_alibi(vp(q.data_ptr()), vp(q.data_ptr()), vp(q2.data_ptr()), 1, 2, 4, 4, 64, 96, 0, None,
                            vp(sl.data_ptr()), ctypes.c_float(-1.0), vp(o.data_ptr()), None, stream)
    assert rc == attn.ATTN_ERR_UNSUPPORTED
    # misaligned slopes
    rc = lib.attn_fwd_alibi(vp(q.data_ptr()), vp(q.data_ptr()), vp(q.data_ptr()), 1, 2, 4, 4, 64, 64, 0, None,
                            vp(sl.data_ptr() + 2), ctypes.c_float(-1.0), vp(o.data_ptr()), None, stream)
    assert rc == attn.ATTN_ERR_MISALIGNED


# ------------------------------------------------------------------ decoding (attn_decode_alibi)

def run_decode(x, slopes):
    Q, K, V = x.Q.cuda(), x.K.cuda(), x.V.cuda()
    lens = x.key_lengths.cuda() if x.key_lengths is not None else None
    O, L = attn.attn_decode(Q, K, V, x.mask, lens, x.scale, slopes=slopes.cuda())
    rc, detail = attn.device_status()
    assert rc == attn.ATTN_OK, (rc, detail)
    return O.float().cpu().numpy(), L.cpu().numpy()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mask,n,m", [("none", 1, 4097), ("none", 8, 129), ("causal", 4, 1000),
                                      ("causal", 8, 5), ("key_padding", 1, 3000),
                                      ("causal_key_padding", 3, 2100)])
def test_decode(d, mask, n, m):
    """Few query rows against a long key sequence (one and several key chunks per head)."""
    lens = [m, m // 2 + 1, 1] if mask in inputs.LENGTH_MASKS else None
    B = 3 if lens else 2
    x = inputs.make_inputs(B, 4, n, m, d, d, mask, seed=5300 + n + m + d, key_lengths=lens)
    slopes = inputs.alibi_slopes(4)
    O, L = run_decode(x, slopes)
    Or, Lr = oracle.attn_fwd(x.Q, x.K, x.V, x.mask, x.key_lengths, x.scale, slopes=slopes)
    A, _ = oracle.attn_fwd(x.Q, x.K, x.V.abs(), x.mask, x.key_lengths, x.scale, slopes=slopes)
    compare(O, L, Or, Lr, A, f"decode {mask} n={n} m={m} d={d}")


def test_decode_matches_forward():
    """The decoding form gives the forward's result for the same rows."""
    x = inputs.make_inputs(2, 8, 4, 2000, 128, 128, "causal", seed=5400)
    slopes = inputs.alibi_slopes(8)
    O, L = run_decode(x, slopes)
    Of, Lf = run_gpu(x, slopes)
    assert np.abs(O - Of).max() <= 2e-2
    assert np.abs(L - Lf).max() <= 1e-3


def test_decode_rejects_null_slopes():
    lib = attn.load()
    q = torch.zeros(1, 1, 1, 64, dtype=torch.bfloat16, device="cuda")
    vp = ctypes.c_void_p
    rc = lib.attn_decode_alibi(vp(q.data_ptr()), vp(q.data_ptr()), vp(q.data_ptr()), 1, 1, 1, 1, 64, 64, 0, None,
                               None, ctypes.c_float(-1.0), vp(q.data_ptr()), None, None, ctypes.c_size_t(0),
                               vp(torch.cuda.current_stream().cuda_stream))
    assert rc == attn.ATTN_ERR_INVALID_ARG


# ------------------------------------------------------------------ backward (attn_bwd_alibi)
#
# The GPU differentiates from its own biased forward (bf16 O, fp32 LSE); the bound
# is the backward's (tests/test_bwd_parity.py) with the weights of the biased
# scores: |G - G_ref| <= 2 bound + 1e-6 elementwise, u = 2^-8,
#   dV: u |dV_ref| + u Wᵀ|dO|;  dK: u |dK_ref| + scale Tᵀ|Q|;  dQ: u |dQ_ref| + scale T|K|,
#   T = W (u |dP - D| + E),  E_i = u sum_c |dO_ic| (|O_ic| + A_ic).

def check_bwd(x, slopes, label):
    B, H, n, d = x.Q.shape
    dO = inputs.make_grad_output(B, H, n, x.V.shape[3], seed=77)
    Q, K, V, g, sl = x.Q.cuda(), x.K.cuda(), x.V.cuda(), dO.cuda(), slopes.cuda()
    lens = x.key_lengths.cuda() if x.key_lengths is not None else None
    O, LSE = attn.attn_fwd_alibi(Q, K, V, sl, x.mask, lens, x.scale)
    got = attn.attn_bwd(Q, K, V, O, LSE, g, x.mask, lens, x.scale, slopes=sl)
    rc, detail = attn.device_status()
    assert rc == attn.ATTN_OK, (rc, detail)
    got = [t.float().cpu().numpy() for t in got]
    refs = oracle.attn_bwd(x.Q, x.K, x.V, dO, x.mask, x.key_lengths, x.scale, slopes=slopes)
    Qd, Kd, Vd, gd = (t.double().numpy() for t in (x.Q, x.K, x.V, dO))
    Or, _, W = oracle.attn_fwd(x.Q, x.K, x.V, x.mask, x.key_lengths, x.scale, slopes=slopes, weights=True)
    A, _ = oracle.attn_fwd(x.Q, x.K, x.V.abs(), x.mask, x.key_lengths, x.scale, slopes=slopes)
    dP = np.einsum("bhic,bhjc->bhij", gd, Vd)
    D = np.sum(gd * Or, axis=-1)
    E = BF16_U * np.sum(np.abs(gd) * (np.abs(Or) + A), axis=-1)
    T = W * (BF16_U * np.abs(dP - D[..., None]) + E[..., None])
    dQr, dKr, dVr = refs
    bds = (BF16_U * np.abs(dQr) + x.scale * np.einsum("bhij,bhjc->bhic", T, np.abs(Kd)),
           BF16_U * np.abs(dKr) + x.scale * np.einsum("bhij,bhic->bhjc", T, np.abs(Qd)),
           BF16_U * np.abs(dVr) + BF16_U * np.einsum("bhij,bhic->bhjc", W, np.abs(gd)))
    for name, G, R, bd in zip(("dQ", "dK", "dV"), got, refs, bds):
        assert np.all(np.isfinite(G)), f"{label}: non-finite {name}"
        excess = np.abs(G - R) - (2 * bd + 1e-6)
        assert excess.max() <= 0, f"{label}: {name} exceeds its bound by {excess.max():.3e}"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mask,n,m", [("none", 200, 200), ("causal", 256, 256), ("causal", 130, 300),
                                      ("key_padding", 150, 260), ("causal_key_padding", 200, 200)])
def test_bwd(d, mask, n, m):
    lens = [m, m // 2, 1] if mask in inputs.LENGTH_MASKS else None
    B = 3 if lens else 2
    x = inputs.make_inputs(B, 4, n, m, d, d, mask, seed=5500 + n + m + d, key_lengths=lens)
    check_bwd(x, inputs.alibi_slopes(4), f"bwd {mask} n={n} m={m} d={d}")


def test_bwd_rejects_null_slopes():
    lib = attn.load()
    q = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 4, device="cuda")
    vp = ctypes.c_void_p
    rc = lib.attn_bwd_alibi(vp(q.data_ptr()), vp(q.data_ptr()), vp(q.data_ptr()), vp(q.data_ptr()), vp(q.data_ptr()),
                            vp(lse.data_ptr()), 1, 1, 4, 4, 64, 64, 0, None, None, ctypes.c_float(-1.0),
                            vp(q.data_ptr()), vp(q.data_ptr()), vp(q.data_ptr()), None, ctypes.c_size_t(0),
                            vp(torch.cuda.current_stream().cuda_stream))
    assert rc == attn.ATTN_ERR_INVALID_ARG

"""GPU parity of the attention backward (dQ, dK, dV) against the fp64 CPU oracle.

The GPU runs its own forward first (O in bf16, LSE in fp32) and differentiates
from those, as a training step would; the oracle differentiates the exact
function of the same bf16 inputs. Tolerance, derived from the path's roundings
(every other error source is below 2^-18 relative): for each gradient G,
elementwise |G - G_ref| <= 2 * bound + 1e-6 with

  dV: bound = u |dV_ref| + u (Wᵀ |dO|)              (bf16 output; bf16 P)
  dK: bound = u |dK_ref| + scale * Tᵀ |Q|
  dQ: bound = u |dQ_ref| + scale * T |K|
      T_ij  = W_ij (u |dP_ij - D_i| + E_i)           (bf16 dS; D from the bf16 O)
      E_i   = u sum_c |dO_ic| (|O_ic| + A_ic)        (the forward's O error)
      u     = 2^-8, the unit roundoff of bf16 (8-bit significand)

where W are the oracle's weights, dP = dO Vᵀ, D_i = dO_i . O_i, and A = the
oracle's output on |V| (the sum of w_j |v_j| that bounds the forward's P
rounding). The factor 2 covers the first-order derivation.
"""

import numpy as np
import pytest
import torch

from oracle import oracle
from transformer_scaled_dot_03_gb300 import attn, build, inputs

pytestmark = pytest.mark.gpu

U = 2.0 ** -8          # unit roundoff of bf16 (8-bit significand)


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return attn.load()


def run_gpu_bwd(x: inputs.Inputs, dO: torch.Tensor):
    Q, K, V, g = x.Q.cuda(), x.K.cuda(), x.V.cuda(), dO.cuda()
    lens = x.key_lengths.cuda() if x.key_lengths is not None else None
    O, LSE = attn.attn_fwd(Q, K, V, x.mask, lens, x.scale)
    dQ, dK, dV = attn.attn_bwd(Q, K, V, O, LSE, g, x.mask, lens, x.scale)
    rc, detail = attn.device_status()
    assert rc == attn.ATTN_OK, (rc, detail)
    torch.cuda.synchronize()
    return tuple(t.float().cpu().numpy() for t in (dQ, dK, dV))


def bounds(x: inputs.Inputs, dO: torch.Tensor, refs):
    Qd, Kd, Vd, g = (t.double().numpy() for t in (x.Q, x.K, x.V, dO))
    Or, _, W = oracle.attn_fwd(x.Q, x.K, x.V, x.mask, x.key_lengths, x.scale, weights=True)
    A, _ = oracle.attn_fwd(x.Q, x.K, x.V.abs(), x.mask, x.key_lengths, x.scale)
    dP = np.einsum("bhic,bhjc->bhij", g, Vd, optimize=True)
    D = np.sum(g * Or, axis=-1)
    E = U * np.sum(np.abs(g) * (np.abs(Or) + A), axis=-1)
    T = W * (U * np.abs(dP - D[..., None]) + E[..., None])
    dQr, dKr, dVr = refs
    bq = U * np.abs(dQr) + x.scale * np.einsum("bhij,bhjc->bhic", T, np.abs(Kd), optimize=True)
    bk = U * np.abs(dKr) + x.scale * np.einsum("bhij,bhic->bhjc", T, np.abs(Qd), optimize=True)
    bv = U * np.abs(dVr) + U * np.einsum("bhij,bhic->bhjc", W, np.abs(g), optimize=True)
    return bq, bk, bv


def check_bwd(x: inputs.Inputs, dO: torch.Tensor, label=""):
    got = run_gpu_bwd(x, dO)
    refs = oracle.attn_bwd(x.Q, x.K, x.V, dO, x.mask, x.key_lengths, x.scale)
    for name, G, R, bd in zip(("dQ", "dK", "dV"), got, refs, bounds(x, dO, refs)):
        assert np.all(np.isfinite(G)), f"{label}: non-finite {name}"
        excess = np.abs(G - R) - (2 * bd + 1e-6)
        worst = np.unravel_index(np.argmax(excess), excess.shape)
        assert excess.max() <= 0, (f"{label}: {name} exceeds its bound by {excess.max():.3e} at {worst} "
                                   f"(got {G[worst]:.5f}, ref {R[worst]:.5f}, bound {2 * bd[worst]:.2e})")
    return got, refs


def case(B, H, n, m, d, mask, seed, lens=None, value_scale=1.0):
    x = inputs.make_inputs(B, H, n, m, d, d, mask, seed=seed, key_lengths=lens, value_scale=value_scale)
    dO = inputs.make_grad_output(B, H, n, d, seed=seed + 1)
    return x, dO


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mask,n,m,lens", [
    ("none", 200, 200, None),
    ("none", 1, 300, None),
    ("none", 300, 77, None),
    ("causal", 256, 256, None),
    ("causal", 130, 300, None),
    ("causal", 300, 130, None),
    ("key_padding", 150, 260, [260, 1, 0, 129]),
    ("causal_key_padding", 200, 200, [200, 128, 5, 0]),
    ("causal_key_padding", 100, 333, [333, 250, 234, 1]),
])
def test_bwd_matches_oracle(d, mask, n, m, lens):
    B = len(lens) if lens else 2
    x, dO = case(B, 2, n, m, d, mask, seed=8000 + n + m + d, lens=lens)
    check_bwd(x, dO, f"{mask} n={n} m={m} d={d}")


@pytest.mark.parametrize("dk,dv", [(64, 128), (128, 64)])
@pytest.mark.parametrize("mask,n,m,lens", [
    ("none", 200, 200, None),
    ("causal", 256, 256, None),
    ("causal", 130, 300, None),
    ("key_padding", 150, 260, [260, 1, 0, 129]),
    ("causal_key_padding", 100, 333, [333, 250, 234, 1]),
])
def test_bwd_mixed_head_dims(dk, dv, mask, n, m, lens):
    """Value heads of another width than the query/key heads."""
    B = len(lens) if lens else 2
    x = inputs.make_inputs(B, 2, n, m, dk, dv, mask, seed=8500 + n + m + dk, key_lengths=lens)
    dO = inputs.make_grad_output(B, 2, n, dv, seed=8501 + n + m + dk)
    check_bwd(x, dO, f"{mask} n={n} m={m} d_k={dk} d_v={dv}")


def test_bwd_big_decoder_small_batch():
    """Big-decoder sizes (n = m = 1024, d 64, causal) on 2 x 4 heads, every element."""
    x, dO = case(2, 4, 1024, 1024, 64, "causal", seed=8100)
    check_bwd(x, dO, "big decoder")


def test_bwd_long_d128_small_batch():
    """d 128, n = m = 2048, causal, x0.5 inputs (the long-context recipe), 1 x 2 heads."""
    x, dO = case(1, 2, 2048, 2048, 128, "causal", seed=8200, value_scale=0.5)
    check_bwd(x, dO, "long d128")


@pytest.mark.parametrize("mask,B,H,n,m,lens", [
    ("causal", 3, 64, 256, 256, None),
    ("key_padding", 4, 40, 200, 300, [300, 129, 0, 64]),
    ("none", 3, 64, 64, 256, None),
])
def test_bwd_d128_many_items_per_cta(mask, B, H, n, m, lens):
    """More work items (128-key tiles) than SMs at d = 128, so that the persistent
    CTAs move from one item to the next (new keys, dV and dK read out and restarted);
    with n = 64 every item is a single 64-query step."""
    x, dO = case(B, H, n, m, 128, mask, seed=8600 + n + H, lens=lens)
    check_bwd(x, dO, f"d128 items {mask}")


def test_bwd_sharp_rows():
    """Q and K scaled by 8: nearly one-hot rows, large dS spread."""
    x, dO = case(2, 2, 256, 384, 64, "key_padding", seed=8300, lens=[384, 200])
    x.Q = (x.Q.float() * 8).to(torch.bfloat16)
    x.K = (x.K.float() * 8).to(torch.bfloat16)
    check_bwd(x, dO, "sharp")


def test_bwd_full_size_every_head():
    """Big-decoder workload at full size (16 x 16 heads, n = m = 1024) under the
    decoder target mask, in one launch: the softmax identities hold on the GPU's
    gradients for every head (dK sums to zero over the keys of a head; dV sums to the
    dO of the rows that see a key), and every element of dQ, dK and dV of every head
    matches the oracle within the bound (the oracle runs four heads at a time)."""
    B, H, n, d = 16, 16, 1024, 64
    x = inputs.make_inputs(B, H, n, n, d, d, "causal_key_padding", seed=8400, len_lo=512, len_hi=n)
    dO = inputs.make_grad_output(B, H, n, d, seed=8401)
    dQ, dK, dV = run_gpu_bwd(x, dO)
    for G in (dQ, dK, dV):
        assert np.all(np.isfinite(G))
    g = dO.double().numpy()
    # dK: the column sums cancel; compare against the sum of magnitudes it cancels from
    scale_k = np.abs(dK).sum(axis=2)
    assert np.all(np.abs(dK.sum(axis=2)) <= 2.0 ** -6 * scale_k + 1e-3)
    dv_sum = dV.sum(axis=2)
    np.testing.assert_allclose(dv_sum, g.sum(axis=2), atol=2.0 ** -6 * np.abs(g).sum(axis=2).max())
    for b in range(B):
        for h0 in range(0, H, 4):
            hs = slice(h0, h0 + 4)
            xs = inputs.Inputs(x.Q[b:b + 1, hs].contiguous(), x.K[b:b + 1, hs].contiguous(),
                               x.V[b:b + 1, hs].contiguous(), x.key_lengths[b:b + 1].clone(), x.mask, x.scale)
            gs = dO[b:b + 1, hs].contiguous()
            refs = oracle.attn_bwd(xs.Q, xs.K, xs.V, gs, xs.mask, xs.key_lengths, xs.scale)
            for name, G, R, bd in zip(("dQ", "dK", "dV"), (dQ[b:b + 1, hs], dK[b:b + 1, hs], dV[b:b + 1, hs]),
                                      refs, bounds(xs, gs, refs)):
                assert np.all(np.abs(G - R) <= 2 * bd + 1e-6), (name, b, h0)


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128)])
@pytest.mark.parametrize("mask,n,m,lens", [
    ("causal", 300, 130, None),                     # rows 0..169 see no key
    ("key_padding", 97, 200, [200, 0, 33]),         # an entry without keys; 97 = 3 * 32 + 1 rows
    ("causal_cache", 70, 300, [300, 70, 150, 0]),   # the queries end each entry's filled cache
])
def test_bwd_every_output_written(dk, dv, mask, n, m, lens):
    """Outputs pre-filled with NaN and a workspace of 0xFF bytes, used for two calls:
    every element of dQ, dK and dV is written (rows that no key tile adds to, the
    partial last 32-row group), whatever the workspace held on entry, and both calls
    match the oracle."""
    B, H = (len(lens) if lens else 2), 2
    x = inputs.make_inputs(B, H, n, m, dk, dv, mask, seed=8700 + n + dk + dv, key_lengths=lens)
    dO = inputs.make_grad_output(B, H, n, dv, seed=8701 + n)
    Q, K, V, g = x.Q.cuda(), x.K.cuda(), x.V.cuda(), dO.cuda()
    lens_d = x.key_lengths.cuda() if x.key_lengths is not None else None
    O, LSE = attn.attn_fwd(Q, K, V, x.mask, lens_d, x.scale)
    ws = torch.full((attn.bwd_workspace_size(B, H, n, m, dk, dv),), 255, dtype=torch.uint8, device="cuda")
    refs = oracle.attn_bwd(x.Q, x.K, x.V, dO, x.mask, x.key_lengths, x.scale)
    bds = bounds(x, dO, refs)
    for call in range(2):
        outs = [torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
                for shape in ((B, H, n, dk), (B, H, m, dk), (B, H, m, dv))]
        attn.attn_bwd(Q, K, V, O, LSE, g, x.mask, lens_d, x.scale, *outs, workspace=ws)
        rc, detail = attn.device_status()
        assert rc == attn.ATTN_OK, (rc, detail)
        for name, G, R, bd in zip(("dQ", "dK", "dV"), outs, refs, bds):
            G = G.float().cpu().numpy()
            assert np.all(np.isfinite(G)), f"call {call}: {name} has unwritten elements"
            assert np.all(np.abs(G - R) <= 2 * bd + 1e-6), f"call {call}: {name}"


def test_bwd_dk_dv_deterministic():
    x, dO = case(2, 3, 300, 300, 64, "causal", seed=8500)
    a = run_gpu_bwd(x, dO)
    b = run_gpu_bwd(x, dO)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    assert np.max(np.abs(a[0] - b[0])) <= 2.0 ** -7 * max(1.0, float(np.abs(a[0]).max()))

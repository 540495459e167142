"""Pins of the fp64 CPU oracle against what the pages and the mathematics fix.

Every pin is a function ``pin_*(plant)`` that raises AssertionError on a
mismatch. The tests run each pin on the shipped oracle (plant 0), and then
rebuild the oracle with each planted mistake (a dropped scale, a wrong causal
boundary, a wrong K index, a missing max shift in the LSE, padding applied to
queries, a dropped key, a causal diagonal not shifted for n != m, a union in
place of the intersection of the two masks) and require that at least one pin
catches it.
"""

import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import oracle
from transformer_scaled_dot_03_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = np.array([float(v) for v in vals])
    return out


def rnd(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g, dtype=torch.float64) * scale).numpy()


# --------------------------------------------------------------------------- pins

def pin_worked_example(plant=0):
    """"从 RNN 到 Transformer（二）" §4.3: the 4-token example, the 4th token's output."""
    g = read_golden("worked_example_4token.txt")
    K = np.stack([g["K0"], g["K1"], g["K2"], g["K3"]])[None, None]
    V = np.stack([g["V0"], g["V1"], g["V2"], g["V3"]])[None, None]
    q = g["q"][None, None, None]
    O, L, W = oracle.attn_fwd(q, K, V, "none", weights=True, plant=plant)
    tol = g["tol"][0]
    np.testing.assert_allclose(W[0, 0, 0], g["weights"], atol=tol)
    np.testing.assert_allclose(O[0, 0, 0], g["output"], atol=tol)
    # LSE = ln Z; the page's Z is a sum of exps rounded to two decimals
    assert abs(math.exp(L[0, 0, 0]) - g["Z"][0]) <= g["tol_Z"][0]
    # the page's raw dot products are exact: with scale 1 the log-weight gaps equal them
    _, _, W1 = oracle.attn_fwd(q, K, V, "none", scale=1.0, weights=True, plant=plant)
    gaps = np.log(W1[0, 0, 0]) - np.log(W1[0, 0, 0, 0])
    np.testing.assert_allclose(gaps, g["dots"] - g["dots"][0], atol=1e-12)
    # and with the default 1/sqrt(d_k) the gaps are the page's scaled scores (2 decimals)
    gaps2 = np.log(W[0, 0, 0]) - np.log(W[0, 0, 0, 0])
    np.testing.assert_allclose(gaps2, g["scaled"] - g["scaled"][0], atol=tol)


def pin_causal_3x3(plant=0):
    """"第2章：完整的 Transformer 架构" §6: masked scores and their softmax (Q=I, K=Sᵀ, V=I)."""
    g = read_golden("causal_3x3.txt")
    S = np.stack([g["scores_row0"], g["scores_row1"], g["scores_row2"]])
    Q = np.eye(3)[None, None]
    K = S.T.copy()[None, None]
    V = np.eye(3)[None, None]
    O, L = oracle.attn_fwd(Q, K, V, "causal", scale=1.0, plant=plant)
    W = O[0, 0]                      # V = I, so O is the weight matrix
    tol = g["tol"][0]
    np.testing.assert_allclose(W[0], g["weights_row0"], atol=tol)
    np.testing.assert_allclose(W[1], g["weights_row1"], atol=tol)
    # row 2 is misprinted on the page; pin it to the library softmax of its scores
    np.testing.assert_allclose(W[2], scipy.special.softmax(g["scores_row2"]), atol=1e-12)
    assert np.max(np.abs(W[2] - g["row2_printed_misprint"])) > 0.02
    # LSE: one visible key gives the score itself; else the library logsumexp
    assert abs(L[0, 0, 0] - S[0, 0]) < 1e-12
    assert abs(L[0, 0, 1] - scipy.special.logsumexp(S[1, :2])) < 1e-12
    assert abs(L[0, 0, 2] - scipy.special.logsumexp(S[2, :3])) < 1e-12


def _mask_cases():
    return [("none", 5, 7, None), ("causal", 6, 6, None), ("key_padding", 4, 9, [3, 9])]


def pin_rows_sum_to_one(plant=0):
    """Each weight row sums to 1 ("Transformer 详解" §4.1 step 5): V = 1 gives O = 1."""
    for mask, n, m, lens in _mask_cases():
        B = 2
        Q, K = rnd((B, 3, n, 8), 1), rnd((B, 3, m, 8), 2)
        V = np.ones((B, 3, m, 5))
        O, _ = oracle.attn_fwd(Q, K, V, mask, key_lengths=lens, plant=plant)
        np.testing.assert_allclose(O, 1.0, atol=1e-12)


def pin_equal_scores_mean(plant=0):
    """Q = 0 makes every visible score equal: O_i is the mean of the visible v_j and
    LSE_i = ln |J| (weighted average with equal weights, "从 RNN 到 Transformer（二）" §4.1)."""
    B, H, n, m, d = 2, 2, 6, 6, 4
    Q = np.zeros((B, H, n, d))
    K, V = rnd((B, H, m, d), 3), rnd((B, H, m, 3), 4)
    O, L = oracle.attn_fwd(Q, K, V, "none", plant=plant)
    np.testing.assert_allclose(O, np.broadcast_to(V.mean(axis=2, keepdims=True), O.shape), atol=1e-12)
    np.testing.assert_allclose(L, math.log(m), atol=1e-12)
    O, L = oracle.attn_fwd(Q, K, V, "causal", plant=plant)
    counts = np.arange(1, n + 1)
    running = np.cumsum(V, axis=2) / counts[None, None, :, None]
    np.testing.assert_allclose(O, running, atol=1e-12)
    np.testing.assert_allclose(L, np.broadcast_to(np.log(counts), L.shape), atol=1e-12)
    lens = [2, 5]
    O, L = oracle.attn_fwd(Q, K, V, "key_padding", key_lengths=lens, plant=plant)
    for b, ln in enumerate(lens):
        np.testing.assert_allclose(O[b], np.broadcast_to(V[b, :, :ln].mean(axis=1, keepdims=True),
                                                         O[b].shape), atol=1e-12)
        np.testing.assert_allclose(L[b], math.log(ln), atol=1e-12)


def pin_causal_row0(plant=0):
    """Causal row 0 sees only key 0 ("Token 0 只看自己", "第2章" §6): o_0 = v_0, LSE_0 = s_00."""
    B, H, n, d = 2, 3, 9, 16
    Q, K, V = rnd((B, H, n, d), 5), rnd((B, H, n, d), 6), rnd((B, H, n, d), 7)
    sc = 0.3
    O, L = oracle.attn_fwd(Q, K, V, "causal", scale=sc, plant=plant)
    np.testing.assert_allclose(O[:, :, 0], V[:, :, 0], atol=1e-12)
    s00 = sc * np.einsum("bhd,bhd->bh", Q[:, :, 0], K[:, :, 0])
    np.testing.assert_allclose(L[:, :, 0], s00, atol=1e-12)


def pin_permutation(plant=0):
    """Self-attention is permutation-equivariant, f(PX) = P f(X) ("Transformer 详解" §3.6);
    a joint permutation of K and V rows changes nothing; cross-attention queries permute."""
    B, H, n, d = 1, 2, 11, 8
    Q, K, V = rnd((B, H, n, d), 8), rnd((B, H, n, d), 9), rnd((B, H, n, d), 10)
    p = np.random.default_rng(0).permutation(n)
    O, L = oracle.attn_fwd(Q, K, V, "none", plant=plant)
    Op, Lp = oracle.attn_fwd(Q[:, :, p], K[:, :, p], V[:, :, p], "none", plant=plant)
    np.testing.assert_allclose(Op, O[:, :, p], atol=1e-12)
    np.testing.assert_allclose(Lp, L[:, :, p], atol=1e-12)
    Oj, Lj = oracle.attn_fwd(Q, K[:, :, p], V[:, :, p], "none", plant=plant)
    np.testing.assert_allclose(Oj, O, atol=1e-12)
    np.testing.assert_allclose(Lj, L, atol=1e-12)
    Qc = rnd((B, H, 5, d), 11)
    pc = np.array([3, 0, 4, 1, 2])
    Oc, Lc = oracle.attn_fwd(Qc, K, V, "none", plant=plant)
    Ocp, Lcp = oracle.attn_fwd(Qc[:, :, pc], K, V, "none", plant=plant)
    np.testing.assert_allclose(Ocp, Oc[:, :, pc], atol=1e-12)
    np.testing.assert_allclose(Lcp, Lc[:, :, pc], atol=1e-12)


def pin_masked_exactly_zero(plant=0):
    """Masked weights are exactly 0 ("第2章" §6: e^-inf = 0): changing K or V at masked
    positions (even to NaN) leaves O and LSE bit-identical."""
    B, H, n, d = 2, 2, 7, 8
    Q, K, V = rnd((B, H, n, d), 12), rnd((B, H, n, d), 13), rnd((B, H, n, d), 14)
    O, L = oracle.attn_fwd(Q, K, V, "causal", plant=plant)
    for i in range(n):
        K2, V2 = K.copy(), V.copy()
        K2[:, :, i + 1:] = np.nan
        V2[:, :, i + 1:] = np.nan
        O2, L2 = oracle.attn_fwd(Q, K2, V2, "causal", plant=plant)
        assert np.array_equal(O2[:, :, i], O[:, :, i]) and np.array_equal(L2[:, :, i], L[:, :, i])
    lens = [3, 6]
    O, L = oracle.attn_fwd(Q, K, V, "key_padding", key_lengths=lens, plant=plant)
    K2, V2 = K.copy(), V.copy()
    for b, ln in enumerate(lens):
        K2[b, :, ln:] = np.nan
        V2[b, :, ln:] = 1e300
    O2, L2 = oracle.attn_fwd(Q, K2, V2, "key_padding", key_lengths=lens, plant=plant)
    assert np.array_equal(O2, O) and np.array_equal(L2, L)


def pin_fill_minus_1e9(plant=0):
    """With at least one visible key, the -1e9 fill of "Transformer 详解" §3.4 gives the
    same result as exclusion (-inf): library masked_fill + softmax + matmul in fp64."""
    B, H, n, m, d = 2, 3, 6, 10, 8
    Q, K, V = rnd((B, H, n, d), 15), rnd((B, H, m, d), 16), rnd((B, H, m, 4), 17)
    lens = [4, 10]
    O, _ = oracle.attn_fwd(Q, K, V, "key_padding", key_lengths=lens, plant=plant)
    q, k, v = map(torch.from_numpy, (Q, K, V))
    scores = torch.matmul(q, k.transpose(-1, -2)) / math.sqrt(d)
    valid = (torch.arange(m)[None, :] < torch.tensor(lens)[:, None]).view(B, 1, 1, m)
    w = torch.softmax(scores.masked_fill(~valid, -1e9), dim=-1)
    np.testing.assert_allclose(O, torch.matmul(w, v).numpy(), atol=1e-12)


def _torch_ref(Q, K, V, mask, lens, scale):
    """Library reference for cases where every row sees at least one key."""
    q, k, v = map(torch.from_numpy, (Q, K, V))
    B, H, n, d = q.shape
    m = k.shape[2]
    allowed = torch.ones(1, 1, n, m, dtype=torch.bool)
    if mask in ("causal", "causal_key_padding"):
        allowed = allowed & torch.ones(n, m, dtype=torch.bool).tril(diagonal=m - n)
    if mask in ("key_padding", "causal_key_padding"):
        allowed = allowed & (torch.arange(m)[None, :] < torch.tensor(lens)[:, None]).view(B, 1, 1, m)
    O = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=allowed, scale=scale)
    s = torch.matmul(q, k.transpose(-1, -2)) * scale
    L = torch.logsumexp(s.masked_fill(~allowed, float("-inf")), dim=-1)
    return O.numpy(), L.numpy()


def pin_library_brute_force(plant=0):
    """Tiny shapes against torch's fp64 scaled_dot_product_attention with a boolean mask and
    torch.logsumexp (library routines; cross-attention n != m included)."""
    cases = [
        (1, 1, 1, 1, 2, 2, "none", None, None),
        (2, 2, 3, 16, 8, 5, "none", None, None),
        (1, 3, 16, 16, 64, 64, "causal", None, 0.125),
        (2, 2, 9, 9, 2, 3, "causal", None, None),
        (3, 1, 5, 12, 8, 8, "key_padding", [1, 12, 7], None),
        (2, 2, 16, 13, 64, 16, "key_padding", [13, 2], 0.7),
        (2, 2, 4, 11, 8, 8, "causal", None, None),
        (2, 1, 7, 7, 8, 4, "causal_key_padding", [7, 3], None),
        (3, 2, 5, 9, 16, 16, "causal_key_padding", [9, 6, 5], None),
    ]
    for t, (B, H, n, m, dk, dv, mask, lens, sc) in enumerate(cases):
        Q, K, V = rnd((B, H, n, dk), 100 + t), rnd((B, H, m, dk), 200 + t), rnd((B, H, m, dv), 300 + t)
        scale = 1.0 / math.sqrt(dk) if sc is None else sc
        O, L = oracle.attn_fwd(Q, K, V, mask, key_lengths=lens, scale=sc, plant=plant)
        Ot, Lt = _torch_ref(Q, K, V, mask, lens, scale)
        np.testing.assert_allclose(O, Ot, atol=1e-12)
        np.testing.assert_allclose(L, Lt, atol=1e-12)


def pin_two_key_logistic(plant=0):
    """Two keys with scores a and a - delta: weights are the logistic function of delta,
    also when a is far beyond exp's range (no overflow), and LSE = a + ln(1 + e^-delta)."""
    for a, delta in [(0.0, 1.5), (5000.0, 2.0), (-3000.0, 0.25)]:
        Q = np.array([[[[1.0, 0.0]]]])
        K = np.array([[[[a, 0.0], [a - delta, 0.0]]]])
        V = np.array([[[[1.0], [0.0]]]])
        O, L = oracle.attn_fwd(Q, K, V, "none", scale=1.0, plant=plant)
        assert abs(O[0, 0, 0, 0] - scipy.special.expit(delta)) < 1e-12
        assert abs(L[0, 0, 0] - (a + math.log1p(math.exp(-delta)))) < 1e-9 * max(1.0, abs(a))


def pin_causal_suffix(plant=0):
    """Causal attention of n < m queries is the last n rows of the square causal
    self-attention over all m positions ("Transformer 详解" §5.3: row i sees the keys up
    to its own position; the n queries are the last n positions). The square case is
    pinned by the page's 3x3 example and by causal row 0."""
    B, H, m, d = 2, 2, 13, 8
    Qf, K, V = rnd((B, H, m, d), 30), rnd((B, H, m, d), 31), rnd((B, H, m, 6), 32)
    Of, Lf = oracle.attn_fwd(Qf, K, V, "causal", plant=plant)
    for n in (1, 4, 12):
        O, L = oracle.attn_fwd(Qf[:, :, m - n:], K, V, "causal", plant=plant)
        np.testing.assert_allclose(O, Of[:, :, m - n:], atol=1e-12)
        np.testing.assert_allclose(L, Lf[:, :, m - n:], atol=1e-12)
    # a single query (n = 1) therefore sees every key: plain unmasked attention
    O1, L1 = oracle.attn_fwd(Qf[:, :, -1:], K, V, "causal", plant=plant)
    On, Ln = oracle.attn_fwd(Qf[:, :, -1:], K, V, "none", plant=plant)
    np.testing.assert_allclose(O1, On, atol=1e-12)
    np.testing.assert_allclose(L1, Ln, atol=1e-12)


def pin_causal_and_padding(plant=0):
    """The decoder target mask is the intersection of the padding mask and the causal mask
    ("Transformer 详解" §5.3). Row i then sees keys j <= min(i + m - n, len - 1): it equals
    the causal result while i + m - n < len and the key-padding result once
    i + m - n >= len - 1; with len = m it is the causal mask itself."""
    B, H, n, m, d = 3, 2, 9, 12, 8
    Q, K, V = rnd((B, H, n, d), 33), rnd((B, H, m, d), 34), rnd((B, H, m, 5), 35)
    lens = [12, 7, 4]
    O, L = oracle.attn_fwd(Q, K, V, "causal_key_padding", key_lengths=lens, plant=plant)
    Oc, Lc = oracle.attn_fwd(Q, K, V, "causal", plant=plant)
    Op, Lp = oracle.attn_fwd(Q, K, V, "key_padding", key_lengths=lens, plant=plant)
    off = m - n
    for b, ln in enumerate(lens):
        for i in range(n):
            if i + off < ln:
                np.testing.assert_allclose(O[b, :, i], Oc[b, :, i], atol=1e-12)
                np.testing.assert_allclose(L[b, :, i], Lc[b, :, i], atol=1e-12)
            if i + off >= ln - 1:
                np.testing.assert_allclose(O[b, :, i], Op[b, :, i], atol=1e-12)
                np.testing.assert_allclose(L[b, :, i], Lp[b, :, i], atol=1e-12)
    assert any(i + off >= ln for ln in lens for i in range(n))      # both regimes occur
    assert any(i + off < ln - 1 for ln in lens for i in range(n))


PINS = [pin_worked_example, pin_causal_3x3, pin_rows_sum_to_one, pin_equal_scores_mean,
        pin_causal_row0, pin_permutation, pin_masked_exactly_zero, pin_fill_minus_1e9,
        pin_library_brute_force, pin_two_key_logistic, pin_causal_suffix,
        pin_causal_and_padding]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(0)


@pytest.mark.parametrize("plant", [1, 2, 3, 4, 5, 6, 7, 8])
def test_planted_mistake_is_caught(plant):
    caught = []
    for pin in PINS:
        try:
            pin(plant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {plant} passed every pin"


# ------------------------------------------------------------- readings and plumbing

def test_fully_masked_row_reading():
    """Key length 0: no visible key -> O = 0 and LSE = -inf (the library's stated reading)."""
    Q, K, V = rnd((2, 1, 3, 4), 20), rnd((2, 1, 5, 4), 21), rnd((2, 1, 5, 4), 22)
    O, L = oracle.attn_fwd(Q, K, V, "key_padding", key_lengths=[0, 5])
    assert np.all(O[0] == 0.0) and np.all(np.isneginf(L[0]))
    assert np.all(np.isfinite(O[1])) and np.all(np.isfinite(L[1]))


def test_causal_rows_without_keys_reading():
    """Causal with n > m: query row i sees keys j <= i - (n - m), so the first n - m rows
    see none and get O = 0, LSE = -inf (the same reading as a zero key length)."""
    Q, K, V = rnd((1, 2, 7, 4), 36), rnd((1, 2, 3, 4), 37), rnd((1, 2, 3, 4), 38)
    O, L = oracle.attn_fwd(Q, K, V, "causal")
    assert np.all(O[:, :, :4] == 0.0) and np.all(np.isneginf(L[:, :, :4]))
    Ot, Lt = _torch_ref(Q[:, :, 4:], K, V, "causal", None, 0.5)
    np.testing.assert_allclose(O[:, :, 4:], Ot, atol=1e-12)
    np.testing.assert_allclose(L[:, :, 4:], Lt, atol=1e-12)
    O, L = oracle.attn_fwd(Q[:, :, :3], K, V, "causal_key_padding", key_lengths=[0])
    assert np.all(O == 0.0) and np.all(np.isneginf(L))


def test_key_length_clamp():
    Q, K, V = rnd((2, 1, 3, 4), 23), rnd((2, 1, 5, 4), 24), rnd((2, 1, 5, 4), 25)
    O1, L1 = oracle.attn_fwd(Q, K, V, "key_padding", key_lengths=[-4, 99])
    O2, L2 = oracle.attn_fwd(Q, K, V, "key_padding", key_lengths=[0, 5])
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_rows_match_full():
    B, H, n, m, d = 2, 3, 10, 12, 8
    Q, K, V = rnd((B, H, n, d), 26), rnd((B, H, m, d), 27), rnd((B, H, m, d), 28)
    lens = [5, 12]
    O, L = oracle.attn_fwd(Q, K, V, "key_padding", key_lengths=lens)
    rows = inputs.sample_rows(B, H, n, 17, seed=3).numpy()
    Or, Lr = oracle.attn_rows(Q, K, V, rows, "key_padding", key_lengths=lens)
    assert np.array_equal(Or, O.reshape(-1, d)[rows]) and np.array_equal(Lr, L.reshape(-1)[rows])


def test_bf16_inputs_widen_exactly():
    """The oracle reads the bf16-rounded inputs widened exactly to fp64: the worked example
    with 0.7 rounded to bf16 (0.69921875) moves the output by less than 1e-3."""
    g = read_golden("worked_example_4token.txt")
    K = torch.tensor(np.stack([g["K0"], g["K1"], g["K2"], g["K3"]])[None, None]).to(torch.bfloat16)
    V = torch.tensor(np.stack([g["V0"], g["V1"], g["V2"], g["V3"]])[None, None]).to(torch.bfloat16)
    q = torch.tensor(g["q"][None, None, None]).to(torch.bfloat16)
    assert float(K[0, 0, 2, 0]) == 0.69921875
    O, _ = oracle.attn_fwd(q, K, V, "none")
    Kx = np.stack([g["K0"], g["K1"], g["K2"], g["K3"]])[None, None]
    Oexact, _ = oracle.attn_fwd(g["q"][None, None, None], Kx, V.double().numpy(), "none")
    assert np.max(np.abs(O - Oexact)) < 1e-3


@pytest.mark.parametrize("name,d,scale_var", [("big_decoder_causal", 64, 1.0),
                                              ("long_causal", 128, 0.0625)])
def test_input_scale_statistics(name, d, scale_var):
    """Var(q.k) = d_k for i.i.d. N(0,1) components and Var(q.k/sqrt(d_k)) = 1
    ("第2章" §2.3; "从 RNN 到 Transformer（二）" §4.4); with the x0.5 long-context
    recipe the scaled variance is 0.0625. Checked on the generator's own draws."""
    w = inputs.WORKLOADS[name]
    x = inputs.make_inputs(2, 4, 512, 512, d, d, w.mask, w.seed, value_scale=w.value_scale)
    q, k = x.Q.double(), x.K.double()
    s = torch.einsum("bhid,bhjd->bhij", q[:, :, :64], k[:, :, :512]).reshape(-1)
    var_scaled = float((s * x.scale).var())
    assert abs(var_scaled / scale_var - 1.0) < 0.02
    assert abs(float(s.var()) / (d * scale_var) - 1.0) < 0.02


def test_projection_recipe_statistics():
    """Base-encoder recipe: Xavier-uniform projections keep unit variance, so the scaled
    scores again have variance close to 1 (checked loosely: the heads are correlated)."""
    x = inputs.make_projection_inputs(2, 8, 128, 512, "key_padding", 1, 256, 512)
    assert x.Q.shape == (2, 8, 128, 64) and x.key_lengths.shape == (2,)
    s = torch.einsum("bhid,bhjd->bhij", x.Q.double(), x.K.double()) * x.scale
    assert 0.8 < float(s.var()) < 1.25
    assert int(x.key_lengths.min()) >= 256 and int(x.key_lengths.max()) <= 512

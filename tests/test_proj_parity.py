"""GPU parity of the projections around the attention (QKV projection with the head
split; head merge with W_O) against the fp64 oracle.

Tolerance, derived from the arithmetic: bf16 inputs multiply exactly into fp32,
the K products are summed in fp32 (error at most about K·2^-24 of the sum of
their magnitudes; K·2^-22 is used), the bias is added in fp32, and the result is
rounded to bf16 (half an ulp: at most 2^-8 relative, bf16 keeping an 8-bit
significand). So elementwise
|G - G_ref| <= 2^-8 |G_ref| + K·2^-22·A + 1e-6, A the oracle's result on |X|, |W|
and |bias|.
"""

import numpy as np
import pytest
import torch

from oracle import oracle
from transformer_scaled_dot_03_gb300 import attn, build, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return attn.load()


def _np(t):
    return t.float().cpu().numpy()


def _abs(t):
    return None if t is None else t.abs()


def check(G, R, A, K, label):
    bound = 2.0 ** -8 * np.abs(R) + K * 2.0 ** -22 * A + 1e-6
    err = np.abs(G - R)
    assert np.all(np.isfinite(G)), label
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), f"{label}: {err[worst]:.3e} > {bound[worst]:.3e} at {worst}"


def run_proj_heads(X, W, bias, H, num_out):
    outs = attn.proj_heads(X.cuda(), W.cuda(), H, None if bias is None else bias.cuda(), num_out)
    assert attn.device_status() == (attn.ATTN_OK, 0)
    return [_np(t) for t in outs]


@pytest.mark.parametrize("B,n,d_model,H,num_out,use_bias", [
    (2, 64, 512, 8, 3, False),
    (2, 64, 512, 8, 3, True),
    (3, 96, 256, 2, 2, True),       # d = 128, 288 rows (ragged last tile)
    (1, 32, 128, 1, 1, False),      # one head of 128
    (2, 160, 192, 3, 3, True),      # N = 576: a partial 256-column tile
])
def test_proj_heads(B, n, d_model, H, num_out, use_bias):
    X = inputs.make_inputs(B, 1, n, 1, d_model, d_model, seed=10000 + n).Q[:, 0].contiguous()
    W, bias = inputs.make_linear(num_out * d_model, d_model, seed=10001 + d_model, bias=use_bias)
    got = run_proj_heads(X, W, bias, H, num_out)
    ref = oracle.proj_heads(X, W, bias, H, num_out)
    A = oracle.proj_heads(X.abs(), W.abs(), _abs(bias), H, num_out)
    for t in range(num_out):
        check(got[t], ref[t], A[t], d_model, f"proj out {t}")


@pytest.mark.parametrize("B,n,H,d,d_out,use_bias", [
    (2, 64, 8, 64, 512, False),
    (2, 64, 8, 64, 512, True),
    (3, 96, 2, 128, 256, True),
    (1, 32, 3, 64, 64, False),
    (2, 160, 4, 64, 320, True),     # N = 320: a partial tile
])
def test_merge_proj(B, n, H, d, d_out, use_bias):
    O = inputs.make_inputs(B, H, n, 1, d, d, seed=11000 + n).Q
    W, bias = inputs.make_linear(d_out, H * d, seed=11001 + d_out, bias=use_bias)
    Y = attn.merge_proj(O.cuda(), W.cuda(), None if bias is None else bias.cuda())
    assert attn.device_status() == (attn.ATTN_OK, 0)
    ref = oracle.merge_proj(O, W, bias)
    A = oracle.merge_proj(O.abs(), W.abs(), _abs(bias))
    check(_np(Y), ref, A, H * d, "merge")


def test_base_encoder_block_stagewise():
    """The base-encoder block at full size (B 32, n 512, d_model 512, h 8, key padding):
    X -> Q, K, V -> attention -> merge + W_O, every stage against the oracle applied to
    the GPU's own input for that stage (so each stage's bound applies as derived)."""
    B, n, dm, H = 32, 512, 512, 8
    x = inputs.make_inputs(B, 1, n, 1, dm, dm, "none", seed=12000).Q[:, 0].contiguous()
    W, bias = inputs.make_linear(3 * dm, dm, seed=12001, bias=True)
    Wo, bo = inputs.make_linear(dm, dm, seed=12002, bias=True)
    lens = inputs.make_inputs(B, 1, 1, n, 64, 64, "key_padding", seed=12003, len_lo=256, len_hi=n).key_lengths
    Q, K, V = attn.proj_heads(x.cuda(), W.cuda(), H, bias.cuda())
    O, L = attn.attn_fwd(Q, K, V, "key_padding", lens.cuda())
    Y = attn.merge_proj(O, Wo.cuda(), bo.cuda())
    assert attn.device_status() == (attn.ATTN_OK, 0)
    ref = oracle.proj_heads(x, W, bias, H, 3)
    A = oracle.proj_heads(x.abs(), W.abs(), bias.abs(), H, 3)
    for t, G in enumerate((Q, K, V)):
        check(_np(G), ref[t], A[t], dm, f"block proj {t}")
    Or, Lr = oracle.attn_fwd(Q.cpu(), K.cpu(), V.cpu(), "key_padding", lens, 1 / 8,
                             threads=oracle.default_threads())
    err = np.abs(_np(O) - Or)
    assert err.max() <= 1e-2 and err.mean() <= 1e-3
    assert np.max(np.abs(L.cpu().numpy() - Lr)) <= 1e-3
    Yr = oracle.merge_proj(O.cpu(), Wo, bo)
    Ay = oracle.merge_proj(O.cpu().abs(), Wo.abs(), bo.abs())
    check(_np(Y), Yr, Ay, dm, "block merge")

"""GPU parity of the few-row forward (attn_decode: n <= 8 query rows against a long
key/value sequence) against the fp64 CPU oracle, with the forward's tolerances:
O max-abs <= 1e-2 and mean-abs <= 1e-3, LSE max-abs <= 1e-3, LSE = -inf exactly
where a row sees no key. Covers one and several key chunks per (b, h) (the chunk
merge), every mask, ragged lengths and the degenerate ones (0, 1, m)."""

import numpy as np
import pytest
import torch

from oracle import oracle
from transformer_scaled_dot_03_gb300 import attn, build, inputs

from test_parity import GUARD, SENTINEL_BF16, SENTINEL_F32, compare, guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return attn.load()


def run_decode(x: inputs.Inputs):
    Q, K, V = x.Q.cuda(), x.K.cuda(), x.V.cuda()
    lens = x.key_lengths.cuda() if x.key_lengths is not None else None
    B, H, n, _ = Q.shape
    dv = V.shape[3]
    obuf, O = guarded((B, H, n, dv), torch.bfloat16, SENTINEL_BF16)
    lbuf, LSE = guarded((B, H, n), torch.float32, SENTINEL_F32)
    attn.attn_decode(Q, K, V, x.mask, lens, x.scale, O=O, LSE=LSE)
    rc, detail = attn.device_status()
    assert rc == attn.ATTN_OK, (rc, detail)
    torch.cuda.synchronize()
    ob, lb = obuf.cpu(), lbuf.cpu()
    assert torch.all(ob[:GUARD] == SENTINEL_BF16) and torch.all(ob[-GUARD:] == SENTINEL_BF16)
    assert torch.all(lb[:GUARD] == SENTINEL_F32) and torch.all(lb[-GUARD:] == SENTINEL_F32)
    return O.float().cpu().numpy(), LSE.cpu().numpy()


def check(x, label):
    O, L = run_decode(x)
    Or, Lr = oracle.attn_fwd(x.Q, x.K, x.V, x.mask, x.key_lengths, x.scale)
    return compare(O, L, Or, Lr, label, x=x)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("m", [1, 100, 129, 1000, 4097])
def test_decode_no_mask(d, n, m):
    x = inputs.make_inputs(2, 3, n, m, d, d, "none", seed=9000 + 7 * n + m + d)
    check(x, f"none n={n} m={m} d={d}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mask", ["key_padding", "causal_key_padding"])
@pytest.mark.parametrize("n", [1, 4, 8])
def test_decode_key_padding(d, mask, n):
    m = 3000
    lens = [3000, 1, 0, 129, 1024, 2999]
    x = inputs.make_inputs(len(lens), 2, n, m, d, d, mask, seed=9100 + n + d, key_lengths=lens)
    check(x, f"{mask} n={n} d={d}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n,m", [(1, 1), (3, 2), (8, 5), (8, 8), (4, 700), (7, 2049)])
def test_decode_causal(d, n, m):
    """Causal with the n rows at the end of the m keys; n > m leaves rows without keys."""
    x = inputs.make_inputs(2, 2, n, m, d, d, "causal", seed=9200 + n + m + d)
    check(x, f"causal n={n} m={m} d={d}")


@pytest.mark.parametrize("B,H,m", [(1, 1, 40000), (64, 16, 300)])
def test_decode_split_extremes(B, H, m):
    """Many chunks for one (b, h) pair; many (b, h) pairs with a single chunk."""
    x = inputs.make_inputs(B, H, 1, m, 128, 128, "none", seed=9300 + m)
    check(x, f"B={B} H={H} m={m}")


@pytest.mark.parametrize("dk,dv", [(64, 128), (128, 64)])
@pytest.mark.parametrize("mask,n,m", [("none", 1, 4097), ("causal", 8, 1000), ("key_padding", 3, 2000)])
def test_decode_mixed_head_dims(dk, dv, mask, n, m):
    """Value heads of another width than the key heads (one and several key chunks)."""
    lens = [m, m // 3, 1] if mask in inputs.LENGTH_MASKS else None
    x = inputs.make_inputs(3 if lens else 2, 4, n, m, dk, dv, mask, seed=7000 + dk + n + m, key_lengths=lens)
    check(x, f"decode {mask} n={n} m={m} d_k={dk} d_v={dv}")


def test_decode_mixed_head_dims_many_heads():
    """Enough (b, h) pairs for the tensor-core path, d_k != d_v."""
    x = inputs.make_inputs(64, 16, 2, 300, 64, 128, "none", seed=7100)
    check(x, "decode many heads d_k=64 d_v=128")


@pytest.mark.parametrize("n", [9, 16, 130])
def test_decode_more_rows(n):
    """More rows than the split kernel holds: the tensor-core kernel, few heads."""
    x = inputs.make_inputs(2, 3, n, 1500, 128, 128, "causal", seed=7200 + n)
    check(x, f"decode n={n}")


def test_decode_matches_attn_fwd():
    x = inputs.make_inputs(4, 8, 4, 2500, 64, 64, "key_padding", seed=9400, len_lo=1, len_hi=2500)
    Od, Ld = run_decode(x)
    lens = x.key_lengths.cuda()
    Of, Lf = attn.attn_fwd(x.Q.cuda(), x.K.cuda(), x.V.cuda(), x.mask, lens, x.scale)
    torch.cuda.synchronize()
    Of, Lf = Of.float().cpu().numpy(), Lf.cpu().numpy()
    assert np.max(np.abs(Od - Of)) <= 1e-2
    assert np.max(np.abs(Ld - Lf)) <= 1e-3


@pytest.mark.parametrize("name", ["decode_kv_cache", "decode_long_context", "spec_decode_cache"])
def test_decode_workloads_every_row(name):
    """The benchmark's decode workloads at full size, every row against the oracle."""
    w = inputs.WORKLOADS[name]
    x = inputs.workload_inputs(w)
    O, L = run_decode(x)
    Or, Lr = oracle.attn_fwd(x.Q, x.K, x.V, x.mask, x.key_lengths, x.scale, threads=oracle.default_threads())
    compare(O, L, Or, Lr, name, x=x)


def test_decode_m_zero():
    Q = torch.randn(2, 2, 3, 64, device="cuda").to(torch.bfloat16)
    K = torch.empty(2, 2, 0, 64, device="cuda", dtype=torch.bfloat16)
    O, L = attn.attn_decode(Q, K, K, "none")
    torch.cuda.synchronize()
    assert torch.all(O == 0) and torch.all(torch.isneginf(L))

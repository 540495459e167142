"""GPU parity of the causal mask inside a partly filled key/value cache (mask kind
4, "causal_cache": the n queries are the last n of each entry's key_lengths[b]
filled positions) against the fp64 oracle, through the forward, the few-row
decoding path, the backward and the distance-bias forward. Tolerances are those
of the respective paths (test_parity, test_bwd_parity, test_parity_alibi).
"""

import numpy as np
import pytest
import torch

from oracle import oracle
from transformer_scaled_dot_03_gb300 import attn, build, inputs

from test_bwd_parity import check_bwd
from test_parity import check_full, compare

pytestmark = pytest.mark.gpu

MASK = "causal_cache"


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return attn.load()


def lengths(B, n, m, seed):
    """Filled lengths: full, a random one, exactly n, fewer than n (rows that precede the
    filled part see nothing), one and zero."""
    g = torch.Generator().manual_seed(seed)
    pool = [m, int(torch.randint(n, m + 1, (1,), generator=g)), min(n, m), max(0, n // 2), 1, 0]
    return (pool * ((B + len(pool) - 1) // len(pool)))[:B]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n,m", [(1, 300), (7, 1000), (130, 300), (300, 300), (257, 700)])
def test_forward(d, n, m):
    x = inputs.make_inputs(6, 2, n, m, d, d, MASK, seed=6000 + n + m + d, key_lengths=lengths(6, n, m, n + m))
    check_full(x, f"forward n={n} m={m} d={d}")


def test_forward_mixed_head_dims():
    x = inputs.make_inputs(6, 2, 200, 500, 64, 128, MASK, seed=6100, key_lengths=lengths(6, 200, 500, 1))
    check_full(x, "forward d_k=64 d_v=128")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n,m", [(1, 4097), (4, 3000), (8, 129)])
def test_decode(d, n, m):
    """Speculative-style steps: n new tokens against a cache of m slots."""
    x = inputs.make_inputs(6, 4, n, m, d, d, MASK, seed=6200 + n + m + d, key_lengths=lengths(6, n, m, n * m))
    lens = x.key_lengths.cuda()
    O, L = attn.attn_decode(x.Q.cuda(), x.K.cuda(), x.V.cuda(), MASK, lens, x.scale)
    rc, detail = attn.device_status()
    assert rc == attn.ATTN_OK, (rc, detail)
    Or, Lr = oracle.attn_fwd(x.Q, x.K, x.V, MASK, x.key_lengths, x.scale)
    compare(O.float().cpu().numpy(), L.cpu().numpy(), Or, Lr, f"decode n={n} m={m} d={d}")


@pytest.mark.parametrize("d", [64, 128])
def test_backward(d):
    x = inputs.make_inputs(4, 2, 200, 330, d, d, MASK, seed=6300 + d, key_lengths=[330, 250, 200, 129])
    dO = inputs.make_grad_output(4, 2, 200, d, seed=6301 + d)
    check_bwd(x, dO, f"backward d={d}")


def test_distance_bias_uses_the_cache_position():
    """With the bias, query i sits at key position i + key_lengths[b] - n."""
    x = inputs.make_inputs(4, 4, 130, 400, 64, 64, MASK, seed=6400, key_lengths=[400, 300, 131, 60])
    slopes = inputs.alibi_slopes(4)
    O, L = attn.attn_fwd_alibi(x.Q.cuda(), x.K.cuda(), x.V.cuda(), slopes.cuda(), MASK, x.key_lengths.cuda(),
                               x.scale)
    rc, detail = attn.device_status()
    assert rc == attn.ATTN_OK, (rc, detail)
    Or, Lr = oracle.attn_fwd(x.Q, x.K, x.V, MASK, x.key_lengths, x.scale, slopes=slopes)
    A, _ = oracle.attn_fwd(x.Q, x.K, x.V.abs(), MASK, x.key_lengths, x.scale, slopes=slopes)
    compare(O.float().cpu().numpy(), L.cpu().numpy(), Or, Lr, "bias + cache", A)

"""GPU parity of the mask and shape variants against the fp64 CPU oracle:
causal masking with n != m (query row i sees keys j <= i + m - n), the combined
causal-and-key-padding mask of the decoder ("Transformer 详解" §5.3), and value
heads of another width than the query/key heads (d_k != d_v).

Same tolerances and guard bands as the base parity tests (test_parity.py).
"""

import numpy as np
import pytest
import torch

from oracle import oracle
from transformer_scaled_dot_03_gb300 import inputs

from test_parity import check_full, compare, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_scaled_dot_03_gb300 import attn, build
    build.build()
    return attn.load()


# causal with n != m: n < m is new queries against a longer key sequence (the tail of a
# prefill, a few decode steps); n > m leaves the first n - m rows without keys
CAUSAL_NM = [(1, 1), (1, 128), (1, 1000), (2, 129), (7, 300), (64, 65), (128, 1024), (129, 257),
             (300, 1000), (65, 64), (200, 64), (257, 200), (300, 129), (1000, 1)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n,m", CAUSAL_NM)
def test_causal_n_ne_m(d, n, m):
    x = inputs.make_inputs(2, 2, n, m, d, d, "causal", seed=5000 + 3 * n + m + d)
    check_full(x, f"causal n={n} m={m} d={d}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n,m,lens", [
    (150, 150, [150, 1, 0, 128, 129, 77]),
    (300, 300, [300, 200, 129, 128, 1, 0]),
    (100, 400, [400, 301, 300, 299, 0, 50]),
    (400, 100, [100, 99, 1, 0, 64, 65]),
    (1, 500, [500, 1, 0, 250]),
])
def test_causal_key_padding(d, n, m, lens):
    x = inputs.make_inputs(len(lens), 2, n, m, d, d, "causal_key_padding",
                           seed=6000 + n + m + d, key_lengths=lens)
    check_full(x, f"causal+pad n={n} m={m} lens={lens} d={d}")


@pytest.mark.parametrize("dk,dv", [(64, 128), (128, 64)])
@pytest.mark.parametrize("mask", ["none", "causal", "key_padding", "causal_key_padding"])
@pytest.mark.parametrize("n,m", [(130, 130), (257, 600), (600, 257)])
def test_dk_ne_dv(dk, dv, mask, n, m):
    x = inputs.make_inputs(3, 2, n, m, dk, dv, mask, seed=7000 + dk + n + m, len_lo=0, len_hi=m)
    check_full(x, f"{mask} dk={dk} dv={dv} n={n} m={m}")


@pytest.mark.parametrize("mask,n,m", [("causal", 200, 700), ("causal_key_padding", 384, 384),
                                      ("causal_key_padding", 150, 600)])
def test_variant_rescaling(mask, n, m):
    """Q and K scaled by 8 (sharp rows, frequent maximum raises) on the new masks."""
    x = inputs.make_inputs(2, 2, n, m, 64, 64, mask, seed=7100 + n, len_lo=100, len_hi=m)
    x.Q = (x.Q.float() * 8).to(torch.bfloat16)
    x.K = (x.K.float() * 8).to(torch.bfloat16)
    check_full(x, f"x8 {mask} n={n} m={m}", format_aware=True)


@pytest.mark.parametrize("name", ["decoder_target_mask", "prefill_continuation", "wide_values"])
def test_variant_workload_every_row(name):
    """The variant workloads at full size: the decoder target mask at big-decoder sizes
    (B 16, H 16, n = m = 1024, d 64, key lengths in [512, 1024]); 1024 new query rows
    against 8192 keys at d 128 (causal, bottom-right); value heads of 128 against key
    heads of 64. Every row against the oracle."""
    w = inputs.WORKLOADS[name]
    x = inputs.workload_inputs(w)
    O, L = run_gpu(x)
    Or, Lr = oracle.attn_fwd(x.Q, x.K, x.V, x.mask, x.key_lengths, x.scale, threads=oracle.default_threads())
    compare(O, L, Or, Lr, name, x=x)


def test_causal_suffix_on_gpu():
    """The GPU's n < m causal result equals the last n rows of its own square causal
    result over the same keys (the two runs take different tile schedules), within
    the bf16 rounding of O."""
    B, H, m, d = 2, 3, 700, 64
    x = inputs.make_inputs(B, H, m, m, d, d, "causal", seed=7400)
    Of, Lf = run_gpu(x)
    n = 333
    xs = inputs.Inputs(x.Q[:, :, m - n:].contiguous(), x.K, x.V, None, "causal", x.scale)
    Os, Ls = run_gpu(xs)
    assert np.max(np.abs(Os - Of[:, :, m - n:])) <= 2 ** -8 * max(1.0, float(np.abs(Of).max()))
    assert np.max(np.abs(Ls - Lf[:, :, m - n:])) <= 1e-5

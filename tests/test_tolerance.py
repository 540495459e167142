"""The forward's O tolerance against the bf16 format (no GPU).

The path returns O in bf16 and hands the weights P to the tensor cores in bf16,
so its error has two format terms, each first-order in the bf16 unit roundoff
u = 2^-8: the output rounding (up to u |O|) and the weight rounding (up to
u sum_j w_j |v_j|). This file emulates exactly that arithmetic in numpy (fp32
scores and exponentials, weights rounded to bf16, fp32 sums, O rounded to bf16)
on one head of the big-decoder causal workload (B 16, H 16, n = m = 1024, d 64)
and checks against the fp64 oracle that:
  - the format terms alone push an element of a row with three visible keys past
    the stated 1e-2 (so no bf16 implementation of this arithmetic meets 1e-2 on
    every element of this workload), and
  - every element stays within max(1e-2, u (|O_ref| + A)), the bound the GPU
    parity tests apply, A being the oracle's output on |V|.
"""

import numpy as np
import torch

from oracle import oracle
from transformer_scaled_dot_03_gb300 import inputs

U = 2.0 ** -8


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def test_bf16_arithmetic_needs_the_format_bound():
    w = inputs.WORKLOADS["big_decoder_causal"]
    x = inputs.workload_inputs(w)
    b, h, R = 5, 0, 64                      # the head holding the largest excess, its first 64 rows
    Q, K, V = x.Q[b:b + 1, h:h + 1, :R], x.K[b:b + 1, h:h + 1, :R], x.V[b:b + 1, h:h + 1, :R]
    Or, _ = oracle.attn_fwd(Q, K, V, "causal", None, x.scale)
    A, _ = oracle.attn_fwd(Q, K, V.abs(), "causal", None, x.scale)
    Or, A = Or[0, 0], A[0, 0]

    sl2 = np.float32(x.scale * np.log2(np.e))
    S = (Q[0, 0].double().numpy() @ K[0, 0].double().numpy().T).astype(np.float32)
    S = np.where(np.tril(np.ones((R, R), bool)), S, -np.inf).astype(np.float32)
    mx = (S.max(-1, keepdims=True) * sl2).astype(np.float32)
    p = np.exp2((S * sl2 - mx).astype(np.float32)).astype(np.float32)
    l = p.sum(-1, keepdims=True, dtype=np.float32)
    acc = (bf16(p).astype(np.float64) @ V[0, 0].double().numpy()).astype(np.float32)
    O = bf16(acc / l)

    err = np.abs(O - Or)
    assert err.max() > 1e-2                          # the stated bound is out of reach here
    i, c = np.unravel_index(err.argmax(), err.shape)
    assert i < 4 and 2.0 <= abs(Or[i, c]) < 4.0       # a row with few keys, |O| in [2, 4)
    assert np.all(err <= np.maximum(1e-2, U * (np.abs(Or) + A)))
    # with exact weights only the output rounding remains, below 1e-2
    exact = bf16((p.astype(np.float64) @ V[0, 0].double().numpy()) / l)
    assert np.abs(exact - Or).max() < 1e-2

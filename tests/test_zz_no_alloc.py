"""attn_fwd_noalloc: the attention forward for callers that may not allocate
device memory (for example code that runs while another component owns every
device allocation). It must give the same results as attn_fwd, twice in a row
(its scratch array keeps the previous call's contents), without any device
allocation. This file is collected last on purpose, so that a run stopping at
the first failure has run every other test already; it also passes alone in a
fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

from transformer_scaled_dot_03_gb300 import attn, build, inputs

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    lib = attn.load()
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_fwd_noalloc.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, f32, vp, vp, vp]
    lib.attn_fwd_noalloc.restype = i32
    return lib


def call_noalloc(lib, Q, K, V, mask, lens, scale, O, L):
    B, H, n, d = Q.shape
    m = K.shape[2]
    stream = torch.cuda.current_stream().cuda_stream
    return lib.attn_fwd_noalloc(ctypes.c_void_p(Q.data_ptr()), ctypes.c_void_p(K.data_ptr()),
                                ctypes.c_void_p(V.data_ptr()), B, H, n, m, d, V.shape[3],
                                attn.MASK_CODES[mask],
                                ctypes.c_void_p(lens.data_ptr()) if lens is not None else None,
                                ctypes.c_float(scale), ctypes.c_void_p(O.data_ptr()),
                                ctypes.c_void_p(L.data_ptr()), ctypes.c_void_p(stream))


@pytest.mark.parametrize("mask,d,n,m", [("key_padding", 64, 300, 300), ("causal", 128, 200, 200),
                                        ("none", 64, 100, 513), ("causal_key_padding", 64, 150, 400)])
def test_noalloc_matches_attn_fwd(lib, mask, d, n, m):
    x = inputs.make_inputs(2, 3, n, m, d, d, mask, seed=9100 + d + n, len_lo=1, len_hi=m)
    Q, K, V = x.Q.cuda(), x.K.cuda(), x.V.cuda()
    lens = x.key_lengths.cuda() if x.key_lengths is not None else None
    outs = [(torch.full((2, 3, n, d), 7.0, dtype=torch.bfloat16, device="cuda"),
             torch.full((2, 3, n), 7.0, dtype=torch.float32, device="cuda")) for _ in range(3)]
    # first call on this device: looks up the scratch array and loads the kernel
    assert call_noalloc(lib, Q, K, V, mask, lens, x.scale, *outs[0]) == attn.ATTN_OK
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    # two calls in a row; the second sees the array as the first left it
    for O, L in outs[1:]:
        assert call_noalloc(lib, Q, K, V, mask, lens, x.scale, O, L) == attn.ATTN_OK
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before, "device memory was allocated by attn_fwd_noalloc"

    O_ref, L_ref = attn.attn_fwd(Q, K, V, mask, lens, x.scale)
    assert attn.device_status() == (attn.ATTN_OK, 0)
    O_ref = O_ref.float().cpu().numpy()
    L_ref = L_ref.cpu().numpy()
    for O, L in outs[1:]:
        O = O.float().cpu().numpy()
        L = L.cpu().numpy()
        err = np.abs(O - O_ref)
        assert err.max() <= O_MAX and err.mean() <= O_MEAN
        empty = np.isneginf(L_ref)
        assert np.array_equal(np.isneginf(L), empty)
        assert np.all(np.abs(L[~empty] - L_ref[~empty]) <= LSE_MAX)


def test_noalloc_rejects_bad_arguments(lib):
    q = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16, device="cuda")
    O = torch.zeros_like(q)
    L = torch.zeros(1, 1, 4, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.attn_fwd_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(q.data_ptr()),
                              ctypes.c_void_p(q.data_ptr()), 1, 1, 4, 4, 64, 64,
                              attn.MASK_CODES["causal_key_padding"],
                              None, ctypes.c_float(-1.0), ctypes.c_void_p(O.data_ptr()),
                              ctypes.c_void_p(L.data_ptr()), ctypes.c_void_p(stream))
    assert rc == attn.ATTN_ERR_INVALID_ARG
    rc = lib.attn_fwd_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(q.data_ptr()),
                              ctypes.c_void_p(q.data_ptr()), 1, 1, 4, 4, 32, 32, 0, None,
                              ctypes.c_float(-1.0), ctypes.c_void_p(O.data_ptr()),
                              ctypes.c_void_p(L.data_ptr()), ctypes.c_void_p(stream))
    assert rc == attn.ATTN_ERR_UNSUPPORTED

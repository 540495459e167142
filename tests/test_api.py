"""Host-side checks of the C ABI that need no GPU: the library builds and loads,
exports every function include/attn.h declares, and rejects bad arguments with
the documented status codes before touching any device memory."""

import ctypes
import os
import re

import pytest

from transformer_scaled_dot_03_gb300 import attn, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return attn.load()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(attn_[a-z_0-9]+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_expected_api():
    assert declared_functions() == sorted(attn.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    nm = os.popen(f"nm -D --defined-only {attn.LIB_PATH}").read()
    for name in declared_functions():
        assert re.search(rf"\bT {name}\b", nm), name


def test_status_strings(lib):
    for code, name in [(0, "ATTN_OK"), (-1, "ATTN_ERR_INVALID_ARG"), (-2, "ATTN_ERR_UNSUPPORTED"),
                       (-3, "ATTN_ERR_MISALIGNED"), (-4, "ATTN_ERR_CUDA"), (-5, "ATTN_ERR_TIMEOUT")]:
        assert attn.status_string(code) == name


P = ctypes.c_void_p(0x10000)      # aligned fake addresses: never dereferenced (rejected first)
P2 = ctypes.c_void_p(0x20000)


def call(Q=P, K=P, V=P, B=1, H=1, n=4, m=4, dk=64, dv=64, mask=0, lens=None, O=P2, LSE=None):
    return attn.attn_fwd_raw(Q, K, V, B, H, n, m, dk, dv, mask, lens, -1.0, O, LSE, 0)


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(n=-3), attn.ATTN_ERR_INVALID_ARG),
    (dict(m=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(mask=5), attn.ATTN_ERR_INVALID_ARG),
    (dict(mask=4), attn.ATTN_ERR_INVALID_ARG),          # the cache mask without key lengths
    (dict(mask=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(mask=2, lens=None), attn.ATTN_ERR_INVALID_ARG),         # key padding needs lengths
    (dict(mask=3, lens=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(dk=32, dv=32), attn.ATTN_ERR_UNSUPPORTED),
    (dict(dk=64, dv=32), attn.ATTN_ERR_UNSUPPORTED),
    (dict(dk=256, dv=128), attn.ATTN_ERR_UNSUPPORTED),
    (dict(dk=96, dv=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(n=(1 << 30) + 1), attn.ATTN_ERR_UNSUPPORTED),
    (dict(m=(1 << 30) + 1, mask=1), attn.ATTN_ERR_UNSUPPORTED),
    (dict(Q=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(O=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(Q=ctypes.c_void_p(0x10008)), attn.ATTN_ERR_MISALIGNED),
    (dict(V=ctypes.c_void_p(0x10002)), attn.ATTN_ERR_MISALIGNED),
    (dict(O=ctypes.c_void_p(0x20004)), attn.ATTN_ERR_MISALIGNED),
    (dict(LSE=ctypes.c_void_p(0x30002)), attn.ATTN_ERR_MISALIGNED),
    (dict(mask=2, lens=ctypes.c_void_p(0x40001)), attn.ATTN_ERR_MISALIGNED),
])
def test_rejects_bad_arguments(lib, kw, code):
    assert call(**kw) == code


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=0), dict(n=0), dict(B=0, Q=None, O=None)])
def test_empty_problem_is_a_noop(lib, kw):
    # nothing to compute: returns OK without touching the device
    assert call(**kw) == attn.ATTN_OK


def test_binding_fails_loudly_without_gpu_tensors(lib):
    import torch
    q = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        attn.attn_fwd(q, q, q)


def test_flop_model():
    assert attn.flops(32, 8, 512, 512, 64, "key_padding") == 4.0 * 32 * 8 * 512 * 512 * 64
    assert attn.flops(16, 16, 1024, 1024, 64, "causal") == 2.0 * 16 * 16 * 1024 * 1024 * 64
    assert attn.flops(1, 1, 1024, 1024, 64, "causal_key_padding") == attn.flops(1, 1, 1024, 1024, 64,
                                                                                "causal")
    # one query against m keys sees them all (within half a pair of the exact count)
    assert abs(attn.flops(1, 1, 1, 4096, 64, "causal") - 4.0 * 64 * 4096) <= 4.0 * 64 * 0.5
    # the masked triangle's nominal area shrinks as n falls below m
    assert attn.flops(1, 1, 256, 1024, 64, "causal") == 4.0 * 64 * (256 * 1024 - 256 * 256 / 2)
    assert attn.flops(1, 1, 1024, 256, 64, "causal") == 4.0 * 64 * 256 * 256 / 2
    assert attn.flops(2, 3, 128, 96, 64, "none", d_v=128) == 2.0 * 2 * 3 * (64 + 128) * 128 * 96


def call_bwd(B=1, H=1, n=4, m=4, dk=64, dv=64, mask=0, lens=None, dQ=P2, dK=P2, dV=P2, ws=P,
             ws_bytes=1 << 20, Q=P, O=P, LSE=P):
    return attn.attn_bwd_raw(Q, P, P, O, P, LSE, B, H, n, m, dk, dv, mask, lens, -1.0, dQ, dK, dV, ws,
                             ws_bytes, 0)


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(mask=5), attn.ATTN_ERR_INVALID_ARG),
    (dict(mask=4), attn.ATTN_ERR_INVALID_ARG),          # the cache mask without key lengths
    (dict(mask=2, lens=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(mask=3, lens=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(dk=64, dv=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(dk=96, dv=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(dQ=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(dK=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(ws=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(LSE=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(ws_bytes=16), attn.ATTN_ERR_INVALID_ARG),
    (dict(ws=ctypes.c_void_p(0x10080)), attn.ATTN_ERR_MISALIGNED),
    (dict(dQ=ctypes.c_void_p(0x20008)), attn.ATTN_ERR_MISALIGNED),
    (dict(O=ctypes.c_void_p(0x20002)), attn.ATTN_ERR_MISALIGNED),
])
def test_bwd_rejects_bad_arguments(lib, kw, code):
    assert call_bwd(**kw) == code


def test_bwd_workspace_size():
    # dQ accumulator (fp32) + two fp32 vectors over 128-padded rows, each 256-byte aligned
    assert attn.bwd_workspace_size(2, 3, 100, 50, 64, 64) == 2 * 3 * 100 * 64 * 4 + 2 * 3072
    assert attn.bwd_workspace_size(0, 3, 100, 50, 64, 64) == 0
    assert attn.bwd_workspace_size(1, 1, 129, 7, 128, 128) == 129 * 128 * 4 + 2 * 1024


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=0)])
def test_bwd_empty_problem_is_a_noop(lib, kw):
    assert call_bwd(**kw) == attn.ATTN_OK


def call_dec(B=1, H=1, n=1, m=4096, dk=64, dv=64, mask=0, lens=None, O=P2, ws=P, ws_bytes=1 << 24):
    return attn.attn_decode_raw(P, P, P, B, H, n, m, dk, dv, mask, lens, -1.0, O, None, ws, ws_bytes, 0)


@pytest.mark.parametrize("kw,code", [
    (dict(dk=64, dv=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(dk=32, dv=32), attn.ATTN_ERR_UNSUPPORTED),
    (dict(mask=2, lens=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(mask=5), attn.ATTN_ERR_INVALID_ARG),
    (dict(O=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(ws=None), attn.ATTN_ERR_INVALID_ARG),          # this size splits the keys
    (dict(ws_bytes=64), attn.ATTN_ERR_INVALID_ARG),
    (dict(ws=ctypes.c_void_p(0x10040)), attn.ATTN_ERR_MISALIGNED),
])
def test_decode_rejects_bad_arguments(lib, kw, code):
    assert call_dec(**kw) == code


def test_decode_workspace_size():
    # one (b, h) pair with 4096 keys: split into 16 chunks of 256 keys
    assert attn.decode_workspace_size(1, 1, 1, 4096, 64, 64) == 16 * 64 * 4 + 256
    # 2048 or more (b, h) pairs: never split, no workspace
    assert attn.decode_workspace_size(128, 16, 1, 4096, 128, 128) == 0
    # sized for the largest chunk count a launch may pick: min(ceil(m/256), ceil(2048/(B*H)))
    assert attn.decode_workspace_size(40, 16, 2, 4096, 128, 128) == 640 * 4 * 2 * 128 * 4 + 640 * 4 * 2 * 8
    assert attn.decode_workspace_size(0, 16, 1, 4096, 128, 128) == 0
    # more than 8 rows run the tensor-core kernel: no workspace
    assert attn.decode_workspace_size(1, 1, 9, 4096, 64, 64) == 0
    # the partial outputs have the value head dim
    assert attn.decode_workspace_size(1, 1, 1, 4096, 128, 64) == 16 * 64 * 4 + 256
    assert attn.decode_workspace_size(1, 1, 1, 4096, 64, 128) == 16 * 128 * 4 + 256


@pytest.mark.parametrize("kw", [dict(B=0), dict(n=0)])
def test_decode_empty_is_noop(lib, kw):
    assert call_dec(**kw) == attn.ATTN_OK


@pytest.mark.parametrize("args,code", [
    ((P, P, None, 1, 64, 512, 8, 4, P2, P2, P2), attn.ATTN_ERR_INVALID_ARG),     # num_out 4
    ((P, P, None, 1, 64, 512, 8, 0, P2, P2, P2), attn.ATTN_ERR_INVALID_ARG),
    ((P, P, None, 1, 64, 512, 16, 3, P2, P2, P2), attn.ATTN_ERR_UNSUPPORTED),    # head dim 32
    ((P, P, None, 1, 48, 512, 8, 3, P2, P2, P2), attn.ATTN_ERR_UNSUPPORTED),     # n not a multiple of 32
    ((P, P, None, 1, 64, 512, 8, 2, P2, None, P2), attn.ATTN_ERR_INVALID_ARG),   # missing output
    ((P, P, ctypes.c_void_p(0x30008), 1, 64, 512, 8, 1, P2, None, None), attn.ATTN_ERR_MISALIGNED),
    ((P, P, None, 0, 64, 512, 8, 3, None, None, None), attn.ATTN_OK),             # no rows
])
def test_proj_heads_validation(lib, args, code):
    assert lib.attn_proj_heads(*args, None) == code


@pytest.mark.parametrize("args,code", [
    ((P, P, None, 1, 64, 8, 96, 512, P2), attn.ATTN_ERR_UNSUPPORTED),            # head dim 96
    ((P, P, None, 1, 64, 8, 64, 100, P2), attn.ATTN_ERR_UNSUPPORTED),            # d_out % 64
    ((P, P, None, 1, 40, 8, 64, 512, P2), attn.ATTN_ERR_UNSUPPORTED),            # n % 32
    ((P, P, None, 1, 64, 8, 64, 512, None), attn.ATTN_ERR_INVALID_ARG),
    ((P, P, None, 1, 64, 8, 64, 512, ctypes.c_void_p(0x20002)), attn.ATTN_ERR_MISALIGNED),
    ((P, P, None, 1, 0, 8, 64, 512, P2), attn.ATTN_OK),
])
def test_merge_proj_validation(lib, args, code):
    assert lib.attn_merge_proj(*args, None) == code

"""Python loader for the fp64 CPU attention oracle (``attn_oracle.c``).

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline leg import this module. It compiles ``attn_oracle.c`` with gcc into
``oracle/_build/`` and calls it through ctypes. It imports nothing from the
CUDA package and the CUDA package imports nothing from here.

Inputs may be torch tensors (any float dtype; bf16 widens to fp64 exactly) or
numpy arrays. Outputs are fp64 numpy arrays.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "attn_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")

# The oracle's own mask codes (independent of the CUDA library's enum).
MASK_CODES = {"none": 0, "causal": 1, "key_padding": 2, "causal_key_padding": 3, "causal_cache": 4}

_lock = threading.Lock()
_libs: dict[int, ctypes.CDLL] = {}


def lib_path(plant: int = 0) -> str:
    name = "libattn_oracle.so" if plant == 0 else f"libattn_oracle_plant{plant}.so"
    return os.path.join(BUILD_DIR, name)


def build(plant: int = 0, force: bool = False) -> str:
    """Compile the oracle (plain C11, -O2, no fast-math) and return the .so path.

    ``plant`` > 0 builds a copy with one planted mistake (tests only)."""
    out = lib_path(plant)
    with _lock:
        if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
            return out
        os.makedirs(BUILD_DIR, exist_ok=True)
        tmp = f"{out}.{os.getpid()}.tmp"
        cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread",
               f"-DORACLE_PLANT={int(plant)}", SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def _load(plant: int = 0) -> ctypes.CDLL:
    if plant in _libs:
        return _libs[plant]
    lib = ctypes.CDLL(build(plant))
    dp = ctypes.POINTER(ctypes.c_double)
    i32p = ctypes.POINTER(ctypes.c_int32)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    ci = ctypes.c_int
    lib.oracle_attn_fwd.argtypes = [dp, dp, dp, i64, i64, i64, i64, ci, ci, ci, i32p,
                                    ctypes.c_double, dp, dp, dp, ci]
    lib.oracle_attn_fwd.restype = ci
    lib.oracle_attn_rows.argtypes = [dp, dp, dp, i64, i64, i64, i64, ci, ci, ci, i32p,
                                     ctypes.c_double, i64p, i64, dp, dp, ci]
    lib.oracle_attn_rows.restype = ci
    lib.oracle_attn_bwd.argtypes = [dp, dp, dp, dp, i64, i64, i64, i64, ci, ci, ci, i32p,
                                    ctypes.c_double, dp, dp, dp, ci]
    lib.oracle_attn_bwd.restype = ci
    lib.oracle_attn_fwd_alibi.argtypes = [dp, dp, dp, i64, i64, i64, i64, ci, ci, ci, i32p, dp,
                                          ctypes.c_double, dp, dp, dp, ci]
    lib.oracle_attn_fwd_alibi.restype = ci
    lib.oracle_attn_rows_alibi.argtypes = [dp, dp, dp, i64, i64, i64, i64, ci, ci, ci, i32p, dp,
                                           ctypes.c_double, i64p, i64, dp, dp, ci]
    lib.oracle_attn_rows_alibi.restype = ci
    lib.oracle_attn_bwd_alibi.argtypes = [dp, dp, dp, dp, i64, i64, i64, i64, ci, ci, ci, i32p, dp,
                                          ctypes.c_double, dp, dp, dp, ci]
    lib.oracle_attn_bwd_alibi.restype = ci
    _libs[plant] = lib
    return lib


def _f64(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu", torch.float64).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _lens(key_lengths, B):
    if key_lengths is None:
        return None
    arr = np.ascontiguousarray(np.asarray(
        key_lengths.cpu().numpy() if hasattr(key_lengths, "cpu") else key_lengths,
        dtype=np.int32).reshape(B))
    return arr


def _ptr(a, ctype):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _shapes(Q, K, V):
    if Q.ndim != 4 or K.ndim != 4 or V.ndim != 4:
        raise ValueError("Q, K, V must be [B, H, L, d]")
    B, H, n, dk = Q.shape
    m = K.shape[2]
    dv = V.shape[3]
    if K.shape != (B, H, m, dk) or V.shape[:3] != (B, H, m):
        raise ValueError("inconsistent Q/K/V shapes")
    return B, H, n, m, dk, dv


def _slopes(slopes, H):
    if slopes is None:
        return None
    arr = _f64(slopes).reshape(-1)
    if arr.size != H:
        raise ValueError(f"slopes must hold one value per head ({H})")
    return np.ascontiguousarray(arr)


def attn_fwd(Q, K, V, mask="none", key_lengths=None, scale=None, *, slopes=None, threads=None,
             weights=False, plant=0):
    """Oracle forward. Returns (O [B,H,n,dv], LSE [B,H,n]) or, with weights=True,
    (O, LSE, W [B,H,n,m]). ``scale`` defaults to 1/sqrt(d_k). ``slopes`` [H] adds the
    linear distance bias -slopes[h] * |i + m - n - j| to every scaled score."""
    Qd, Kd, Vd = _f64(Q), _f64(K), _f64(V)
    B, H, n, m, dk, dv = _shapes(Qd, Kd, Vd)
    sc = 1.0 / np.sqrt(dk) if scale is None else float(scale)
    lens = _lens(key_lengths, B)
    sl = _slopes(slopes, H)
    O = np.zeros((B, H, n, dv))
    L = np.zeros((B, H, n))
    W = np.zeros((B, H, n, m)) if weights else None
    lib = _load(plant)
    common = (_ptr(Qd, ctypes.c_double), _ptr(Kd, ctypes.c_double), _ptr(Vd, ctypes.c_double),
              B, H, n, m, dk, dv, MASK_CODES[mask], _ptr(lens, ctypes.c_int32))
    outs = (_ptr(O, ctypes.c_double), _ptr(L, ctypes.c_double), _ptr(W, ctypes.c_double),
            threads or min(default_threads(), 16))
    if sl is None:
        rc = lib.oracle_attn_fwd(*common, sc, *outs)
    else:
        rc = lib.oracle_attn_fwd_alibi(*common, _ptr(sl, ctypes.c_double), sc, *outs)
    if rc != 0:
        raise RuntimeError(f"oracle_attn_fwd failed ({rc})")
    return (O, L, W) if weights else (O, L)


def attn_rows(Q, K, V, rows, mask="none", key_lengths=None, scale=None, *, slopes=None,
              threads=None, plant=0):
    """Oracle outputs for selected flat rows (b*H*n + h*n + i): (O [k,dv], LSE [k]).
    ``slopes`` as for ``attn_fwd``."""
    Qd, Kd, Vd = _f64(Q), _f64(K), _f64(V)
    B, H, n, m, dk, dv = _shapes(Qd, Kd, Vd)
    sc = 1.0 / np.sqrt(dk) if scale is None else float(scale)
    lens = _lens(key_lengths, B)
    sl = _slopes(slopes, H)
    r = np.ascontiguousarray(np.asarray(
        rows.cpu().numpy() if hasattr(rows, "cpu") else rows, dtype=np.int64).reshape(-1))
    O = np.zeros((r.size, dv))
    L = np.zeros((r.size,))
    lib = _load(plant)
    common = (_ptr(Qd, ctypes.c_double), _ptr(Kd, ctypes.c_double), _ptr(Vd, ctypes.c_double),
              B, H, n, m, dk, dv, MASK_CODES[mask], _ptr(lens, ctypes.c_int32))
    tail = (_ptr(r, ctypes.c_int64), r.size, _ptr(O, ctypes.c_double), _ptr(L, ctypes.c_double),
            threads or min(default_threads(), 16))
    if sl is None:
        rc = lib.oracle_attn_rows(*common, sc, *tail)
    else:
        rc = lib.oracle_attn_rows_alibi(*common, _ptr(sl, ctypes.c_double), sc, *tail)
    if rc != 0:
        raise RuntimeError(f"oracle_attn_rows failed ({rc})")
    return O, L


def attn_bwd(Q, K, V, dO, mask="none", key_lengths=None, scale=None, *, slopes=None, threads=None,
             plant=0):
    """Oracle backward for the upstream gradient dO [B,H,n,dv]: returns (dQ [B,H,n,dk],
    dK [B,H,m,dk], dV [B,H,m,dv]) in fp64. ``scale`` defaults to 1/sqrt(d_k); ``slopes``
    [H] differentiates the forward with the linear distance bias."""
    Qd, Kd, Vd, dOd = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, H, n, m, dk, dv = _shapes(Qd, Kd, Vd)
    if dOd.shape != (B, H, n, dv):
        raise ValueError("dO must be [B, H, n, d_v]")
    sc = 1.0 / np.sqrt(dk) if scale is None else float(scale)
    lens = _lens(key_lengths, B)
    dQ = np.zeros((B, H, n, dk))
    dK = np.zeros((B, H, m, dk))
    dV = np.zeros((B, H, m, dv))
    sl = _slopes(slopes, H)
    lib = _load(plant)
    head = (_ptr(Qd, ctypes.c_double), _ptr(Kd, ctypes.c_double), _ptr(Vd, ctypes.c_double),
            _ptr(dOd, ctypes.c_double), B, H, n, m, dk, dv, MASK_CODES[mask], _ptr(lens, ctypes.c_int32))
    tail = (_ptr(dQ, ctypes.c_double), _ptr(dK, ctypes.c_double), _ptr(dV, ctypes.c_double),
            threads or min(default_threads(), 16))
    if sl is None:
        rc = lib.oracle_attn_bwd(*head, sc, *tail)
    else:
        rc = lib.oracle_attn_bwd_alibi(*head, _ptr(sl, ctypes.c_double), sc, *tail)
    if rc != 0:
        raise RuntimeError(f"oracle_attn_bwd failed ({rc})")
    return dQ, dK, dV


# ------------------------------------------------------------------ projections around the attention
#
# "从 RNN 到 Transformer（二）" §4.6 and "Transformer 详解" §4.2: the heads are the
# projections of the input split per head, W_Q(x).view(B, n, h, d_k).transpose(1, 2),
# and the output is the heads merged back, out.transpose(1, 2).reshape(B, n, h d_k),
# followed by W_O. Weights are in the pages' nn.Linear layout [out_features,
# in_features] (y = x Wᵀ + b); the bias is optional (one page's projections have
# none, the other's have nn.Linear's default bias). fp64, numpy matmul as the
# library step.

def _plant_split(y, B, n, H, d, plant):
    if plant == 12:
        return y.reshape(B, n, d, H).transpose(0, 3, 1, 2)      # planted: (d, h) order swapped
    return y.reshape(B, n, H, d).transpose(0, 2, 1, 3)


def proj_heads(X, W, bias, H, num_out, *, plant=0):
    """X [B, n, d_model]; W [num_out*d_model, d_model]; bias [num_out*d_model] or None.
    Returns num_out arrays [B, H, n, d_model/H]: the projection y = X Wᵀ + b, column
    block t, split per head."""
    Xd, Wd = _f64(X), _f64(W)
    B, n, dm = Xd.shape
    d = dm // H
    if plant == 13:
        y = Xd.reshape(B * n, dm) @ Wd.reshape(dm, -1)          # planted: weight read as [in, out]
    else:
        y = Xd.reshape(B * n, dm) @ Wd.T
    if bias is not None:
        y = y + _f64(bias)[None, :]
    outs = []
    for t in range(num_out):
        yt = y[:, t * dm:(t + 1) * dm]
        outs.append(np.ascontiguousarray(_plant_split(yt, B, n, H, d, plant)))
    return outs


def merge_proj(O, W_o, bias, *, plant=0):
    """O [B, H, n, d]; W_o [d_out, H*d]; bias [d_out] or None. Returns Y [B, n, d_out]:
    the heads merged back (column h*d + j) times W_oᵀ plus the bias."""
    Od, Wd = _f64(O), _f64(W_o)
    B, H, n, d = Od.shape
    merged = Od.transpose(0, 2, 1, 3).reshape(B * n, H * d)
    y = merged @ Wd.T
    if bias is not None:
        y = y + _f64(bias)[None, :]
    return y.reshape(B, n, Wd.shape[0])

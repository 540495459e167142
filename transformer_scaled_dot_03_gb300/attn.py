"""Python binding of the C-ABI attention library (``libattn_sm103a.so``).

Argument marshalling only: tensors are checked for dtype, shape, device and
contiguity, and their device pointers plus PyTorch's current CUDA stream are
passed to the C entry points declared in ``include/attn.h``. Every step of the
attention forward pass runs in the library's kernels. There is no fallback:
if the library is missing or no GPU is present, the call raises.
"""

from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import inputs as _inputs

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn_sm103a.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_MISALIGNED = -3
ATTN_ERR_CUDA = -4
ATTN_ERR_TIMEOUT = -5

MASK_CODES = {_inputs.MASK_NONE: 0, _inputs.MASK_CAUSAL: 1, _inputs.MASK_KEY_PADDING: 2,
              _inputs.MASK_CAUSAL_KEY_PADDING: 3, _inputs.MASK_CAUSAL_CACHE: 4}

# Every symbol include/attn.h declares.
EXPORTS = ("attn_fwd", "attn_fwd_alibi", "attn_decode_alibi", "attn_bwd_alibi", "attn_get_device_status",
           "attn_last_status_detail", "attn_set_watchdog", "attn_status_string", "attn_last_error",
           "attn_fwd_noalloc", "attn_bwd", "attn_bwd_workspace_size", "attn_decode",
           "attn_decode_workspace_size", "attn_proj_heads", "attn_merge_proj")

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status}) {detail}".rstrip())


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the shared library (built by ``transformer_scaled_dot_03_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA attention library not built: {path} "
                               "(run transformer_scaled_dot_03_gb300.build.build())")
        lib = ctypes.CDLL(path)
        vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.attn_fwd.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, f32, vp, vp, vp]
        lib.attn_fwd.restype = i32
        lib.attn_fwd_alibi.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, f32, vp, vp, vp]
        lib.attn_fwd_alibi.restype = i32
        lib.attn_get_device_status.argtypes = [vp]
        lib.attn_get_device_status.restype = i32
        lib.attn_last_status_detail.argtypes = []
        lib.attn_last_status_detail.restype = ctypes.c_uint32
        lib.attn_fwd_noalloc.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, f32, vp, vp, vp]
        lib.attn_fwd_noalloc.restype = i32
        lib.attn_set_watchdog.argtypes = [ctypes.c_uint64, ctypes.c_uint32]
        lib.attn_set_watchdog.restype = None
        lib.attn_status_string.argtypes = [i32]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, f32,
                                 vp, vp, vp, vp, ctypes.c_size_t, vp]
        lib.attn_bwd.restype = i32
        lib.attn_bwd_alibi.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, f32,
                                       vp, vp, vp, vp, ctypes.c_size_t, vp]
        lib.attn_bwd_alibi.restype = i32
        lib.attn_bwd_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.attn_bwd_workspace_size.restype = ctypes.c_size_t
        lib.attn_decode.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, f32, vp, vp, vp,
                                    ctypes.c_size_t, vp]
        lib.attn_decode.restype = i32
        lib.attn_decode_alibi.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, f32, vp, vp, vp,
                                          ctypes.c_size_t, vp]
        lib.attn_decode_alibi.restype = i32
        lib.attn_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.attn_decode_workspace_size.restype = ctypes.c_size_t
        lib.attn_proj_heads.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp]
        lib.attn_proj_heads.restype = i32
        lib.attn_merge_proj.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp]
        lib.attn_merge_proj.restype = i32
        lib.attn_last_error.argtypes = []
        lib.attn_last_error.restype = ctypes.c_char_p
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


def last_error() -> str:
    return load().attn_last_error().decode()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def attn_fwd_raw(Q_ptr, K_ptr, V_ptr, B, H, n, m, d_k, d_v, mask_kind, key_lengths_ptr, scale,
                 O_ptr, LSE_ptr, stream_handle) -> int:
    """The C entry point with plain integers/pointers; returns the status code."""
    return load().attn_fwd(Q_ptr, K_ptr, V_ptr, int(B), int(H), int(n), int(m), int(d_k), int(d_v),
                           int(mask_kind), key_lengths_ptr, ctypes.c_float(scale), O_ptr, LSE_ptr,
                           ctypes.c_void_p(stream_handle))


def attn_fwd(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, mask: str = "none",
             key_lengths: torch.Tensor | None = None, scale: float | None = None,
             O: torch.Tensor | None = None, LSE: torch.Tensor | None = None,
             want_lse: bool = True, stream=None):
    """Attention forward on the GPU. Q [B,H,n,d_k], K [B,H,m,d_k], V [B,H,m,d_v] bf16
    CUDA tensors (contiguous); ``key_lengths`` int32 CUDA [B] for the key-padding masks
    ("key_padding", "causal_key_padding", "causal_cache"). Returns (O [B,H,n,d_v] bf16, LSE [B,H,n] fp32
    or None). Asynchronous on ``stream`` (default: PyTorch's current stream)."""
    if mask not in MASK_CODES:
        raise ValueError(f"unknown mask {mask!r}")
    for name, t in (("Q", Q), ("K", K), ("V", V)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D bf16 CUDA tensor")
    B, H, n, d_k = Q.shape
    m = K.shape[2]
    d_v = V.shape[3]
    if tuple(K.shape) != (B, H, m, d_k) or tuple(V.shape[:3]) != (B, H, m):
        raise ValueError("inconsistent Q/K/V shapes")
    uses_lengths = mask in _inputs.LENGTH_MASKS
    if uses_lengths:
        if key_lengths is None or key_lengths.dtype != torch.int32 or not key_lengths.is_cuda \
                or key_lengths.numel() != B or not key_lengths.is_contiguous():
            raise ValueError(f"{mask} needs key_lengths: contiguous int32 CUDA [B]")
    if O is None:
        O = torch.empty((B, H, n, d_v), dtype=torch.bfloat16, device=Q.device)
    if LSE is None and want_lse:
        LSE = torch.empty((B, H, n), dtype=torch.float32, device=Q.device)
    sc = -1.0 if scale is None else float(scale)
    rc = attn_fwd_raw(_ptr(Q), _ptr(K), _ptr(V), B, H, n, m, d_k, d_v, MASK_CODES[mask],
                      _ptr(key_lengths) if uses_lengths else None, sc, _ptr(O), _ptr(LSE),
                      _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd", last_error() if rc == ATTN_ERR_CUDA else "")
    return O, LSE


def attn_fwd_alibi(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, slopes: torch.Tensor,
                   mask: str = "none", key_lengths: torch.Tensor | None = None, scale: float | None = None,
                   O: torch.Tensor | None = None, LSE: torch.Tensor | None = None,
                   want_lse: bool = True, stream=None):
    """Attention forward with the linear distance bias -slopes[h] * |i + m - n - j| added
    to every scaled score (ALiBi). ``slopes`` is a contiguous fp32 CUDA tensor [H];
    everything else as in ``attn_fwd`` (d_k == d_v in {64, 128})."""
    if mask not in MASK_CODES:
        raise ValueError(f"unknown mask {mask!r}")
    for name, t in (("Q", Q), ("K", K), ("V", V)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D bf16 CUDA tensor")
    B, H, n, d_k = Q.shape
    m = K.shape[2]
    d_v = V.shape[3]
    if tuple(K.shape) != (B, H, m, d_k) or tuple(V.shape[:3]) != (B, H, m):
        raise ValueError("inconsistent Q/K/V shapes")
    if slopes.dtype != torch.float32 or not slopes.is_cuda or slopes.numel() != H or not slopes.is_contiguous():
        raise ValueError("slopes must be a contiguous fp32 CUDA tensor with one value per head")
    uses_lengths = mask in _inputs.LENGTH_MASKS
    if uses_lengths:
        if key_lengths is None or key_lengths.dtype != torch.int32 or not key_lengths.is_cuda \
                or key_lengths.numel() != B or not key_lengths.is_contiguous():
            raise ValueError(f"{mask} needs key_lengths: contiguous int32 CUDA [B]")
    if O is None:
        O = torch.empty((B, H, n, d_v), dtype=torch.bfloat16, device=Q.device)
    if LSE is None and want_lse:
        LSE = torch.empty((B, H, n), dtype=torch.float32, device=Q.device)
    sc = -1.0 if scale is None else float(scale)
    rc = load().attn_fwd_alibi(_ptr(Q), _ptr(K), _ptr(V), int(B), int(H), int(n), int(m), int(d_k), int(d_v),
                               MASK_CODES[mask], _ptr(key_lengths) if uses_lengths else None, _ptr(slopes),
                               ctypes.c_float(sc), _ptr(O), _ptr(LSE), ctypes.c_void_p(_stream_handle(stream)))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_alibi", last_error() if rc == ATTN_ERR_CUDA else "")
    return O, LSE


def attn_bwd_raw(Q_ptr, K_ptr, V_ptr, O_ptr, dO_ptr, LSE_ptr, B, H, n, m, d_k, d_v, mask_kind,
                 key_lengths_ptr, scale, dQ_ptr, dK_ptr, dV_ptr, ws_ptr, ws_bytes, stream_handle) -> int:
    """The C backward entry point with plain integers/pointers; returns the status code."""
    return load().attn_bwd(Q_ptr, K_ptr, V_ptr, O_ptr, dO_ptr, LSE_ptr, int(B), int(H), int(n), int(m),
                           int(d_k), int(d_v), int(mask_kind), key_lengths_ptr, ctypes.c_float(scale),
                           dQ_ptr, dK_ptr, dV_ptr, ws_ptr, ctypes.c_size_t(ws_bytes),
                           ctypes.c_void_p(stream_handle))


def bwd_workspace_size(B, H, n, m, d_k, d_v) -> int:
    return int(load().attn_bwd_workspace_size(int(B), int(H), int(n), int(m), int(d_k), int(d_v)))


def attn_bwd(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, O: torch.Tensor, LSE: torch.Tensor,
             dO: torch.Tensor, mask: str = "none", key_lengths: torch.Tensor | None = None,
             scale: float | None = None, dQ: torch.Tensor | None = None, dK: torch.Tensor | None = None,
             dV: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None,
             slopes: torch.Tensor | None = None):
    """Attention backward on the GPU: (dQ, dK, dV) bf16 for the upstream gradient dO, given
    the forward's inputs Q, K, V and outputs O (bf16) and LSE (fp32). ``workspace`` (uint8
    CUDA tensor of at least ``bwd_workspace_size`` bytes) is allocated here when omitted.
    ``slopes`` (contiguous fp32 CUDA [H]) differentiates ``attn_fwd_alibi`` with those
    slopes (attn_bwd_alibi).
    Asynchronous on ``stream`` (default: PyTorch's current stream)."""
    if mask not in MASK_CODES:
        raise ValueError(f"unknown mask {mask!r}")
    for name, t in (("Q", Q), ("K", K), ("V", V), ("O", O), ("dO", dO)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D bf16 CUDA tensor")
    B, H, n, d_k = Q.shape
    m = K.shape[2]
    d_v = V.shape[3]
    if tuple(K.shape) != (B, H, m, d_k) or tuple(V.shape[:3]) != (B, H, m) \
            or tuple(O.shape) != (B, H, n, d_v) or tuple(dO.shape) != (B, H, n, d_v):
        raise ValueError("inconsistent Q/K/V/O/dO shapes")
    if LSE.dtype != torch.float32 or not LSE.is_cuda or tuple(LSE.shape) != (B, H, n) \
            or not LSE.is_contiguous():
        raise ValueError("LSE must be a contiguous fp32 CUDA tensor [B, H, n]")
    uses_lengths = mask in _inputs.LENGTH_MASKS
    if uses_lengths and (key_lengths is None or key_lengths.dtype != torch.int32
                         or not key_lengths.is_cuda or key_lengths.numel() != B
                         or not key_lengths.is_contiguous()):
        raise ValueError(f"{mask} needs key_lengths: contiguous int32 CUDA [B]")
    dev = Q.device
    dQ = torch.empty((B, H, n, d_k), dtype=torch.bfloat16, device=dev) if dQ is None else dQ
    dK = torch.empty((B, H, m, d_k), dtype=torch.bfloat16, device=dev) if dK is None else dK
    dV = torch.empty((B, H, m, d_v), dtype=torch.bfloat16, device=dev) if dV is None else dV
    ws_bytes = bwd_workspace_size(B, H, n, m, d_k, d_v)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    elif workspace.numel() < ws_bytes or workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise ValueError(f"workspace must be a uint8 CUDA tensor of at least {ws_bytes} bytes")
    sc = -1.0 if scale is None else float(scale)
    lens_p = _ptr(key_lengths) if uses_lengths else None
    if slopes is None:
        rc = attn_bwd_raw(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE), B, H, n, m, d_k, d_v,
                          MASK_CODES[mask], lens_p, sc, _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(workspace),
                          workspace.numel(), _stream_handle(stream))
    else:
        if slopes.dtype != torch.float32 or not slopes.is_cuda or slopes.numel() != H or not slopes.is_contiguous():
            raise ValueError("slopes must be a contiguous fp32 CUDA tensor with one value per head")
        rc = load().attn_bwd_alibi(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE), int(B), int(H), int(n),
                                   int(m), int(d_k), int(d_v), MASK_CODES[mask], lens_p, _ptr(slopes),
                                   ctypes.c_float(sc), _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(workspace),
                                   ctypes.c_size_t(workspace.numel()), ctypes.c_void_p(_stream_handle(stream)))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd", last_error() if rc == ATTN_ERR_CUDA else "")
    return dQ, dK, dV


def decode_workspace_size(B, H, n, m, d_k, d_v) -> int:
    return int(load().attn_decode_workspace_size(int(B), int(H), int(n), int(m), int(d_k), int(d_v)))


def attn_decode_raw(Q_ptr, K_ptr, V_ptr, B, H, n, m, d_k, d_v, mask_kind, key_lengths_ptr, scale, O_ptr,
                    LSE_ptr, ws_ptr, ws_bytes, stream_handle) -> int:
    """The C decode entry point with plain integers/pointers; returns the status code."""
    return load().attn_decode(Q_ptr, K_ptr, V_ptr, int(B), int(H), int(n), int(m), int(d_k), int(d_v),
                              int(mask_kind), key_lengths_ptr, ctypes.c_float(scale), O_ptr, LSE_ptr, ws_ptr,
                              ctypes.c_size_t(ws_bytes), ctypes.c_void_p(stream_handle))


def attn_decode(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, mask: str = "none",
                key_lengths: torch.Tensor | None = None, scale: float | None = None,
                O: torch.Tensor | None = None, LSE: torch.Tensor | None = None, want_lse: bool = True,
                workspace: torch.Tensor | None = None, stream=None, slopes: torch.Tensor | None = None):
    """Few-row attention forward (n <= 8 query rows per head against m keys, e.g. one
    decoding step against a key/value cache): same arguments and results as
    ``attn_fwd``. ``workspace`` (uint8 CUDA tensor of at least ``decode_workspace_size``
    bytes) is allocated here when omitted and needed. ``slopes`` (contiguous fp32 CUDA
    [H]) adds the linear distance bias of ``attn_fwd_alibi`` (attn_decode_alibi)."""
    if mask not in MASK_CODES:
        raise ValueError(f"unknown mask {mask!r}")
    for name, t in (("Q", Q), ("K", K), ("V", V)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D bf16 CUDA tensor")
    B, H, n, d_k = Q.shape
    m = K.shape[2]
    d_v = V.shape[3]
    if tuple(K.shape) != (B, H, m, d_k) or tuple(V.shape[:3]) != (B, H, m):
        raise ValueError("inconsistent Q/K/V shapes")
    uses_lengths = mask in _inputs.LENGTH_MASKS
    if uses_lengths and (key_lengths is None or key_lengths.dtype != torch.int32
                         or not key_lengths.is_cuda or key_lengths.numel() != B
                         or not key_lengths.is_contiguous()):
        raise ValueError(f"{mask} needs key_lengths: contiguous int32 CUDA [B]")
    if O is None:
        O = torch.empty((B, H, n, d_v), dtype=torch.bfloat16, device=Q.device)
    if LSE is None and want_lse:
        LSE = torch.empty((B, H, n), dtype=torch.float32, device=Q.device)
    ws_bytes = decode_workspace_size(B, H, n, m, d_k, d_v)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=Q.device)
    if workspace is not None and (workspace.numel() < ws_bytes or workspace.dtype != torch.uint8):
        raise ValueError(f"workspace must be a uint8 CUDA tensor of at least {ws_bytes} bytes")
    sc = -1.0 if scale is None else float(scale)
    lens_p = _ptr(key_lengths) if uses_lengths else None
    ws_n = 0 if workspace is None else workspace.numel()
    if slopes is None:
        rc = attn_decode_raw(_ptr(Q), _ptr(K), _ptr(V), B, H, n, m, d_k, d_v, MASK_CODES[mask], lens_p, sc,
                             _ptr(O), _ptr(LSE), _ptr(workspace), ws_n, _stream_handle(stream))
    else:
        if slopes.dtype != torch.float32 or not slopes.is_cuda or slopes.numel() != H or not slopes.is_contiguous():
            raise ValueError("slopes must be a contiguous fp32 CUDA tensor with one value per head")
        rc = load().attn_decode_alibi(_ptr(Q), _ptr(K), _ptr(V), int(B), int(H), int(n), int(m), int(d_k),
                                      int(d_v), MASK_CODES[mask], lens_p, _ptr(slopes), ctypes.c_float(sc), _ptr(O),
                                      _ptr(LSE), _ptr(workspace), ctypes.c_size_t(ws_n),
                                      ctypes.c_void_p(_stream_handle(stream)))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode", last_error() if rc == ATTN_ERR_CUDA else "")
    return O, LSE


def _bf16_cuda(name, t, dim):
    if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != dim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dim}-D bf16 CUDA tensor")


def proj_heads(X: torch.Tensor, W: torch.Tensor, H: int, bias: torch.Tensor | None = None,
               num_out: int | None = None, outs=None, stream=None):
    """Input projections with the per-head split: X [B, n, d_model], W [num_out*d_model,
    d_model] (nn.Linear layout), optional bias [num_out*d_model]; returns num_out tensors
    [B, H, n, d_model/H] (e.g. Q, K, V). Asynchronous on ``stream``."""
    _bf16_cuda("X", X, 3)
    _bf16_cuda("W", W, 2)
    B, n, d_model = X.shape
    num_out = W.shape[0] // d_model if num_out is None else num_out
    if tuple(W.shape) != (num_out * d_model, d_model):
        raise ValueError("W must be [num_out*d_model, d_model]")
    if bias is not None:
        _bf16_cuda("bias", bias, 1)
        if bias.numel() != num_out * d_model:
            raise ValueError("bias must be [num_out*d_model]")
    d = d_model // H if H > 0 else 0
    if outs is None:
        outs = [torch.empty((B, H, n, d), dtype=torch.bfloat16, device=X.device) for _ in range(num_out)]
    ptrs = [_ptr(t) for t in outs] + [None] * (3 - len(outs))
    rc = load().attn_proj_heads(_ptr(X), _ptr(W), _ptr(bias), int(B), int(n), int(d_model), int(H), int(num_out),
                                ptrs[0], ptrs[1], ptrs[2], ctypes.c_void_p(_stream_handle(stream)))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_proj_heads", last_error() if rc == ATTN_ERR_CUDA else "")
    return outs


def merge_proj(O: torch.Tensor, W_o: torch.Tensor, bias: torch.Tensor | None = None, Y=None, stream=None):
    """Output projection of the merged heads: O [B, H, n, d], W_o [d_out, H*d] (nn.Linear
    layout), optional bias [d_out]; returns Y [B, n, d_out]. Asynchronous on ``stream``."""
    _bf16_cuda("O", O, 4)
    _bf16_cuda("W_o", W_o, 2)
    B, H, n, d = O.shape
    d_out = W_o.shape[0]
    if W_o.shape[1] != H * d:
        raise ValueError("W_o must be [d_out, H*d]")
    if bias is not None:
        _bf16_cuda("bias", bias, 1)
    if Y is None:
        Y = torch.empty((B, n, d_out), dtype=torch.bfloat16, device=O.device)
    rc = load().attn_merge_proj(_ptr(O), _ptr(W_o), _ptr(bias), int(B), int(n), int(H), int(d), int(d_out),
                                _ptr(Y), ctypes.c_void_p(_stream_handle(stream)))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_merge_proj", last_error() if rc == ATTN_ERR_CUDA else "")
    return Y


def device_status(stream=None) -> tuple[int, int]:
    """Synchronise the stream, read and clear the device's status words; return
    (status, detail bits)."""
    lib = load()
    rc = lib.attn_get_device_status(ctypes.c_void_p(_stream_handle(stream)))
    return rc, int(lib.attn_last_status_detail())


def set_watchdog(limit_ns: int = 0, debug_flags: int = 0) -> None:
    load().attn_set_watchdog(ctypes.c_uint64(limit_ns), ctypes.c_uint32(debug_flags))


def flops(B, H, n, m, d_k, mask, d_v=None) -> float:
    """Nominal forward FLOPs: 2*B*H*(d_k + d_v) per visible (query, key) pair (d_v
    defaults to d_k). Without a causal mask every pair counts (n*m); with it the masked
    triangle counts as half its square, n*m - n*n/2 for n <= m (n*m/2 when n = m) and
    m*m/2 for n > m."""
    d_v = d_k if d_v is None else d_v
    return 2.0 * B * H * (d_k + d_v) * _inputs.nominal_pairs(n, m, mask)


def default_scale(d_k: int) -> float:
    return 1.0 / math.sqrt(d_k)

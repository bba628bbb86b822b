"""ctypes binding of libdfa.so: argument marshalling only.

Every function here has the name of the C entry point it calls (see
``include/dfa.h``) and does nothing but check tensor shapes, dtypes and
devices, allocate outputs with PyTorch, and pass raw pointers, sizes and the
current CUDA stream to the library.  Every step of the computation runs in
the library's CUDA kernels; there is no other implementation to fall back to,
so a missing or unloadable library raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdfa.so")

DFA_OK = 0
DFA_EINVAL = -1
DFA_EUNSUPPORTED = -2
DFA_ECUDA = -3
DFA_ETIMEOUT = -4
DFA_EDEVICE = -5
DFA_DETERMINISTIC = 1
DFA_NOISY_DIAG_PASS = 2
MODE_DIFFUSION = 0
MODE_CAUSAL = 1

_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGNATURES = {
    "dfa_version": (_I, []),
    "dfa_error_string": (ctypes.c_char_p, [_I]),
    "dfa_last_cuda_error": (ctypes.c_char_p, []),
    "dfa_forward": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "dfa_backward": (_I, [_P] * 9 + [_I, _I, _I, _I, _I, _P]),
    "dfa_forward_gqa": (_I, [_P] * 5 + [_I] * 6 + [_P]),
    "dfa_backward_gqa": (_I, [_P] * 9 + [_I] * 6 + [_P]),
    "dfa_forward_varlen": (_I, [_P] * 6 + [_I] * 5 + [_P]),
    "dfa_backward_varlen": (_I, [_P] * 10 + [_I] * 5 + [_P]),
    "dfa_backward_ex": (_I, [_P] * 10 + [_I] * 7 + [_P]),
    "dfa_forward_fp8": (_I, [_P] * 5 + [ctypes.c_float] * 3 + [_I] * 6 + [_P]),
    "dfa_fp8_vt_bytes": (ctypes.c_longlong, [_I] * 4),
    "dfa_fp8_transpose_v": (_I, [_P] * 2 + [_I] * 4 + [_P]),
    "dfa_forward_fp8_vt": (_I, [_P] * 5 + [ctypes.c_float] * 3 + [_I] * 6 + [_P]),
    "dfa_causal_forward": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "dfa_causal_backward": (_I, [_P] * 9 + [_I, _I, _I, _I, _P]),
    "dfa_status": (_I, [_P]),
    "dfa_selftest_wait_timeout": (_I, [_I, _P]),
    "dfa_fwd_main": (_I, [_P] * 6 + [_I] * 6 + [_P]),
    "dfa_bwd_preprocess": (_I, [_P] * 4 + [_I] * 4 + [_P]),
    "dfa_bwd_main": (_I, [_P] * 9 + [_I] * 6 + [_P]),
    "dfa_bwd_dq_convert": (_I, [_P] * 2 + [_I] * 4 + [_P]),
    "dfa_bwd_preprocess_ex": (_I, [_P] * 4 + [_I] * 5 + [_P]),
    "dfa_bwd_dq_convert_ex": (_I, [_P] * 2 + [_I] * 5 + [_P]),
    "dfa_fwd_main_gqa": (_I, [_P] * 6 + [_I] * 7 + [_P]),
    "dfa_bwd_main_gqa": (_I, [_P] * 9 + [_I] * 7 + [_P]),
    "dfa_bwd_main_ex": (_I, [_P] * 9 + [_I] * 8 + [_P]),
    "dfa_fwd_segments": (_I, [_I] * 7 + [ctypes.POINTER(_I)]),
    "dfa_bwd_segments": (_I, [_I] * 7 + [ctypes.POINTER(_I)]),
    "dfa_tile_full": (_I, [_I] * 7),
    "dfa_tile_visits": (ctypes.c_longlong, [_I] * 6),
    "dfa_tile_shape": (_I, [_I] + [ctypes.POINTER(_I)] * 4),
    "dfa_work_item": (_I, [_I] * 7 + [ctypes.POINTER(_I)]),
}


class DfaError(RuntimeError):
    def __init__(self, fn, code):
        msg = lib().dfa_error_string(code).decode()
        if code == DFA_ECUDA:
            msg += ": " + lib().dfa_last_cuda_error().decode()
        super().__init__(f"{fn} failed: {msg} ({code})")
        self.code = code


def lib():
    """Load libdfa.so (built in-tree by ``build()``) once and return it."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdfa.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(fn, rc):
    if rc != DFA_OK:
        raise DfaError(fn, rc)


def _stream_ptr(t):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _check_buf(t, shape, dtype, device, name):
    """A caller-supplied buffer must be exactly what the library will write."""
    if (not isinstance(t, torch.Tensor) or tuple(t.shape) != tuple(shape) or t.dtype != dtype
            or t.device != device or not t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} "
                         f"on {device}")
    return t


def _out_or_new(t, shape, dtype, device, name):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    return _check_buf(t, shape, dtype, device, name)


def _check_qkv(*ts):
    q = ts[0]
    if q.dim() != 4:
        raise ValueError("expected (batch, seqlen, heads, headdim) tensors")
    for t in ts:
        if t.shape != q.shape:
            raise ValueError("all tensors must have the shape of q")
        if t.dtype != torch.bfloat16:
            raise TypeError("tensors must be bfloat16")
        if not t.is_cuda or t.device != q.device:
            raise ValueError("tensors must live on the same CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def dfa_forward(q, k, v, block_size, out=None, lse=None):
    """Block-diffusion attention forward.  q, k, v: (B, 2n, H, d) bf16 CUDA.

    Returns (out, lse) with out (B, 2n, H, d) bf16 and lse (B, H, 2n) fp32.
    """
    _check_qkv(q, k, v)
    B, L, H, d = q.shape
    if L % 2:
        raise ValueError("the sequence must be [noisy | clean] with an even length 2n")
    out = _out_or_new(out, q.shape, torch.bfloat16, q.device, "out")
    lse = _out_or_new(lse, (B, H, L), torch.float32, q.device, "lse")
    with torch.cuda.device(q.device):
        rc = lib().dfa_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, L // 2, H, d,
                               int(block_size), _stream_ptr(q))
    _check("dfa_forward", rc)
    return out, lse


def dfa_backward(q, k, v, out, dout, lse, block_size, dq=None, dk=None, dv=None):
    """Block-diffusion attention backward; returns (dq, dk, dv) bf16."""
    _check_qkv(q, k, v, out, dout)
    B, L, H, d = q.shape
    if L % 2:
        raise ValueError("the sequence must be [noisy | clean] with an even length 2n")
    _check_buf(lse, (B, H, L), torch.float32, q.device, "lse")
    dq = _out_or_new(dq, q.shape, torch.bfloat16, q.device, "dq")
    dk = _out_or_new(dk, k.shape, torch.bfloat16, q.device, "dk")
    dv = _out_or_new(dv, v.shape, torch.bfloat16, q.device, "dv")
    with torch.cuda.device(q.device):
        rc = lib().dfa_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                                _ptr(dq), _ptr(dk), _ptr(dv), B, L // 2, H, d, int(block_size),
                                _stream_ptr(q))
    _check("dfa_backward", rc)
    return dq, dk, dv


def _check_grouped(q, k, v, *more):
    """q (and ``more``) share one shape, k and v another with fewer heads."""
    _check_qkv(q, *more)
    _check_qkv(k, v)
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("expected (batch, seqlen, heads, headdim) tensors")
    if k.device != q.device:
        raise ValueError("tensors must live on the same CUDA device")
    B, L, H, d = q.shape
    Hk = k.shape[2]
    if k.shape[0] != B or k.shape[1] != L or k.shape[3] != d:
        raise ValueError("k and v must be (batch, seqlen, kv_heads, headdim) like q")
    if Hk < 1 or H % Hk:
        raise ValueError("kv_heads must divide the query heads")
    return Hk


def dfa_forward_gqa(q, k, v, block_size, out=None, lse=None):
    """Forward with grouped key/value heads: q (B, 2n, H, d), k, v (B, 2n, Hk, d).

    Query head h reads key/value head h // (H // Hk).  Returns (out, lse)
    like :func:`dfa_forward`.
    """
    Hk = _check_grouped(q, k, v)
    B, L, H, d = q.shape
    if L % 2:
        raise ValueError("the sequence must be [noisy | clean] with an even length 2n")
    out = _out_or_new(out, q.shape, torch.bfloat16, q.device, "out")
    lse = _out_or_new(lse, (B, H, L), torch.float32, q.device, "lse")
    with torch.cuda.device(q.device):
        rc = lib().dfa_forward_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, L // 2, H,
                                   Hk, d, int(block_size), _stream_ptr(q))
    _check("dfa_forward_gqa", rc)
    return out, lse


def dfa_backward_gqa(q, k, v, out, dout, lse, block_size, dq=None, dk=None, dv=None):
    """Backward with grouped key/value heads; dk, dv have the shape of k.

    The gradient of a key/value head sums over its query heads.
    """
    Hk = _check_grouped(q, k, v, out, dout)
    B, L, H, d = q.shape
    if L % 2:
        raise ValueError("the sequence must be [noisy | clean] with an even length 2n")
    _check_buf(lse, (B, H, L), torch.float32, q.device, "lse")
    dq = _out_or_new(dq, q.shape, torch.bfloat16, q.device, "dq")
    dk = _out_or_new(dk, k.shape, torch.bfloat16, q.device, "dk")
    dv = _out_or_new(dv, v.shape, torch.bfloat16, q.device, "dv")
    with torch.cuda.device(q.device):
        rc = lib().dfa_backward_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                                    _ptr(dq), _ptr(dk), _ptr(dv), B, L // 2, H, Hk, d,
                                    int(block_size), _stream_ptr(q))
    _check("dfa_backward_gqa", rc)
    return dq, dk, dv


def _cu_array(cu_seqlens, rows):
    """Host int32 copy of cu_seqlens (list, NumPy array or tensor) as a ctypes array."""
    if isinstance(cu_seqlens, torch.Tensor):
        cu_seqlens = cu_seqlens.detach().cpu().tolist()
    cu = [int(x) for x in cu_seqlens]
    if len(cu) < 1 or cu[0] != 0 or cu[-1] != rows:
        raise ValueError("cu_seqlens must start at 0 and end at the packed rows")
    return (ctypes.c_int * len(cu))(*cu), len(cu) - 1


def _check_packed(q, k, v, *more):
    for t in (q, k, v) + more:
        if t.dim() != 3:
            raise ValueError("expected packed (rows, heads, headdim) tensors")
    _check_qkv(q[None], *(t[None] for t in more))
    _check_qkv(k[None], v[None])
    if k.device != q.device or k.shape[0] != q.shape[0] or k.shape[2] != q.shape[2]:
        raise ValueError("k and v must be (rows, kv_heads, headdim) like q")
    if k.shape[1] < 1 or q.shape[1] % k.shape[1]:
        raise ValueError("kv_heads must divide the query heads")
    return k.shape[1]


def dfa_forward_varlen(q, k, v, cu_seqlens, block_size, out=None, lse=None):
    """Forward on a packed batch: q (rows, H, d), k, v (rows, Hk, d) bf16 CUDA.

    ``cu_seqlens`` (host: list, array or tensor) holds batch + 1 prefix sums;
    every sample length is even ([noisy | clean]).  Returns out (rows, H, d)
    and lse (H, rows) float32.
    """
    Hk = _check_packed(q, k, v)
    rows, H, d = q.shape
    cu, batch = _cu_array(cu_seqlens, rows)
    out = _out_or_new(out, q.shape, torch.bfloat16, q.device, "out")
    lse = _out_or_new(lse, (H, rows), torch.float32, q.device, "lse")
    with torch.cuda.device(q.device):
        rc = lib().dfa_forward_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), cu, batch,
                                      H, Hk, d, int(block_size), _stream_ptr(q))
    _check("dfa_forward_varlen", rc)
    return out, lse


def dfa_backward_varlen(q, k, v, out, dout, lse, cu_seqlens, block_size, dq=None, dk=None,
                        dv=None):
    """Backward on a packed batch; returns (dq, dk, dv) bf16."""
    Hk = _check_packed(q, k, v, out, dout)
    rows, H, d = q.shape
    _check_buf(lse, (H, rows), torch.float32, q.device, "lse")
    cu, batch = _cu_array(cu_seqlens, rows)
    dq = _out_or_new(dq, q.shape, torch.bfloat16, q.device, "dq")
    dk = _out_or_new(dk, k.shape, torch.bfloat16, q.device, "dk")
    dv = _out_or_new(dv, v.shape, torch.bfloat16, q.device, "dv")
    with torch.cuda.device(q.device):
        rc = lib().dfa_backward_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout),
                                       _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), cu, batch, H, Hk,
                                       d, int(block_size), _stream_ptr(q))
    _check("dfa_backward_varlen", rc)
    return dq, dk, dv


def dfa_forward_fp8(q, k, v, q_descale, k_descale, v_descale, block_size, out=None, lse=None):
    """FP8 forward: q (B, 2n, H, 128), k, v (B, 2n, Hk, 128) float8_e4m3fn CUDA tensors.

    The attention of q * q_descale, k * k_descale, v * v_descale; returns
    out (B, 2n, H, 128) bf16 and lse (B, H, 2n) float32.
    """
    for t in (q, k, v):
        if t.dtype != torch.float8_e4m3fn or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous float8_e4m3fn CUDA tensors")
    if q.dim() != 4 or k.shape != v.shape or k.shape[:2] != q.shape[:2] or k.shape[3] != q.shape[3]:
        raise ValueError("q (B, 2n, H, d), k and v (B, 2n, Hk, d)")
    B, L, H, d = q.shape
    Hk = k.shape[2]
    if L % 2 or H % Hk:
        raise ValueError("even 2n and kv_heads dividing heads required")
    if k.device != q.device or v.device != q.device:
        raise ValueError("q, k, v must live on the same CUDA device")
    out = _out_or_new(out, q.shape, torch.bfloat16, q.device, "out")
    lse = _out_or_new(lse, (B, H, L), torch.float32, q.device, "lse")
    with torch.cuda.device(q.device):
        rc = lib().dfa_forward_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                   float(q_descale), float(k_descale), float(v_descale), B, L // 2,
                                   H, Hk, d, int(block_size), _stream_ptr(q))
    _check("dfa_forward_fp8", rc)
    return out, lse


def dfa_fp8_transpose_v(v, vt=None):
    """V^T of an e4m3 v (B, 2n, Hk, 128) for dfa_forward_fp8_vt (a uint8 tensor).

    A caller-supplied ``vt`` must be a contiguous uint8 tensor on v's device
    with exactly dfa_fp8_vt_bytes(B, n, Hk, 128) elements.
    """
    if (v.dtype != torch.float8_e4m3fn or v.dim() != 4 or not v.is_contiguous()
            or not v.is_cuda):
        raise ValueError("v must be a contiguous float8_e4m3fn (B, 2n, Hk, 128) CUDA tensor")
    B, L, Hk, d = v.shape
    if L % 2:
        raise ValueError("the sequence must be [noisy | clean] with an even length 2n")
    nbytes = lib().dfa_fp8_vt_bytes(B, L // 2, Hk, d)
    if nbytes < 0:
        raise DfaError("dfa_fp8_vt_bytes", int(nbytes))
    vt = _out_or_new(vt, (int(nbytes),), torch.uint8, v.device, "vt")
    with torch.cuda.device(v.device):
        rc = lib().dfa_fp8_transpose_v(_ptr(v), _ptr(vt), B, L // 2, Hk, d, _stream_ptr(v))
    _check("dfa_fp8_transpose_v", rc)
    return vt


def dfa_forward_fp8_vt(q, k, vt, kv_heads, q_descale, k_descale, v_descale, block_size,
                       out=None, lse=None):
    """dfa_forward_fp8 on a V^T from dfa_fp8_transpose_v (no scratch).

    ``kv_heads`` must equal k.shape[2]; ``vt`` must be the uint8 tensor
    dfa_fp8_transpose_v wrote for a v of k's shape.
    """
    for t in (q, k):
        if t.dtype != torch.float8_e4m3fn or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k must be contiguous float8_e4m3fn CUDA tensors")
    if q.dim() != 4 or k.dim() != 4 or k.shape[:2] != q.shape[:2] or k.shape[3] != q.shape[3]:
        raise ValueError("q (B, 2n, H, d), k (B, 2n, Hk, d)")
    if k.device != q.device:
        raise ValueError("q and k must live on the same CUDA device")
    B, L, H, d = q.shape
    if L % 2:
        raise ValueError("the sequence must be [noisy | clean] with an even length 2n")
    Hk = k.shape[2]
    if int(kv_heads) != Hk:
        raise ValueError(f"kv_heads ({kv_heads}) must equal k.shape[2] ({Hk})")
    if H % Hk:
        raise ValueError("kv_heads must divide the query heads")
    nbytes = lib().dfa_fp8_vt_bytes(B, L // 2, Hk, d)
    if nbytes < 0:
        raise DfaError("dfa_fp8_vt_bytes", int(nbytes))
    _check_buf(vt, (int(nbytes),), torch.uint8, q.device, "vt")
    out = _out_or_new(out, q.shape, torch.bfloat16, q.device, "out")
    lse = _out_or_new(lse, (B, H, L), torch.float32, q.device, "lse")
    with torch.cuda.device(q.device):
        rc = lib().dfa_forward_fp8_vt(_ptr(q), _ptr(k), _ptr(vt), _ptr(out), _ptr(lse),
                                      float(q_descale), float(k_descale), float(v_descale), B,
                                      L // 2, H, Hk, d, int(block_size), _stream_ptr(q))
    _check("dfa_forward_fp8_vt", rc)
    return out, lse


def dfa_backward_ex(q, k, v, out, dout, lse, block_size, cu_seqlens=None, deterministic=False,
                    dq=None, dk=None, dv=None, noisy_diag_pass=False):
    """Backward with options: batched (q 4-D) or packed (q 3-D, ``cu_seqlens``).

    ``deterministic``: dQ contributions are added in a fixed order, so the
    results are bitwise reproducible.  ``noisy_diag_pass``: the noisy key
    tiles in a launch of their own before the clean ones, where the block
    size allows it (DFA_NOISY_DIAG_PASS).
    """
    if cu_seqlens is None:
        Hk = _check_grouped(q, k, v, out, dout)
        B, L, H, d = q.shape
        if lse.shape != (B, H, L):
            raise ValueError("lse must be (B, H, 2n)")
        cu, batch, n = None, B, L // 2
    else:
        Hk = _check_packed(q, k, v, out, dout)
        rows, H, d = q.shape
        if lse.shape != (H, rows):
            raise ValueError("lse must be (heads, rows)")
        cu, batch = _cu_array(cu_seqlens, rows)
        n = 0
    if lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    flags = (DFA_DETERMINISTIC if deterministic else 0) | \
        (DFA_NOISY_DIAG_PASS if noisy_diag_pass else 0)
    with torch.cuda.device(q.device):
        rc = lib().dfa_backward_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                                   _ptr(dq), _ptr(dk), _ptr(dv), cu, batch, n, H, Hk, d,
                                   int(block_size), flags, _stream_ptr(q))
    _check("dfa_backward_ex", rc)
    return dq, dk, dv


def dfa_causal_forward(q, k, v, out=None, lse=None):
    """Causal attention on (Bc, L, H, d), any Bc: the yardstick."""
    _check_qkv(q, k, v)
    B, L, H, d = q.shape
    out = _out_or_new(out, q.shape, torch.bfloat16, q.device, "out")
    lse = _out_or_new(lse, (B, H, L), torch.float32, q.device, "lse")
    with torch.cuda.device(q.device):
        rc = lib().dfa_causal_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, L, H, d,
                                      _stream_ptr(q))
    _check("dfa_causal_forward", rc)
    return out, lse


def dfa_causal_backward(q, k, v, out, dout, lse, dq=None, dk=None, dv=None):
    _check_qkv(q, k, v, out, dout)
    B, L, H, d = q.shape
    _check_buf(lse, (B, H, L), torch.float32, q.device, "lse")
    dq = _out_or_new(dq, q.shape, torch.bfloat16, q.device, "dq")
    dk = _out_or_new(dk, k.shape, torch.bfloat16, q.device, "dk")
    dv = _out_or_new(dv, v.shape, torch.bfloat16, q.device, "dv")
    with torch.cuda.device(q.device):
        rc = lib().dfa_causal_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout),
                                       _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), B, L, H, d,
                                       _stream_ptr(q))
    _check("dfa_causal_backward", rc)
    return dq, dk, dv


def _ptr_or_null(t):
    return ctypes.c_void_p(None) if t is None else _ptr(t)


def _step_shape(q, mode):
    """(batch, n, rows per batch entry) of a step-API tensor for `mode`.

    Diffusion: q is (B, 2n, H, d); causal: q is (Bc, n, H, d), Bc sequences.
    """
    B, L, H, d = q.shape
    if mode == MODE_CAUSAL:
        return B, L, L
    if mode != MODE_DIFFUSION:
        raise ValueError("mode must be MODE_DIFFUSION or MODE_CAUSAL")
    if L % 2:
        raise ValueError("the sequence must be [noisy | clean] with an even length 2n")
    return B, L // 2, L


def _check_scratch(q, lse, delta, dq_acc):
    B, L, H, d = q.shape
    if lse is not None:
        _check_buf(lse, (B, H, L), torch.float32, q.device, "lse")
    if delta is not None:
        _check_buf(delta, (B, H, L), torch.float32, q.device, "delta")
    if dq_acc is not None:
        _check_buf(dq_acc, q.shape, torch.float32, q.device, "dq_acc")


def dfa_fwd_main(q, k, v, out, lse, dq_acc, block_size, mode=MODE_DIFFUSION):
    """The forward step; also zeroes dq_acc (float32, shape of q) unless None.

    Diffusion: q, k, v, out (B, 2n, H, d) bf16, lse (B, H, 2n) fp32.  Causal:
    q, k, v, out (Bc, n, H, d), lse (Bc, H, n), as dfa_causal_forward.
    """
    _check_qkv(q, k, v, out)
    B, n, L = _step_shape(q, mode)
    H, d = q.shape[2], q.shape[3]
    _check_scratch(q, lse, None, dq_acc)
    with torch.cuda.device(q.device):
        rc = lib().dfa_fwd_main(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                _ptr_or_null(dq_acc), B, n, H, d, int(block_size), int(mode),
                                _stream_ptr(q))
    _check("dfa_fwd_main", rc)


def dfa_bwd_preprocess(out, dout, delta, dq_acc, mode=MODE_DIFFUSION):
    """Step 1 of the backward: delta = rowsum(dout * out); dq_acc = 0 unless None."""
    _check_qkv(out, dout)
    B, n, L = _step_shape(out, mode)
    H, d = out.shape[2], out.shape[3]
    _check_scratch(out, None, delta, dq_acc)
    with torch.cuda.device(out.device):
        rc = lib().dfa_bwd_preprocess_ex(_ptr(out), _ptr(dout), _ptr(delta),
                                         _ptr_or_null(dq_acc), B, n, H, d, int(mode),
                                         _stream_ptr(out))
    _check("dfa_bwd_preprocess_ex", rc)


def dfa_bwd_main(q, k, v, dout, lse, delta, dq_acc, dk, dv, block_size, mode=MODE_DIFFUSION):
    """Step 2 of the backward: the tensor-core kernel (dk, dv, dq_acc += dq)."""
    _check_qkv(q, k, v, dout, dk, dv)
    B, n, L = _step_shape(q, mode)
    H, d = q.shape[2], q.shape[3]
    _check_scratch(q, lse, delta, dq_acc)
    with torch.cuda.device(q.device):
        rc = lib().dfa_bwd_main(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(lse), _ptr(delta),
                                _ptr(dq_acc), _ptr(dk), _ptr(dv), B, n, H, d,
                                int(block_size), int(mode), _stream_ptr(q))
    _check("dfa_bwd_main", rc)


def dfa_fwd_main_gqa(q, k, v, out, lse, dq_acc, block_size, mode=MODE_DIFFUSION):
    """dfa_fwd_main with k, v of fewer heads (grouped key/value heads)."""
    Hk = _check_grouped(q, k, v, out)
    B, n, L = _step_shape(q, mode)
    H, d = q.shape[2], q.shape[3]
    _check_scratch(q, lse, None, dq_acc)
    with torch.cuda.device(q.device):
        rc = lib().dfa_fwd_main_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                    _ptr_or_null(dq_acc), B, n, H, Hk, d, int(block_size),
                                    int(mode), _stream_ptr(q))
    _check("dfa_fwd_main_gqa", rc)


def dfa_bwd_main_gqa(q, k, v, dout, lse, delta, dq_acc, dk, dv, block_size, mode=MODE_DIFFUSION):
    """dfa_bwd_main with k, v, dk, dv of fewer heads (grouped key/value heads)."""
    Hk = _check_grouped(q, k, v, dout)
    B, n, L = _step_shape(q, mode)
    H, d = q.shape[2], q.shape[3]
    _check_scratch(q, lse, delta, dq_acc)
    _check_buf(dk, k.shape, torch.bfloat16, q.device, "dk")
    _check_buf(dv, v.shape, torch.bfloat16, q.device, "dv")
    with torch.cuda.device(q.device):
        rc = lib().dfa_bwd_main_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(lse),
                                    _ptr(delta), _ptr(dq_acc), _ptr(dk), _ptr(dv), B, n, H,
                                    Hk, d, int(block_size), int(mode), _stream_ptr(q))
    _check("dfa_bwd_main_gqa", rc)


def dfa_bwd_main_ex(q, k, v, dout, lse, delta, dq_acc, dk, dv, block_size, mode=MODE_DIFFUSION,
                    noisy_diag_pass=False):
    """dfa_bwd_main_gqa with flags (``noisy_diag_pass``: DFA_NOISY_DIAG_PASS)."""
    Hk = _check_grouped(q, k, v, dout)
    B, n, L = _step_shape(q, mode)
    H, d = q.shape[2], q.shape[3]
    _check_scratch(q, lse, delta, dq_acc)
    _check_buf(dk, k.shape, torch.bfloat16, q.device, "dk")
    _check_buf(dv, v.shape, torch.bfloat16, q.device, "dv")
    flags = DFA_NOISY_DIAG_PASS if noisy_diag_pass else 0
    with torch.cuda.device(q.device):
        rc = lib().dfa_bwd_main_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(lse),
                                   _ptr(delta), _ptr(dq_acc), _ptr(dk), _ptr(dv), B, n, H,
                                   Hk, d, int(block_size), int(mode), flags, _stream_ptr(q))
    _check("dfa_bwd_main_ex", rc)


def dfa_bwd_dq_convert(dq_acc, dq, mode=MODE_DIFFUSION):
    """Step 3 of the backward: dq = bf16(dq_acc)."""
    _check_qkv(dq)
    B, n, L = _step_shape(dq, mode)
    H, d = dq.shape[2], dq.shape[3]
    _check_scratch(dq, None, None, dq_acc)
    with torch.cuda.device(dq.device):
        rc = lib().dfa_bwd_dq_convert_ex(_ptr(dq_acc), _ptr(dq), B, n, H, d, int(mode),
                                         _stream_ptr(dq))
    _check("dfa_bwd_dq_convert_ex", rc)


def dfa_selftest_wait_timeout(limit_us=20000):
    """Run the bounded-wait self-test on the current stream (see dfa.h)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        rc = lib().dfa_selftest_wait_timeout(int(limit_us),
                                             ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    _check("dfa_selftest_wait_timeout", rc)


def dfa_status(device=None):
    """Synchronise the current stream and return (and clear) the device status code."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        return lib().dfa_status(ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))


# ------------------------------------------------------------- geometry

def dfa_fwd_segments(mode, n, block_size, block_m, block_n, q_half, q_tile):
    buf = (_I * 8)()
    cnt = lib().dfa_fwd_segments(mode, n, block_size, block_m, block_n, q_half, q_tile, buf)
    _check("dfa_fwd_segments", 0 if cnt >= 0 else cnt)
    return [tuple(buf[4 * i:4 * i + 4]) for i in range(cnt)]


def dfa_bwd_segments(mode, n, block_size, block_m, block_n, k_half, k_tile):
    buf = (_I * 8)()
    cnt = lib().dfa_bwd_segments(mode, n, block_size, block_m, block_n, k_half, k_tile, buf)
    _check("dfa_bwd_segments", 0 if cnt >= 0 else cnt)
    return [tuple(buf[4 * i:4 * i + 4]) for i in range(cnt)]


def dfa_tile_full(rule, n, block_size, q_start, block_m, k_start, block_n):
    return lib().dfa_tile_full(rule, n, block_size, q_start, block_m, k_start, block_n)


def dfa_tile_visits(mode, n, block_size, block_m, block_n, pass_):
    return lib().dfa_tile_visits(mode, n, block_size, block_m, block_n, pass_)


def dfa_work_item(pass_, mode, w, batch, heads, tiles, group):
    """(batch, head, half, tile) of the w-th work item of a pass (0 forward, 1 backward)."""
    buf = (_I * 4)()
    _check("dfa_work_item", lib().dfa_work_item(pass_, mode, w, batch, heads, tiles, group, buf))
    return tuple(buf)


def dfa_tile_shape(headdim):
    vals = [_I() for _ in range(4)]
    _check("dfa_tile_shape", lib().dfa_tile_shape(headdim, *[ctypes.byref(x) for x in vals]))
    return tuple(x.value for x in vals)

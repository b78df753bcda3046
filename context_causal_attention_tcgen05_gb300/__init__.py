"""Python binding of libcp_attn.so (causal context-parallel attention on one GB300).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  Functions carry the C ABI's names
(``include/cp_attn.h``), take torch CUDA tensors, pass their device pointers
and the current CUDA stream, and raise :class:`CpAttnError` when the library
refuses a call.  Output tensors and workspaces are allocated here with torch
(the library itself allocates nothing).  There is no fallback: if the library
is missing or cannot load, importing the functions raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

# CP_ATTN_LIBRARY may name another build of the library (the index-checking debug
# build, libcp_attn_debug.so); it must exist: there is no fallback either way.
LIB_PATH = os.environ.get("CP_ATTN_LIBRARY") or os.path.join(os.path.dirname(os.path.abspath(__file__)),
                                                            "libcp_attn.so")

__all__ = [
    "CpAttnError", "load_library", "library_path", "header_functions",
    "cp_attn_block_fwd", "cp_attn_block_bwd", "cp_attn_block_bwd_typed", "cp_attn_block_bwd_noalloc",
    "cp_lse_merge",
    "cp_ulysses_seq2head", "cp_ulysses_head2seq",
    "cp_zigzag_reorder", "cp_zigzag_restore", "cp_striped_reorder", "cp_striped_restore",
    "cp_lse_reorder", "cp_ring_reorder_qkv", "cp_ring_restore",
    "cp_ring_attention", "cp_ring_attention_reordered", "cp_ring_attention_reordered_to_seq",
    "cp_ring_attention_bwd", "cp_ulysses_attention",
    "cp_ulysses_attention_bwd", "cp_usp_attention",
    "cp_workspace_size", "cp_check_device_status", "cp_debug_bounded_wait",
    "cp_status_string", "cp_last_error", "cp_version",
    "CP_F32", "CP_BF16", "REORDER", "RING_MODE", "OP",
]

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "cp_attn.h")

CP_F32, CP_BF16 = 0, 1
REORDER = {"contiguous": 0, "dual_chunk_swap": 1, "zigzag": 1, "striped": 2, "auto": 3}
RING_MODE = {"fused": 0, "stepwise": 1}
OP = {"ring_fwd": 0, "ring_bwd": 1, "ulysses_fwd": 2, "block_bwd": 3, "ring_fwd_reordered": 4,
      "ulysses_bwd": 5, "usp_fwd": 6}

_c_i32, _c_i64, _c_f32, _c_p, _c_size = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t


class cp_mask(ctypes.Structure):
    _fields_ = [("causal", _c_i32), ("q_offset", _c_i64), ("k_offset", _c_i64),
                ("q_stride", _c_i64), ("k_stride", _c_i64), ("cu_seqlens", _c_p), ("n_docs", _c_i32),
                ("window", _c_i32)]


_SIGS = {
    "cp_attn_block_fwd": [_c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32,
                          ctypes.POINTER(cp_mask), _c_f32, _c_p, _c_p, _c_p],
    "cp_attn_block_bwd": [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i32, _c_i32, _c_i32,
                          _c_i32, ctypes.POINTER(cp_mask), _c_f32, _c_p, _c_p, _c_p, _c_i32, _c_p, _c_size,
                          _c_p],
    "cp_attn_block_bwd_typed": [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i32, _c_i32, _c_i32,
                                _c_i32, ctypes.POINTER(cp_mask), _c_f32, _c_p, _c_p, _c_p, _c_p, _c_size, _c_p],
    "cp_attn_block_bwd_noalloc": [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i32, _c_i32,
                                  _c_i32, _c_i32, ctypes.POINTER(cp_mask), _c_f32, _c_p, _c_p, _c_p, _c_p],
    "cp_lse_merge": [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_p],
    "cp_ulysses_seq2head": [_c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_p],
    "cp_ulysses_head2seq": [_c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_p],
    "cp_zigzag_reorder": [_c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_p],
    "cp_zigzag_restore": [_c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_p],
    "cp_striped_reorder": [_c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_p],
    "cp_striped_restore": [_c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_p],
    "cp_lse_reorder": [_c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_p],
    "cp_ring_reorder_qkv": [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32,
                            _c_i32, _c_i32, _c_p],
    "cp_ring_restore": [_c_p, _c_p, _c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_p],
    "cp_ring_attention": [_c_p, _c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                          _c_i32, _c_p, _c_i32, _c_p, _c_p, _c_p, _c_size, _c_p],
    "cp_ring_attention_reordered": [_c_p, _c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                                    _c_i32, _c_i32, _c_p, _c_i32, _c_p, _c_p, _c_p, _c_size, _c_p],
    "cp_ring_attention_reordered_to_seq": [_c_p, _c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                                           _c_i32, _c_p, _c_i32, _c_p, _c_p, _c_p],
    "cp_ring_attention_bwd": [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32,
                              _c_i32, _c_i32, _c_i32, _c_p, _c_i32, _c_p, _c_p, _c_p, _c_p, _c_size, _c_p],
    "cp_ulysses_attention": [_c_p, _c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_p,
                             _c_i32, _c_i32, _c_p, _c_p, _c_p, _c_size, _c_p],
    "cp_ulysses_attention_bwd": [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32,
                                 _c_i32, _c_i32, _c_p, _c_i32, _c_i32, _c_p, _c_p, _c_p, _c_p, _c_size, _c_p],
    "cp_usp_attention": [_c_p, _c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                         _c_p, _c_i32, _c_p, _c_p, _c_p, _c_size, _c_p],
    "cp_workspace_size": [_c_i32, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                          ctypes.POINTER(_c_size)],
    "cp_check_device_status": [_c_p],
    "cp_debug_bounded_wait": [_c_i32, _c_p],
    "cp_status_string": [_c_i32],
    "cp_last_error": [],
    "cp_version": [],
}
_STR_RET = {"cp_status_string", "cp_last_error", "cp_version"}

_lib = None


class CpAttnError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn} failed: {status} ({_status_name(status)}): {message}")
        self.status = status
        self.fn = fn


def library_path() -> str:
    return LIB_PATH


def load_library():
    """Loads libcp_attn.so (built in-tree by build_lib).  Raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m context_causal_attention_tcgen05_gb300.build_lib`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, args in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_char_p if name in _STR_RET else ctypes.c_int32
    _lib = lib
    return lib


def header_functions() -> list[str]:
    """Function names declared in include/cp_attn.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"CP_API\s+(?:cp_status|const char\*)\s+(cp_\w+)\s*\(", text)))


def _status_name(st: int) -> str:
    try:
        return load_library().cp_status_string(st).decode()
    except Exception:  # pragma: no cover - only for error formatting
        return "?"


def _check(fn: str, st: int):
    if st != 0:
        raise CpAttnError(fn, st, load_library().cp_last_error().decode())


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return CP_F32
    if t.dtype == torch.bfloat16:
        return CP_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _mask(causal=True, q_offset=0, k_offset=0, q_stride=1, k_stride=1, cu_seqlens=None, window=0):
    m = cp_mask()
    m.causal = int(bool(causal))
    m.window = int(window)
    m.q_offset, m.k_offset = int(q_offset), int(k_offset)
    m.q_stride, m.k_stride = int(q_stride), int(k_stride)
    if cu_seqlens is not None:
        assert cu_seqlens.dtype == torch.int32 and cu_seqlens.is_cuda
        m.cu_seqlens = cu_seqlens.data_ptr()
        m.n_docs = cu_seqlens.numel() - 1
    else:
        m.cu_seqlens = None
        m.n_docs = 0
    return m


def cp_workspace_size(op: str, S: int, Hq: int, Hkv: int, D: int, dtype, P: int, mode: str = "fused") -> int:
    dt = dtype if isinstance(dtype, int) else (CP_F32 if dtype == torch.float32 else CP_BF16)
    out = ctypes.c_size_t(0)
    _check("cp_workspace_size", load_library().cp_workspace_size(
        OP[op], S, Hq, Hkv, D, dt, P, RING_MODE[mode], ctypes.byref(out)))
    return out.value


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


def cp_attn_block_fwd(q, k, v, causal=True, q_offset=0, k_offset=0, q_stride=1, k_stride=1,
                      cu_seqlens=None, scale=0.0, out=None, lse=None, stream=None, window=0):
    """out [Sq,Hq,D], lse [Hq,Sq] (fp32) of one block pair."""
    Sq, Hq, D = q.shape
    Sk, Hkv, _ = k.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(Hq, Sq, dtype=torch.float32, device=q.device)
    m = _mask(causal, q_offset, k_offset, q_stride, k_stride, cu_seqlens, window)
    _check("cp_attn_block_fwd", load_library().cp_attn_block_fwd(
        _ptr(q), _ptr(k), _ptr(v), Sq, Sk, Hq, Hkv, D, _dt(q), ctypes.byref(m), float(scale),
        _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def cp_attn_block_bwd(q, k, v, out, dout, lse, causal=True, q_offset=0, k_offset=0, q_stride=1,
                      k_stride=1, cu_seqlens=None, scale=0.0, dq_acc=None, dk_acc=None, dv_acc=None,
                      accumulate=False, workspace=None, stream=None, window=0):
    """fp32 (dq_acc, dk_acc, dv_acc) of one block pair given the FINAL out and lse:
    overwritten, or (accumulate=True) this pair's gradients added to what they hold."""
    Sq, Hq, D = q.shape
    Sk, Hkv, _ = k.shape
    f32 = dict(dtype=torch.float32, device=q.device)
    dq_acc = torch.empty(Sq, Hq, D, **f32) if dq_acc is None else dq_acc
    dk_acc = torch.empty(Sk, Hkv, D, **f32) if dk_acc is None else dk_acc
    dv_acc = torch.empty(Sk, Hkv, D, **f32) if dv_acc is None else dv_acc
    for t in (dq_acc, dk_acc, dv_acc):
        if t.dtype != torch.float32:
            raise TypeError("the accumulating block backward takes fp32 gradient buffers")
    if workspace is None:
        workspace = _workspace(cp_workspace_size("block_bwd", max(Sq, Sk), Hq, Hkv, D, q.dtype, 1), q.device)
    m = _mask(causal, q_offset, k_offset, q_stride, k_stride, cu_seqlens, window)
    _check("cp_attn_block_bwd", load_library().cp_attn_block_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), Sq, Sk, Hq, Hkv, D, _dt(q),
        ctypes.byref(m), float(scale), _ptr(dq_acc), _ptr(dk_acc), _ptr(dv_acc), int(bool(accumulate)),
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return dq_acc, dk_acc, dv_acc


def cp_attn_block_bwd_typed(q, k, v, out, dout, lse, causal=True, q_offset=0, k_offset=0, q_stride=1,
                            k_stride=1, cu_seqlens=None, scale=0.0, stream=None, window=0):
    """(dq, dk, dv) in the input dtype of one block pair given the final out and lse."""
    Sq, Hq, D = q.shape
    Sk, Hkv, _ = k.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = _workspace(cp_workspace_size("block_bwd", max(Sq, Sk), Hq, Hkv, D, q.dtype, 1), q.device)
    m = _mask(causal, q_offset, k_offset, q_stride, k_stride, cu_seqlens, window)
    _check("cp_attn_block_bwd_typed", load_library().cp_attn_block_bwd_typed(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), Sq, Sk, Hq, Hkv, D, _dt(q),
        ctypes.byref(m), float(scale), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(),
        _stream(stream)))
    return dq, dk, dv


def cp_attn_block_bwd_noalloc(q, k, v, out, dout, lse, causal=True, q_offset=0, k_offset=0,
                              q_stride=1, k_stride=1, cu_seqlens=None, scale=0.0, dq=None, dk=None,
                              dv=None, stream=None, window=0):
    """cp_attn_block_bwd_typed without a workspace: the library uses its built-in
    32 MiB scratch array and allocates no device memory (outputs are allocated
    here unless passed in)."""
    Sq, Hq, D = q.shape
    Sk, Hkv, _ = k.shape
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    m = _mask(causal, q_offset, k_offset, q_stride, k_stride, cu_seqlens, window)
    _check("cp_attn_block_bwd_noalloc", load_library().cp_attn_block_bwd_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), Sq, Sk, Hq, Hkv, D, _dt(q),
        ctypes.byref(m), float(scale), _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream)))
    return dq, dk, dv


def cp_lse_merge(o1, lse1, o2, lse2, out=None, lse=None, stream=None):
    Sq, H, D = o1.shape
    if out is None:
        out = torch.empty_like(o1)
    if lse is None:
        lse = torch.empty_like(lse1)
    _check("cp_lse_merge", load_library().cp_lse_merge(
        _ptr(o1), _ptr(lse1), _ptr(o2), _ptr(lse2), _ptr(out), _ptr(lse), Sq, H, D, _dt(o1),
        _stream(stream)))
    return out, lse


def cp_ulysses_seq2head(x, P, y=None, stream=None):
    """x [S,H,D] -> y [P,S,H/P,D]."""
    S, H, D = x.shape
    if y is None:
        y = torch.empty(P, S, H // P, D, dtype=x.dtype, device=x.device)
    _check("cp_ulysses_seq2head", load_library().cp_ulysses_seq2head(
        _ptr(x), _ptr(y), S, H, D, P, _dt(x), _stream(stream)))
    return y


def cp_ulysses_head2seq(y, P, x=None, stream=None):
    """y [P,S,H/P,D] -> x [S,H,D]."""
    P_, S, Hp, D = y.shape
    assert P_ == P
    if x is None:
        x = torch.empty(S, Hp * P, D, dtype=y.dtype, device=y.device)
    _check("cp_ulysses_head2seq", load_library().cp_ulysses_head2seq(
        _ptr(y), _ptr(x), S, Hp * P, D, P, _dt(y), _stream(stream)))
    return x


def _reorder_call(name, x, P, y=None, stream=None):
    S, H, D = x.shape
    if y is None:
        y = torch.empty_like(x)
    _check(name, getattr(load_library(), name)(_ptr(x), _ptr(y), S, H, D, P, _dt(x), _stream(stream)))
    return y


def cp_zigzag_reorder(x, P, y=None, stream=None):
    return _reorder_call("cp_zigzag_reorder", x, P, y, stream)


def cp_zigzag_restore(y, P, x=None, stream=None):
    return _reorder_call("cp_zigzag_restore", y, P, x, stream)


def cp_striped_reorder(x, P, y=None, stream=None):
    return _reorder_call("cp_striped_reorder", x, P, y, stream)


def cp_striped_restore(y, P, x=None, stream=None):
    return _reorder_call("cp_striped_restore", y, P, x, stream)


def cp_lse_reorder(x, P, reorder="zigzag", inverse=False, y=None, stream=None):
    """Column permute of an lse [H,S] array into (inverse=False) or out of the ranks' layout."""
    H, S = x.shape
    if y is None:
        y = torch.empty_like(x)
    _check("cp_lse_reorder", load_library().cp_lse_reorder(
        _ptr(x), _ptr(y), S, H, P, REORDER[reorder], int(bool(inverse)), _stream(stream)))
    return y


def cp_ring_reorder_qkv(q, k, v, P, reorder="zigzag", q_re=None, k_re=None, v_re=None, stream=None):
    """q, k, v in sequence order -> the ranks' order, in one launch."""
    S, Hq, D = q.shape
    Hkv = k.shape[1]
    q_re = torch.empty_like(q) if q_re is None else q_re
    k_re = torch.empty_like(k) if k_re is None else k_re
    v_re = torch.empty_like(v) if v_re is None else v_re
    _check("cp_ring_reorder_qkv", load_library().cp_ring_reorder_qkv(
        _ptr(q), _ptr(k), _ptr(v), _ptr(q_re), _ptr(k_re), _ptr(v_re), S, Hq, Hkv, D, _dt(q), P,
        REORDER[reorder], _stream(stream)))
    return q_re, k_re, v_re


def cp_ring_restore(o_re, lse_re, P, reorder="zigzag", out=None, lse=None, stream=None):
    """The ring's out (and lse, unless lse_re is None) back to sequence order, in one launch."""
    S, Hq, D = o_re.shape
    out = torch.empty_like(o_re) if out is None else out
    if lse_re is not None and lse is None:
        lse = torch.empty_like(lse_re)
    _check("cp_ring_restore", load_library().cp_ring_restore(
        _ptr(o_re), None if lse_re is None else _ptr(lse_re), _ptr(out), None if lse is None else _ptr(lse),
        S, Hq, D, _dt(o_re), P, REORDER[reorder], _stream(stream)))
    return out, lse


def cp_ring_attention(q, k, v, P, reorder="auto", mode="fused", cu_seqlens=None, out=None, lse=None,
                      workspace=None, stream=None):
    """Ring attention over P virtual ranks; inputs/outputs in sequence order."""
    S, Hq, D = q.shape
    Hkv = k.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(Hq, S, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = _workspace(cp_workspace_size("ring_fwd", S, Hq, Hkv, D, q.dtype, P, mode), q.device)
    n_docs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    _check("cp_ring_attention", load_library().cp_ring_attention(
        _ptr(q), _ptr(k), _ptr(v), S, Hq, Hkv, D, _dt(q), P, REORDER[reorder], RING_MODE[mode],
        _ptr(cu_seqlens), n_docs, _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
        _stream(stream)))
    return out, lse


def cp_ring_attention_reordered_to_seq(q, k, v, P, reorder="zigzag", cu_seqlens=None, out=None, lse=None,
                                       stream=None):
    """Fused ring on inputs already in the ranks' layout (zigzag or contiguous); out and
    lse come back in sequence order (the restore is done by the attention's writes)."""
    S, Hq, D = q.shape
    Hkv = k.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(Hq, S, dtype=torch.float32, device=q.device)
    n_docs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    _check("cp_ring_attention_reordered_to_seq", load_library().cp_ring_attention_reordered_to_seq(
        _ptr(q), _ptr(k), _ptr(v), S, Hq, Hkv, D, _dt(q), P, REORDER[reorder], _ptr(cu_seqlens), n_docs,
        _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def cp_ring_attention_reordered(q, k, v, P, reorder="auto", mode="fused", cu_seqlens=None, out=None,
                                lse=None, workspace=None, stream=None):
    """Ring attention on inputs already in the ranks' layout; outputs stay in that layout."""
    S, Hq, D = q.shape
    Hkv = k.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(Hq, S, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = _workspace(cp_workspace_size("ring_fwd_reordered", S, Hq, Hkv, D, q.dtype, P, mode),
                               q.device)
    n_docs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    _check("cp_ring_attention_reordered", load_library().cp_ring_attention_reordered(
        _ptr(q), _ptr(k), _ptr(v), S, Hq, Hkv, D, _dt(q), P, REORDER[reorder], RING_MODE[mode],
        _ptr(cu_seqlens), n_docs, _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
        _stream(stream)))
    return out, lse


def cp_ring_attention_bwd(q, k, v, out, lse, dout, P, reorder="auto", cu_seqlens=None,
                          dq=None, dk=None, dv=None, workspace=None, stream=None):
    S, Hq, D = q.shape
    Hkv = k.shape[1]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = _workspace(cp_workspace_size("ring_bwd", S, Hq, Hkv, D, q.dtype, P), q.device)
    n_docs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    _check("cp_ring_attention_bwd", load_library().cp_ring_attention_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), S, Hq, Hkv, D, _dt(q), P,
        REORDER[reorder], _ptr(cu_seqlens), n_docs, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return dq, dk, dv


def cp_ulysses_attention(q, k, v, P, cu_seqlens=None, out=None, lse=None, workspace=None, stream=None,
                         window=0):
    S, Hq, D = q.shape
    Hkv = k.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(Hq, S, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = _workspace(cp_workspace_size("ulysses_fwd", S, Hq, Hkv, D, q.dtype, P), q.device)
    n_docs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    _check("cp_ulysses_attention", load_library().cp_ulysses_attention(
        _ptr(q), _ptr(k), _ptr(v), S, Hq, Hkv, D, _dt(q), P, _ptr(cu_seqlens), n_docs, int(window),
        _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out, lse


def cp_ulysses_attention_bwd(q, k, v, out, lse, dout, P, cu_seqlens=None, dq=None, dk=None, dv=None,
                             workspace=None, stream=None, window=0):
    """Backward of cp_ulysses_attention: (dq, dk, dv) from the forward's out and lse."""
    S, Hq, D = q.shape
    Hkv = k.shape[1]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = _workspace(cp_workspace_size("ulysses_bwd", S, Hq, Hkv, D, q.dtype, P), q.device)
    n_docs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    _check("cp_ulysses_attention_bwd", load_library().cp_ulysses_attention_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), S, Hq, Hkv, D, _dt(q), P,
        _ptr(cu_seqlens), n_docs, int(window), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return dq, dk, dv


def cp_usp_attention(q, k, v, P_ulysses, P_ring, reorder="auto", cu_seqlens=None, out=None, lse=None,
                     workspace=None, stream=None):
    """Ulysses inside groups of P_ulysses ranks x the ring across P_ring groups."""
    S, Hq, D = q.shape
    Hkv = k.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(Hq, S, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = _workspace(cp_workspace_size("usp_fwd", S, Hq, Hkv, D, q.dtype, P_ring), q.device)
    n_docs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    _check("cp_usp_attention", load_library().cp_usp_attention(
        _ptr(q), _ptr(k), _ptr(v), S, Hq, Hkv, D, _dt(q), P_ulysses, P_ring, REORDER[reorder],
        _ptr(cu_seqlens), n_docs, _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out, lse


def cp_check_device_status(stream=None) -> int:
    """Synchronises the stream; returns the library status (0 = OK) without raising."""
    return load_library().cp_check_device_status(_stream(stream))


def cp_debug_bounded_wait(timeout_us: int, stream=None):
    _check("cp_debug_bounded_wait", load_library().cp_debug_bounded_wait(int(timeout_us), _stream(stream)))


def cp_status_string(st: int) -> str:
    return load_library().cp_status_string(st).decode()


def cp_last_error() -> str:
    return load_library().cp_last_error().decode()


def cp_version() -> str:
    return load_library().cp_version().decode()

"""Thin ctypes binding of libfa.so (include/fa.h), with the same entry-point names.

Argument marshalling only: shapes are read off the tensors, pointers and the
current CUDA stream are passed through, outputs and the workspace are
allocated with torch.  Every step of attention runs in the library's kernels;
there is no fallback of any kind, and a missing library is an error.
"""
from __future__ import annotations

import ctypes
import math
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa.so")

FA_OK = 0
STATUS = {
    0: "FA_OK", 1: "FA_ERR_NULL_PTR", 2: "FA_ERR_BAD_SHAPE", 3: "FA_ERR_UNSUPPORTED_HEAD_DIM",
    4: "FA_ERR_UNSUPPORTED_DTYPE", 5: "FA_ERR_MISALIGNED", 6: "FA_ERR_WORKSPACE", 7: "FA_ERR_LAUNCH",
    8: "FA_ERR_TIMEOUT", 9: "FA_ERR_NO_DEVICE", 10: "FA_ERR_BAD_ARG",
}
FA_DTYPE_F32, FA_DTYPE_BF16 = 0, 1

# every function include/fa.h declares
EXPORTS = ("fa_fwd", "fa_bwd_workspace_size", "fa_bwd", "fa_bwd_preprocess", "fa_bwd_dkdv", "fa_bwd_dq",
           "fa_bwd_grads",
           "fa_bwd_noalloc", "fa_noalloc_scratch_bytes", "fa_path_name", "fa_get_device_status",
           "fa_reset_device_status", "fa_set_wait_limit", "fa_debug_force_stall", "fa_status_string")

_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


def lib() -> ctypes.CDLL:
    """Load the in-tree libfa.so (built by __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
    L.fa_bwd_workspace_size.argtypes = [i, i, i, i, i, i, i]
    L.fa_bwd_workspace_size.restype = sz
    L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, sz, vp]
    L.fa_bwd_preprocess.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, vp, sz, vp]
    L.fa_bwd_dkdv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, sz, vp]
    L.fa_bwd_dq.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, sz, vp]
    L.fa_bwd_grads.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, sz, vp]
    L.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
    L.fa_bwd_noalloc.restype = ctypes.c_int
    L.fa_noalloc_scratch_bytes.argtypes = []
    L.fa_noalloc_scratch_bytes.restype = sz
    L.fa_path_name.argtypes = [i, i, i, i, i]
    L.fa_path_name.restype = ctypes.c_char_p
    L.fa_get_device_status.argtypes = [vp]
    L.fa_reset_device_status.argtypes = [vp]
    L.fa_set_wait_limit.argtypes = [ctypes.c_uint32]
    L.fa_set_wait_limit.restype = None
    L.fa_debug_force_stall.argtypes = [ctypes.c_int]
    L.fa_debug_force_stall.restype = None
    L.fa_status_string.argtypes = [i]
    L.fa_status_string.restype = ctypes.c_char_p
    for name in ("fa_fwd", "fa_bwd", "fa_bwd_preprocess", "fa_bwd_dkdv", "fa_bwd_dq", "fa_bwd_grads",
                 "fa_get_device_status",
                 "fa_reset_device_status"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def check(status: int, what: str):
    if status != FA_OK:
        raise FaError(status, what)


# ------------------------------------------------------------------ tensor helpers

def _torch():
    import torch
    return torch


def dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return FA_DTYPE_F32
    if t.dtype == torch.bfloat16:
        return FA_DTYPE_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _bh(t):
    """(B, H) for a (..., N, d) tensor: (B, H) for 4-D input, else (prod(leading), 1)."""
    if t.dim() == 4:
        return t.shape[0], t.shape[1]
    return math.prod(t.shape[:-2]), 1


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _check_inputs(*ts):
    t0 = ts[0]
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous (B, H, N, d) or (..., N, d)")
        if t.dtype != t0.dtype:
            raise ValueError("Q, K, V (and O, dO) must share a dtype")


def path_name(Nq, Nk, d, is_causal, dtype_c) -> str | None:
    r = lib().fa_path_name(Nq, Nk, d, int(is_causal), dtype_c)
    return r.decode() if r else None


# ------------------------------------------------------------------ entry points

def fa_fwd(Q, K, V, is_causal=False, scale=None, O=None, L=None, stream=None):
    """O (like Q) and L (Q.shape[:-1], fp32) of attention; see include/fa.h."""
    torch = _torch()
    _check_inputs(Q, K, V)
    B, H = _bh(Q)
    Nq, d = Q.shape[-2], Q.shape[-1]
    Nk = K.shape[-2]
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if O is None:
        O = torch.empty_like(Q)
    if L is None:
        L = torch.empty(Q.shape[:-1], dtype=torch.float32, device=Q.device)
    check(lib().fa_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(L), B, H, Nq, Nk, d, sc, int(is_causal),
                       dtype_code(Q), _stream(stream)), "fa_fwd")
    return O, L


def fa_bwd_workspace_size(Q, K, is_causal=False) -> int:
    B, H = _bh(Q)
    return int(lib().fa_bwd_workspace_size(B, H, Q.shape[-2], K.shape[-2], Q.shape[-1], int(is_causal),
                                           dtype_code(Q)))


def alloc_workspace(Q, K, is_causal=False):
    torch = _torch()
    n = fa_bwd_workspace_size(Q, K, is_causal)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=Q.device)


def fa_bwd(Q, K, V, O, dO, L, is_causal=False, scale=None, dQ=None, dK=None, dV=None, workspace=None,
           stream=None):
    """dQ, dK, dV of attention given the forward's O and L; see include/fa.h."""
    torch = _torch()
    _check_inputs(Q, K, V, O, dO)
    B, H = _bh(Q)
    Nq, d = Q.shape[-2], Q.shape[-1]
    Nk = K.shape[-2]
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    ws = alloc_workspace(Q, K, is_causal) if workspace is None else workspace
    check(lib().fa_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(L), _ptr(dQ), _ptr(dK), _ptr(dV),
                       B, H, Nq, Nk, d, sc, int(is_causal), dtype_code(Q), _ptr(ws), ws.numel(),
                       _stream(stream)), "fa_bwd")
    return dQ, dK, dV


def fa_bwd_noalloc(Q, K, V, O, dO, L, is_causal=False, scale=None, dQ=None, dK=None, dV=None, stream=None):
    """fa_bwd with the library's own fixed scratch array instead of a workspace (see include/fa.h)."""
    torch = _torch()
    _check_inputs(Q, K, V, O, dO)
    B, H = _bh(Q)
    Nq, d = Q.shape[-2], Q.shape[-1]
    Nk = K.shape[-2]
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    check(lib().fa_bwd_noalloc(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(L), _ptr(dQ), _ptr(dK),
                               _ptr(dV), B, H, Nq, Nk, d, sc, int(is_causal), dtype_code(Q), _stream(stream)),
          "fa_bwd_noalloc")
    return dQ, dK, dV


def fa_bwd_preprocess(O, dO, L, Q, K, is_causal, workspace, stream=None):
    B, H = _bh(Q)
    check(lib().fa_bwd_preprocess(_ptr(O), _ptr(dO), _ptr(L), B, H, Q.shape[-2], K.shape[-2], Q.shape[-1],
                                  int(is_causal), dtype_code(Q), _ptr(workspace), workspace.numel(),
                                  _stream(stream)), "fa_bwd_preprocess")


def fa_bwd_dkdv(Q, K, V, dO, L, dQ, dK, dV, is_causal, workspace, scale=None, stream=None):
    B, H = _bh(Q)
    d = Q.shape[-1]
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    check(lib().fa_bwd_dkdv(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(L), _ptr(dQ), _ptr(dK), _ptr(dV), B, H,
                            Q.shape[-2], K.shape[-2], d, sc, int(is_causal), dtype_code(Q), _ptr(workspace),
                            workspace.numel(), _stream(stream)), "fa_bwd_dkdv")


def fa_bwd_dq(Q, K, V, dO, L, dQ, is_causal, workspace, scale=None, stream=None):
    B, H = _bh(Q)
    d = Q.shape[-1]
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    check(lib().fa_bwd_dq(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(L), _ptr(dQ), B, H, Q.shape[-2],
                          K.shape[-2], d, sc, int(is_causal), dtype_code(Q), _ptr(workspace), workspace.numel(),
                          _stream(stream)), "fa_bwd_dq")


def fa_bwd_grads(Q, K, V, dO, L, dQ, dK, dV, is_causal, workspace, scale=None, stream=None):
    B, H = _bh(Q)
    d = Q.shape[-1]
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    check(lib().fa_bwd_grads(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(L), _ptr(dQ), _ptr(dK), _ptr(dV), B, H,
                             Q.shape[-2], K.shape[-2], d, sc, int(is_causal), dtype_code(Q), _ptr(workspace),
                             workspace.numel(), _stream(stream)), "fa_bwd_grads")


def fa_get_device_status(stream=None) -> int:
    return int(lib().fa_get_device_status(_stream(stream)))


def fa_reset_device_status(stream=None):
    check(lib().fa_reset_device_status(_stream(stream)), "fa_reset_device_status")


def fa_set_wait_limit(spins: int):
    lib().fa_set_wait_limit(int(spins))


def fa_debug_force_stall(on: bool):
    lib().fa_debug_force_stall(1 if on else 0)

"""Thin ctypes binding of libfa.so (include/fa.h), with the same entry-point names.

Argument marshalling only: shapes are read off the tensors, pointers and the
current CUDA stream are passed through, outputs and the workspace are
allocated with torch.  Every step of attention runs in the library's kernels;
there is no fallback of any kind, and a missing library is an error.
"""
from __future__ import annotations

import contextlib
import ctypes
import math
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa.so")
DEBUG_LIB_PATH = os.path.join(PKG, "libfa_debug.so")

FA_OK = 0
STATUS = {
    0: "FA_OK", 1: "FA_ERR_NULL_PTR", 2: "FA_ERR_BAD_SHAPE", 3: "FA_ERR_UNSUPPORTED_HEAD_DIM",
    4: "FA_ERR_UNSUPPORTED_DTYPE", 5: "FA_ERR_MISALIGNED", 6: "FA_ERR_WORKSPACE", 7: "FA_ERR_LAUNCH",
    8: "FA_ERR_TIMEOUT", 9: "FA_ERR_NO_DEVICE", 10: "FA_ERR_BAD_ARG", 11: "FA_ERR_BOUNDS",
}
FA_DTYPE_F32, FA_DTYPE_BF16 = 0, 1
FA_DQ_AUTO, FA_DQ_SEPARATE_PASS, FA_DQ_REDUCTION = 0, 1, 2
FA_FP32_AUTO, FA_FP32_EXACT, FA_FP32_SPLIT = 0, 1, 2

# every function include/fa.h declares
EXPORTS = ("fa_fwd", "fa_bwd_workspace_size", "fa_bwd", "fa_bwd_preprocess", "fa_bwd_dkdv", "fa_bwd_dq",
           "fa_bwd_grads", "fa_fwd_strided", "fa_bwd_strided", "fa_fwd_bwd",
           "fa_bwd_noalloc", "fa_noalloc_scratch_bytes", "fa_path_name", "fa_set_fp32_mode", "fa_set_dq_strategy",
           "fa_bwd_dq_strategy", "fa_get_device_status",
           "fa_reset_device_status", "fa_set_wait_limit", "fa_debug_force_stall", "fa_debug_build",
           "fa_debug_tile_rows", "fa_debug_reset_tile_rows", "fa_status_string")

_lib = None


class FaStrides(ctypes.Structure):
    """fa_strides of include/fa.h: element strides (batch, head, row) of a (B, H, N, d) view."""
    _fields_ = [("b", ctypes.c_int64), ("h", ctypes.c_int64), ("n", ctypes.c_int64)]


class FaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


def lib() -> ctypes.CDLL:
    """The library every call of this module goes to: the in-tree libfa.so (built by
    __graft_entry__.build()), or libfa_debug.so inside a debug_library() block."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = _load(LIB_PATH)
    return _lib


_debug_lib = None


@contextlib.contextmanager
def debug_library():
    """Within the block, this module's calls go to libfa_debug.so (the same library
    built with FA_DEBUG: in-kernel bounds checks and tile-load counters)."""
    global _lib, _debug_lib
    if _debug_lib is None:
        _debug_lib = _load(DEBUG_LIB_PATH)
    prev = lib()
    _lib = _debug_lib
    try:
        yield _debug_lib
    finally:
        _lib = prev


def _load(path) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build()")
    L = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
    L.fa_bwd_workspace_size.argtypes = [i, i, i, i, i, i, i]
    L.fa_bwd_workspace_size.restype = sz
    L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, sz, vp]
    L.fa_bwd_preprocess.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, vp, sz, vp]
    L.fa_bwd_dkdv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, sz, vp]
    L.fa_bwd_dq.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, sz, vp]
    L.fa_bwd_grads.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, sz, vp]
    L.fa_fwd_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, sz, vp]
    sp = ctypes.POINTER(FaStrides)
    L.fa_fwd_strided.argtypes = [vp, sp, vp, sp, vp, sp, vp, sp, vp, i, i, i, i, i, f, i, i, vp]
    L.fa_bwd_strided.argtypes = [vp, sp, vp, sp, vp, sp, vp, sp, vp, sp, vp, vp, sp, vp, sp, vp, sp,
                                 i, i, i, i, i, f, i, i, vp, sz, vp]
    L.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
    L.fa_bwd_noalloc.restype = ctypes.c_int
    L.fa_noalloc_scratch_bytes.argtypes = []
    L.fa_noalloc_scratch_bytes.restype = sz
    L.fa_path_name.argtypes = [i, i, i, i, i]
    L.fa_path_name.restype = ctypes.c_char_p
    L.fa_set_fp32_mode.argtypes = [i]
    L.fa_set_fp32_mode.restype = i
    L.fa_set_dq_strategy.argtypes = [i]
    L.fa_set_dq_strategy.restype = i
    L.fa_bwd_dq_strategy.argtypes = [i, i, i, i, i, i, i]
    L.fa_bwd_dq_strategy.restype = i
    L.fa_get_device_status.argtypes = [vp]
    L.fa_reset_device_status.argtypes = [vp]
    L.fa_set_wait_limit.argtypes = [ctypes.c_uint32]
    L.fa_set_wait_limit.restype = None
    L.fa_debug_force_stall.argtypes = [ctypes.c_int]
    L.fa_debug_force_stall.restype = None
    L.fa_status_string.argtypes = [i]
    L.fa_status_string.restype = ctypes.c_char_p
    L.fa_debug_build.argtypes = []
    L.fa_debug_build.restype = i
    L.fa_debug_tile_rows.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), i, vp]
    L.fa_debug_tile_rows.restype = i
    L.fa_debug_reset_tile_rows.argtypes = [vp]
    L.fa_debug_reset_tile_rows.restype = i
    for name in ("fa_fwd", "fa_bwd", "fa_bwd_preprocess", "fa_bwd_dkdv", "fa_bwd_dq", "fa_bwd_grads",
                 "fa_fwd_strided", "fa_bwd_strided", "fa_fwd_bwd", "fa_get_device_status",
                 "fa_reset_device_status"):
        getattr(L, name).restype = ctypes.c_int
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


_raw_stream = None


def _stream(stream, t=None):
    """The CUDA stream handle (an int) to launch on: `stream`, else the current
    stream of t's device (through torch's raw-stream query when it has one, which
    skips building a Stream object on every call)."""
    global _raw_stream
    if stream is not None:
        return stream.cuda_stream
    torch = _torch()
    if t is not None:
        if _raw_stream is None:
            _raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", False)
        if _raw_stream:
            return _raw_stream(t.get_device())
    return torch.cuda.current_stream().cuda_stream


def _ptr(t):
    return t.data_ptr() if t is not None else None


def _check_inputs(*ts, strided=False):
    dt = ts[0].dtype
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if t.dtype != dt:
            raise ValueError("Q, K, V (and O, dO) must share a dtype")
        if not strided and not t.is_contiguous():
            raise ValueError("tensors must be contiguous (B, H, N, d) or (..., N, d)")


def _on_gpu(*ts):
    """Every tensor handed to the kernels must live in device memory."""
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")


_strides_seen = {}   # (shape, strides) -> FaStrides: the library only reads them


def _strides(t):
    """fa_strides of a (B, H, N, d) or (B, N, d) view whose last dimension is contiguous,
    or None for a contiguous tensor (the plain layout)."""
    if t.is_contiguous():
        return None
    shape, st = tuple(t.shape), t.stride()
    key = (shape, st)
    fs = _strides_seen.get(key)
    if fs is not None:
        return fs
    if len(shape) not in (3, 4) or (shape[-1] > 1 and st[-1] != 1):
        raise ValueError("a non-contiguous view must be (B, H, N, d) or (B, N, d) with the last dimension "
                         "contiguous")
    fs = FaStrides(st[0], st[0], st[1]) if len(shape) == 3 else FaStrides(st[0], st[1], st[2])
    if len(_strides_seen) < 1024:
        _strides_seen[key] = fs
    return fs


def accepts_view(t) -> bool:
    """True when the library reads this tensor in place (the rules of fa_strides in
    include/fa.h): contiguous, or a 3-/4-D view with a contiguous last dimension, a
    16-byte aligned start and positive strides that are multiples of 16 bytes."""
    if t.is_contiguous():
        return t.data_ptr() % 16 == 0
    if t.dim() not in (3, 4) or (t.shape[-1] > 1 and t.stride(-1) != 1) or t.data_ptr() % 16:
        return False
    eb = t.element_size()
    for size, stride in zip(t.shape[:-1], t.stride()[:-1]):
        if size > 1 and (stride <= 0 or (stride * eb) % 16):
            return False
    return True


def _sp(st):
    return ctypes.byref(st) if st is not None else None


def _like_rows(Q, shape):
    """An output with Q's order of heads and rows: a (B, N, H, d) buffer seen as
    (B, H, N, d) when Q's rows are outer to its heads (a transposed projection),
    else contiguous."""
    torch = _torch()
    if Q.dim() == 4 and not Q.is_contiguous() and Q.shape[1] > 1 and Q.stride(2) > Q.stride(1):
        B, H, N, d = shape
        return torch.empty((B, N, H, d), dtype=Q.dtype, device=Q.device).transpose(1, 2)
    return torch.empty(shape, dtype=Q.dtype, device=Q.device)


def set_dq_strategy(strategy: int) -> int:
    """fa_set_dq_strategy: FA_DQ_AUTO, FA_DQ_SEPARATE_PASS or FA_DQ_REDUCTION; returns the previous one."""
    prev = int(lib().fa_set_dq_strategy(int(strategy)))
    if prev < 0:
        raise ValueError(f"unknown dQ strategy {strategy}")
    return prev


def set_fp32_mode(mode: int) -> int:
    """fa_set_fp32_mode: FA_FP32_AUTO, FA_FP32_EXACT or FA_FP32_SPLIT; returns the previous one."""
    prev = int(lib().fa_set_fp32_mode(int(mode)))
    if prev < 0:
        raise ValueError(f"unknown fp32 mode {mode}")
    return prev


@contextlib.contextmanager
def fp32_mode(mode: int):
    """Within the block, fp32 inputs run in `mode` (the library's setting, restored after)."""
    prev = set_fp32_mode(mode)
    try:
        yield
    finally:
        set_fp32_mode(prev)


def dq_strategy(Q, K, is_causal=False) -> int:
    """The dQ strategy fa_bwd uses for these tensors (FA_DQ_SEPARATE_PASS or FA_DQ_REDUCTION)."""
    B, H = _bh(Q)
    return int(lib().fa_bwd_dq_strategy(B, H, Q.shape[-2], K.shape[-2], Q.shape[-1], int(is_causal),
                                        dtype_code(Q)))


def path_name(Nq, Nk, d, is_causal, dtype_c) -> str | None:
    r = lib().fa_path_name(Nq, Nk, d, int(is_causal), dtype_c)
    return r.decode() if r else None


# ------------------------------------------------------------------ entry points

def fa_fwd(Q, K, V, is_causal=False, scale=None, O=None, L=None, stream=None):
    """O (shaped like Q) and L (Q.shape[:-1], fp32) of attention; see include/fa.h.

    Contiguous inputs go to fa_fwd.  Strided (B, H, N, d) views (for example a
    (B, N, H, d) projection transposed to (B, H, N, d)) go to fa_fwd_strided and
    are read in place; O then follows Q's order of heads and rows."""
    torch = _torch()
    strided = not (Q.is_contiguous() and K.is_contiguous() and V.is_contiguous()
                   and (O is None or O.is_contiguous()))
    _check_inputs(Q, K, V, strided=strided)
    B, H = _bh(Q)
    shape = Q.shape
    Nq, d = shape[-2], shape[-1]
    Nk = K.shape[-2]
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if L is None:
        L = torch.empty(shape[:-1], dtype=torch.float32, device=Q.device)
    if not strided:
        if O is None:
            O = torch.empty_like(Q)
        check(lib().fa_fwd(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), L.data_ptr(), B, H, Nq, Nk, d,
                           sc, int(is_causal), dtype_code(Q), _stream(stream, Q)), "fa_fwd")
        return O, L
    if Q.shape[:-2] != K.shape[:-2] or K.shape[:-2] != V.shape[:-2]:
        raise ValueError("Q, K and V need the same batch and head sizes")
    if O is None:
        O = _like_rows(Q, tuple(Q.shape))
    sQ, sK, sV, sO = _strides(Q), _strides(K), _strides(V), _strides(O)
    check(lib().fa_fwd_strided(_ptr(Q), _sp(sQ), _ptr(K), _sp(sK), _ptr(V), _sp(sV), _ptr(O), _sp(sO), _ptr(L),
                               B, H, Nq, Nk, d, sc, int(is_causal), dtype_code(Q), _stream(stream, Q)),
          "fa_fwd_strided")
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
    """dQ, dK, dV of attention given the forward's O and L; see include/fa.h.

    Contiguous tensors go to fa_bwd; strided views to fa_bwd_strided, with each
    gradient laid out like its input when that input is dense (else contiguous)."""
    torch = _torch()
    _check_inputs(Q, K, V, O, dO, strided=True)
    B, H = _bh(Q)
    Nq, d = Q.shape[-2], Q.shape[-1]
    Nk = K.shape[-2]
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    ws = alloc_workspace(Q, K, is_causal) if workspace is None else workspace
    if all(t.is_contiguous() for t in (Q, K, V, O, dO, dQ, dK, dV)):
        check(lib().fa_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(L), _ptr(dQ), _ptr(dK), _ptr(dV),
                           B, H, Nq, Nk, d, sc, int(is_causal), dtype_code(Q), _ptr(ws), ws.numel(),
                           _stream(stream, Q)), "fa_bwd")
        return dQ, dK, dV
    if not (Q.shape[:-2] == K.shape[:-2] == V.shape[:-2] == O.shape[:-2] == dO.shape[:-2]):
        raise ValueError("Q, K, V, O and dO need the same batch and head sizes")
    st = [_strides(t) for t in (Q, K, V, O, dO, dQ, dK, dV)]
    check(lib().fa_bwd_strided(_ptr(Q), _sp(st[0]), _ptr(K), _sp(st[1]), _ptr(V), _sp(st[2]), _ptr(O), _sp(st[3]),
                               _ptr(dO), _sp(st[4]), _ptr(L), _ptr(dQ), _sp(st[5]), _ptr(dK), _sp(st[6]), _ptr(dV),
                               _sp(st[7]), B, H, Nq, Nk, d, sc, int(is_causal), dtype_code(Q), _ptr(ws), ws.numel(),
                               _stream(stream, Q)), "fa_bwd_strided")
    return dQ, dK, dV


def fa_fwd_bwd(Q, K, V, dO, is_causal=False, scale=None, O=None, L=None, dQ=None, dK=None, dV=None, workspace=None,
               stream=None):
    """Forward then backward in one library call (contiguous tensors): O, L, dQ,
    dK, dV with a given dO -- the leaderboard's timed unit; see include/fa.h."""
    torch = _torch()
    _check_inputs(Q, K, V, dO)
    B, H = _bh(Q)
    shape = Q.shape
    Nq, d = shape[-2], shape[-1]
    Nk = K.shape[-2]
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    O = torch.empty_like(Q) if O is None else O
    L = torch.empty(shape[:-1], dtype=torch.float32, device=Q.device) if L is None else L
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    _check_inputs(O, dQ, dK, dV)
    ws = alloc_workspace(Q, K, is_causal) if workspace is None else workspace
    check(lib().fa_fwd_bwd(Q.data_ptr(), K.data_ptr(), V.data_ptr(), dO.data_ptr(), O.data_ptr(), L.data_ptr(),
                           dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(), B, H, Nq, Nk, d, sc, int(is_causal),
                           dtype_code(Q), ws.data_ptr(), ws.numel(), _stream(stream, Q)), "fa_fwd_bwd")
    return O, L, dQ, dK, dV


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
                               _ptr(dV), B, H, Nq, Nk, d, sc, int(is_causal), dtype_code(Q), _stream(stream, Q)),
          "fa_bwd_noalloc")
    return dQ, dK, dV


def fa_bwd_preprocess(O, dO, L, Q, K, is_causal, workspace, stream=None):
    _on_gpu(O, dO, L, workspace)
    B, H = _bh(Q)
    check(lib().fa_bwd_preprocess(_ptr(O), _ptr(dO), _ptr(L), B, H, Q.shape[-2], K.shape[-2], Q.shape[-1],
                                  int(is_causal), dtype_code(Q), _ptr(workspace), workspace.numel(),
                                  _stream(stream, Q)), "fa_bwd_preprocess")


def fa_bwd_dkdv(Q, K, V, dO, L, dQ, dK, dV, is_causal, workspace, scale=None, stream=None):
    _on_gpu(Q, K, V, dO, L, dQ, dK, dV, workspace)
    B, H = _bh(Q)
    d = Q.shape[-1]
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    check(lib().fa_bwd_dkdv(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(L), _ptr(dQ), _ptr(dK), _ptr(dV), B, H,
                            Q.shape[-2], K.shape[-2], d, sc, int(is_causal), dtype_code(Q), _ptr(workspace),
                            workspace.numel(), _stream(stream, Q)), "fa_bwd_dkdv")


def fa_bwd_dq(Q, K, V, dO, L, dQ, is_causal, workspace, scale=None, stream=None):
    _on_gpu(Q, K, V, dO, L, dQ, workspace)
    B, H = _bh(Q)
    d = Q.shape[-1]
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    check(lib().fa_bwd_dq(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(L), _ptr(dQ), B, H, Q.shape[-2],
                          K.shape[-2], d, sc, int(is_causal), dtype_code(Q), _ptr(workspace), workspace.numel(),
                          _stream(stream, Q)), "fa_bwd_dq")


def fa_bwd_grads(Q, K, V, dO, L, dQ, dK, dV, is_causal, workspace, scale=None, stream=None):
    _on_gpu(Q, K, V, dO, L, dQ, dK, dV, workspace)
    B, H = _bh(Q)
    d = Q.shape[-1]
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    check(lib().fa_bwd_grads(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(L), _ptr(dQ), _ptr(dK), _ptr(dV), B, H,
                             Q.shape[-2], K.shape[-2], d, sc, int(is_causal), dtype_code(Q), _ptr(workspace),
                             workspace.numel(), _stream(stream, Q)), "fa_bwd_grads")


def fa_get_device_status(stream=None) -> int:
    return int(lib().fa_get_device_status(_stream(stream)))


def fa_reset_device_status(stream=None):
    check(lib().fa_reset_device_status(_stream(stream)), "fa_reset_device_status")


def fa_set_wait_limit(spins: int):
    lib().fa_set_wait_limit(int(spins))


def fa_debug_force_stall(on: bool):
    lib().fa_debug_force_stall(1 if on else 0)


def debug_tile_rows(stream=None):
    """fa_debug_tile_rows: [forward key rows, dK/dV-item query rows, dQ-item key rows] loaded."""
    out = (ctypes.c_ulonglong * 3)()
    check(lib().fa_debug_tile_rows(out, 3, _stream(stream)), "fa_debug_tile_rows")
    return [int(x) for x in out]


def debug_reset_tile_rows(stream=None):
    check(lib().fa_debug_reset_tile_rows(_stream(stream)), "fa_debug_reset_tile_rows")

"""Host-side checks of the C ABI: the library builds, loads, exports every
function include/fa.h declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def L():
    from tiled_attention_04_gb300 import binding, build
    build.build()
    return binding.lib()


def declared_functions():
    txt = open(HEADER).read()
    return re.findall(r"^FA_API\s+[\w\s\*]+?\b(fa_\w+)\s*\(", txt, flags=re.M)


def test_header_declares_the_binding_exports():
    from tiled_attention_04_gb300 import binding
    assert sorted(declared_functions()) == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    # and nothing internal leaks out with default visibility
    assert not hasattr(L, "simt_fwd")


def test_debug_library_exports_the_same_symbols_and_says_so(L):
    """libfa_debug.so (FA_DEBUG: in-kernel bounds checks, tile-load counters) exports
    the same functions; fa_debug_build tells the two apart."""
    from tiled_attention_04_gb300 import binding
    with binding.debug_library() as D:
        for name in declared_functions():
            assert hasattr(D, name), name
        assert not hasattr(D, "simt_fwd")
        assert D.fa_debug_build() == 1
    assert L.fa_debug_build() == 0
    assert binding.lib() is L


def test_status_strings(L):
    for s in range(12):
        assert L.fa_status_string(s)
    assert L.fa_status_string(99) == b"unknown status"


V16 = ctypes.c_void_p(16)   # a non-null, 16-byte-aligned address that is never dereferenced
VP = ctypes.c_void_p


def fwd(L, Q=V16, K=V16, V=V16, O=V16, Lse=V16, B=1, H=1, Nq=128, Nk=128, d=64, scale=0.125, causal=1, dt=1):
    return L.fa_fwd(Q, K, V, O, Lse, B, H, Nq, Nk, d, scale, causal, dt, None)


@pytest.mark.parametrize("kw,status", [
    (dict(d=48), 3), (dict(d=256), 3), (dict(d=0), 3),
    (dict(dt=2), 4), (dict(dt=-1), 4),
    (dict(B=-1), 2), (dict(Nq=-5), 2), (dict(Nk=0), 2), (dict(B=1 << 20, H=1 << 12), 2),
    (dict(Q=VP(0)), 1), (dict(Lse=VP(0)), 1),
    (dict(K=VP(24)), 5), (dict(O=VP(8)), 5),
    (dict(causal=2), 10), (dict(scale=float("inf")), 10), (dict(scale=float("nan")), 10),
])
def test_fwd_rejects_bad_arguments(L, kw, status):
    assert fwd(L, **kw) == status


def test_empty_calls_are_noops(L):
    assert fwd(L, B=0) == 0
    assert fwd(L, Nq=0, Q=VP(0), O=VP(0), Lse=VP(0)) == 0
    assert fwd(L, Nq=0, Nk=0) == 0


def test_workspace_size(L):
    n = L.fa_bwd_workspace_size(2, 3, 1000, 512, 64, 1, 1)
    assert n >= 2 * 3 * 1000 * 4 and n % 256 == 0
    assert L.fa_bwd_workspace_size(1, 1, 128, 128, 48, 0, 1) == 0
    assert L.fa_bwd_workspace_size(1, 1, 128, 128, 64, 0, 7) == 0


def bwd(L, ws=V16, ws_bytes=1 << 30, **kw):
    a = dict(B=1, H=1, Nq=128, Nk=128, d=64, scale=0.125, causal=1, dt=1)
    a.update(kw)
    return L.fa_bwd(V16, V16, V16, V16, V16, V16, V16, V16, V16, a["B"], a["H"], a["Nq"], a["Nk"], a["d"],
                    a["scale"], a["causal"], a["dt"], ws, ws_bytes, None)


def test_bwd_rejects_bad_workspace(L):
    assert bwd(L, ws=VP(0)) == 6
    assert bwd(L, ws_bytes=16) == 6
    assert bwd(L, ws=VP(40)) == 5
    assert bwd(L, d=100) == 3


def test_path_choice(L):
    from tiled_attention_04_gb300 import binding
    assert binding.path_name(128, 128, 48, 1, binding.FA_DTYPE_F32) is None
    assert binding.path_name(4096, 4096, 64, 1, binding.FA_DTYPE_BF16) == "tc"
    assert binding.path_name(4096, 4096, 16, 1, binding.FA_DTYPE_BF16) == "tc"    # padded to 64 columns
    assert binding.path_name(4096, 4096, 32, 0, binding.FA_DTYPE_BF16) == "tc"
    assert binding.path_name(100, 4096, 64, 1, binding.FA_DTYPE_BF16) == "simt"   # shorter than one tile
    # fp32 up to d = 64: split into bf16 pairs, three products per contraction
    assert binding.path_name(128, 128, 16, 1, binding.FA_DTYPE_F32) == "tc"
    assert binding.path_name(4096, 4096, 64, 1, binding.FA_DTYPE_F32) == "tc"
    assert binding.path_name(4096, 4096, 128, 1, binding.FA_DTYPE_F32) == "tc"    # 256-column split rows
    assert binding.path_name(100, 4096, 32, 1, binding.FA_DTYPE_F32) == "simt"


def test_valid_call_without_a_device_reports_no_device(L):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert fwd(L) == 9


# ------------------------------------------------------------------ strided views (fa_strides)

def _st(b, h, n):
    from tiled_attention_04_gb300 import binding
    return ctypes.byref(binding.FaStrides(b, h, n))


def fwd_strided(L, sQ=None, sK=None, sV=None, sO=None, B=2, H=4, Nq=256, Nk=256, d=64, dt=1):
    return L.fa_fwd_strided(V16, sQ, V16, sK, V16, sV, V16, sO, V16, B, H, Nq, Nk, d, 0.125, 1, dt, None)


def bwd_strided(L, s=None, B=2, H=4, Nq=256, Nk=256, d=64, dt=1):
    s = s or {}
    g = lambda k: s.get(k)   # noqa: E731
    return L.fa_bwd_strided(V16, g("Q"), V16, g("K"), V16, g("V"), V16, g("O"), V16, g("dO"), V16,
                            V16, g("dQ"), V16, g("dK"), V16, g("dV"), B, H, Nq, Nk, d, 0.125, 1, dt,
                            V16, 1 << 30, None)


# (B, H, N, d) = (2, 4, 256, 64): contiguous strides are (65536, 16384, 64); a transposed
# (B, N, H, d) buffer gives (65536, 64, 256)
@pytest.mark.parametrize("kw,status", [
    (dict(sQ=(65536, 64, 256)), None),                  # transposed projection layout: accepted
    (dict(sK=(3 * 65536, 64, 3 * 256)), None),          # one third of a fused QKV buffer
    (dict(sQ=(65536, 16384, 72)), None),                # padded rows (inputs may have gaps)
    (dict(sQ=(65536, 16384, 68)), 5),                   # row stride not a multiple of 16 bytes
    (dict(sV=(65536, 20, 256)), 5),                     # head stride not a multiple of 16 bytes
    (dict(sQ=(65536, 0, 64)), 2),                       # broadcast head: not supported
    (dict(sK=(-65536, 16384, 64)), 2),                  # negative stride
    (dict(sQ=(1 << 40, 16384, 64)), 2),                 # beyond the 2^40-byte stride limit
    (dict(sO=(65536, 64, 256)), None),                  # dense transposed output
    (dict(sO=(65536, 16384, 32)), 2),                   # output rows overlap (row stride < d)
    (dict(sO=(65536, 64, 64)), 2),                      # output heads and rows collide
    (dict(sO=(16384, 16384, 64)), 2),                   # output batches and heads collide
    (dict(sQ=(65536, 16384, 32)), None),                # overlapping input rows are fine
])
def test_fwd_strided_checks_views(L, kw, status):
    args = {k: _st(*v) for k, v in kw.items()}
    got = fwd_strided(L, **args)
    if status is None:
        # accepted: the call goes on to find no device here (or runs, where one exists)
        assert got in (0, 9)
    else:
        assert got == status


def test_strided_extent_one_dimensions_ignore_their_stride(L):
    # B = 1 and H = 1: the batch and head strides are never used, whatever they are
    got = fwd_strided(L, sQ=_st(0, -7, 64), sO=_st(3, 5, 64), B=1, H=1)
    assert got in (0, 9)


def test_fp32_strides_need_multiples_of_4_elements(L):
    assert fwd_strided(L, sQ=_st(65536, 16384, 68), dt=0) in (0, 9)
    assert fwd_strided(L, sQ=_st(65536, 16384, 66), dt=0) == 5


def test_bwd_strided_checks_every_view(L):
    assert bwd_strided(L) in (0, 9)
    assert bwd_strided(L, {"dO": _st(65536, 64, 256), "dQ": _st(65536, 64, 256)}) in (0, 9)
    assert bwd_strided(L, {"dO": _st(65536, 16384, 60)}) == 5
    assert bwd_strided(L, {"dK": _st(65536, 16384, 32)}) == 2      # overlapping gradient rows
    assert bwd_strided(L, {"O": _st(65536, 16384, 32)}) in (0, 9)  # O is read, not written
    assert bwd_strided(L, {"dV": _st(65536, 0, 64)}) == 2


def test_binding_stride_helpers():
    torch = pytest.importorskip("torch")
    from tiled_attention_04_gb300 import binding
    x = torch.empty(2, 256, 4, 64, dtype=torch.bfloat16)
    q = x.transpose(1, 2)                                   # (B, H, N, d) view of a (B, N, H, d) buffer
    s = binding._strides(q)
    assert (s.b, s.h, s.n) == (65536, 64, 256)
    assert binding._strides(q.contiguous()) is None
    assert binding.accepts_view(q) == (q.data_ptr() % 16 == 0)
    qkv = torch.empty(2, 256, 3, 4, 64, dtype=torch.bfloat16)
    k = qkv.unbind(2)[1].transpose(1, 2)
    s = binding._strides(k)
    assert (s.b, s.h, s.n) == (3 * 65536, 64, 3 * 256)
    assert not binding.accepts_view(q[..., ::2])              # last dimension not contiguous
    assert not binding.accepts_view(q.expand(2, 4, 256, 64).as_strided((2, 4, 256, 64), (0, 64, 256, 1)))
    o = binding._like_rows(q, (2, 4, 256, 64))
    assert o.shape == (2, 4, 256, 64) and o.stride() == (65536, 64, 256, 1)
    assert binding._like_rows(q.contiguous(), (2, 4, 256, 64)).is_contiguous()


def fwd_bwd(L, O=V16, ws=V16, ws_bytes=1 << 30, **kw):
    a = dict(B=1, H=1, Nq=128, Nk=128, d=64, scale=0.125, causal=1, dt=1)
    a.update(kw)
    return L.fa_fwd_bwd(V16, V16, V16, V16, O, V16, V16, V16, V16, a["B"], a["H"], a["Nq"], a["Nk"], a["d"],
                        a["scale"], a["causal"], a["dt"], ws, ws_bytes, None)


def test_fwd_bwd_checks_both_passes_before_launching(L):
    assert fwd_bwd(L, ws=VP(0)) == 6           # the backward's workspace, checked before the forward runs
    assert fwd_bwd(L, ws_bytes=16) == 6
    assert fwd_bwd(L, O=VP(0)) == 1
    assert fwd_bwd(L, O=VP(24)) == 5
    assert fwd_bwd(L, d=100) == 3
    assert fwd_bwd(L, causal=3) == 10
    assert fwd_bwd(L, B=0) == 0                # empty
    assert fwd_bwd(L) in (0, 9)


def test_autograd_copies_views_the_kernels_cannot_read():
    torch = pytest.importorskip("torch")
    from tiled_attention_04_gb300 import binding
    from tiled_attention_04_gb300.autograd import _in_place
    base = torch.zeros(2 * 256 * 64 + 1, dtype=torch.bfloat16)
    odd = base[1:].view(2, 1, 256, 64)                 # contiguous, but 2 bytes off a 16-byte boundary
    assert odd.is_contiguous() and not binding.accepts_view(odd)
    fixed = _in_place(odd)
    assert fixed.data_ptr() % 16 == 0 and torch.equal(fixed, odd)
    x = torch.zeros(2, 4, 256, 64, dtype=torch.bfloat16)
    assert _in_place(x) is x                            # contiguous and aligned: used in place
    t = x.transpose(1, 2).contiguous().transpose(1, 2)  # (B, N, H, d) buffer seen as (B, H, N, d)
    assert _in_place(t) is t
    bcast = torch.zeros(1, 1, 256, 64, dtype=torch.bfloat16).expand(2, 4, 256, 64)
    c = _in_place(bcast)                                # stride-0 heads: copied
    assert c is not bcast and c.is_contiguous()

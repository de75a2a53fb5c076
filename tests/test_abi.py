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


def test_status_strings(L):
    for s in range(11):
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
    assert binding.path_name(128, 128, 16, 1, binding.FA_DTYPE_F32) == "simt"
    assert binding.path_name(128, 128, 48, 1, binding.FA_DTYPE_F32) is None
    assert binding.path_name(4096, 4096, 64, 1, binding.FA_DTYPE_BF16) in ("tc", "simt")


def test_valid_call_without_a_device_reports_no_device(L):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert fwd(L) == 9

"""Host-side tests of the C ABI: the library builds and loads without a GPU,
exports every symbol include/fa.h declares, and rejects bad arguments with a
status code before touching the device (no call here reaches CUDA)."""
import ctypes
import os
import re
import subprocess

import pytest

import attention_fa_fwd_03_gb300 as fa
from attention_fa_fwd_03_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return fa.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_status_string",
              "fa_device_status", "fa_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build_lib.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert getattr(lib, n) is not None


def test_status_strings_and_version(lib):
    assert fa.fa_abi_version() == 101
    for code in range(7):
        s = fa.fa_status_string(code)
        assert isinstance(s, str) and s
    assert fa.fa_status_string(99) == "unknown status"


def test_workspace_size(lib):
    assert fa.fa_bwd_workspace_size(4, 32, 4096) == 4 * 32 * 4096 * 4
    assert fa.fa_bwd_workspace_size(1, 1, 1) == 256
    assert fa.fa_bwd_workspace_size(0, 8, 8) == 0
    assert fa.fa_bwd_workspace_size(2, -1, 8) == 0


# Fake, well-separated, 16-byte aligned "device" addresses: validation rejects
# every call below before any CUDA API is reached.
BASE = 1 << 40
GAP = 1 << 34


def ptrs(n):
    return [BASE + i * GAP for i in range(n)]


GOOD = dict(B=2, Hq=8, Hkv=2, Tq=100, Tkv=100, D=128, scale=0.125, causal=1, window=0, dt=1)


def call_fwd(lib, p=None, **kw):
    a = dict(GOOD, **kw)
    p = p or ptrs(5)
    return lib.fa_fwd(*p, a["B"], a["Hq"], a["Hkv"], a["Tq"], a["Tkv"], a["D"], a["scale"],
                      a["causal"], a["window"], a["dt"], None)


def call_bwd(lib, p=None, ws_bytes=None, **kw):
    a = dict(GOOD, **kw)
    p = p or ptrs(10)
    if ws_bytes is None:
        ws_bytes = max(fa.fa_bwd_workspace_size(a["B"], a["Hq"], a["Tq"]), 256)
    return lib.fa_bwd(*p[:9], a["B"], a["Hq"], a["Hkv"], a["Tq"], a["Tkv"], a["D"], a["scale"],
                      a["causal"], a["window"], a["dt"], p[9], ws_bytes, None)


INVALID, HEAD_DIM, DTYPE, MISALIGNED = 1, 2, 3, 4

BAD_ARGS = [
    (dict(B=0), INVALID), (dict(Hq=0), INVALID), (dict(Tq=0), INVALID), (dict(Tkv=-3), INVALID),
    (dict(Hq=6, Hkv=4), INVALID),                        # Hq not a multiple of Hkv
    (dict(D=80), HEAD_DIM), (dict(D=512), HEAD_DIM), (dict(D=32), HEAD_DIM),
    (dict(dt=2), DTYPE), (dict(dt=-1), DTYPE),
    (dict(scale=0.0), INVALID), (dict(scale=-0.1), INVALID), (dict(scale=float("nan")), INVALID),
    (dict(scale=float("inf")), INVALID),
    (dict(causal=2), INVALID), (dict(window=-1), INVALID),
    (dict(Tq=(1 << 22) + 1), INVALID),                   # beyond the supported length
]


@pytest.mark.parametrize("kw,code", BAD_ARGS)
def test_fwd_rejects_bad_arguments(lib, kw, code):
    assert call_fwd(lib, **kw) == code


@pytest.mark.parametrize("kw,code", BAD_ARGS)
def test_bwd_rejects_bad_arguments(lib, kw, code):
    assert call_bwd(lib, **kw) == code


@pytest.mark.parametrize("i", range(5))
def test_fwd_null_and_misaligned_pointers(lib, i):
    p = ptrs(5)
    p[i] = None
    assert call_fwd(lib, p=p) == INVALID
    p = ptrs(5)
    p[i] += 8
    assert call_fwd(lib, p=p) == MISALIGNED


@pytest.mark.parametrize("i", range(10))
def test_bwd_null_and_misaligned_pointers(lib, i):
    p = ptrs(10)
    p[i] = None
    assert call_bwd(lib, p=p) == INVALID
    p = ptrs(10)
    p[i] += 4
    assert call_bwd(lib, p=p) == MISALIGNED


def test_overlapping_outputs_are_rejected(lib):
    p = ptrs(5)
    p[3] = p[0] + 4096          # O inside Q
    assert call_fwd(lib, p=p) == INVALID
    p = ptrs(5)
    p[4] = p[3] + 1024          # LSE inside O
    assert call_fwd(lib, p=p) == INVALID
    p = ptrs(10)
    p[7] = p[6] + 16            # dK inside dQ
    assert call_bwd(lib, p=p) == INVALID
    p = ptrs(10)
    p[9] = p[4]                 # workspace aliases dO
    assert call_bwd(lib, p=p) == INVALID


def test_small_workspace_is_rejected(lib):
    need = fa.fa_bwd_workspace_size(GOOD["B"], GOOD["Hq"], GOOD["Tq"])
    assert call_bwd(lib, ws_bytes=need - 1) == INVALID


def test_binding_refuses_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 1, 8, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q, q, q.clone(), torch.zeros(1, 1, 8), 0.125)


def test_binding_without_library_fails_loudly(tmp_path, monkeypatch):
    """No silent fallback: a missing library is an error at the first call."""
    monkeypatch.setattr(fa, "_lib", None)
    monkeypatch.setattr(fa, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        fa.library()


def call_dkv(lib, p=None, **kw):
    a = dict(GOOD, **kw)
    p = p or ptrs(8)
    return lib.fa_bwd_dkv(*p, a["B"], a["Hq"], a["Hkv"], a["Tq"], a["Tkv"], a["D"], a["scale"],
                          a["causal"], a["window"], a["dt"], None)


def call_dq(lib, p=None, **kw):
    a = dict(GOOD, **kw)
    p = p or ptrs(7)
    return lib.fa_bwd_dq(*p, a["B"], a["Hq"], a["Hkv"], a["Tq"], a["Tkv"], a["D"], a["scale"],
                         a["causal"], a["window"], a["dt"], None)


@pytest.mark.parametrize("kw,code", BAD_ARGS)
def test_backward_phases_reject_bad_arguments(lib, kw, code):
    """The phase entry points validate like fa_bwd, before any launch."""
    assert call_dkv(lib, **kw) == code
    assert call_dq(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [(dict(B=0), INVALID), (dict(Tq=0), INVALID),
                                     (dict(D=80), HEAD_DIM), (dict(dt=5), DTYPE)])
def test_preprocess_rejects_bad_arguments(lib, kw, code):
    a = dict(GOOD, **kw)
    p = ptrs(3)
    assert lib.fa_bwd_preprocess(*p, a["B"], a["Hq"], a["Tq"], a["D"], a["dt"], None) == code


def test_noalloc_rejects_too_many_rows(lib):
    """fa_bwd_noalloc keeps the D-vector in a fixed array: more rows than it
    holds is an argument error, reported before anything is launched."""
    f = lib.fa_bwd_noalloc
    vp, i, fl = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [vp] * 9 + [i] * 6 + [fl, i, i, i, vp]
    f.restype = i
    lib.fa_bwd_noalloc_max_rows.restype = ctypes.c_size_t
    rows = int(lib.fa_bwd_noalloc_max_rows())
    a = dict(GOOD, B=1, Hq=2, Hkv=1, Tq=rows // 2 + 1)
    assert f(*ptrs(9), a["B"], a["Hq"], a["Hkv"], a["Tq"], a["Tkv"], a["D"], a["scale"],
             a["causal"], a["window"], a["dt"], None) == INVALID
    for kw, code in BAD_ARGS[:10]:
        a = dict(GOOD, **kw)
        assert f(*ptrs(9), a["B"], a["Hq"], a["Hkv"], a["Tq"], a["Tkv"], a["D"], a["scale"],
                 a["causal"], a["window"], a["dt"], None) == code, kw

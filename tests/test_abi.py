"""The C ABI boundary on the CPU: the library builds, loads and exports every
function include/*.h declares; host-side argument checks return their
status codes before any CUDA call; workspace sizing is a pure host function.
No kernel is launched here."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_212_gb300 import build as B
    try:
        B.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    B.build()
    import paged_kv_cache_212_gb300 as P
    return P.load_library()


def declared_functions():
    names = []
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_the_five_calls_and_helpers():
    names = declared_functions()
    for n in ("paged_kv_write", "paged_kv_write_int8", "paged_kv_gather", "paged_decode_attention",
              "paged_prefill_attention", "pkv_decode_workspace_bytes", "pkv_status_string",
              "pkv_last_cuda_error"):
        assert n in names, n


def test_header_is_plain_c():
    assert len(HEADERS) >= 2
    for h in HEADERS:
        r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-x", "c", h],
                           capture_output=True, text=True)
        assert r.returncode == 0, (h, r.stderr)


def test_library_exports_every_declared_symbol(lib):
    from paged_kv_cache_212_gb300 import EXPORTS
    names = declared_functions()
    assert set(EXPORTS) == set(names)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if " T " in line)
    assert set(names) <= exported


def test_status_strings(lib):
    assert lib.pkv_status_string(0) == b"PKV_OK"
    assert lib.pkv_status_string(4) == b"PKV_ERR_WORKSPACE"
    assert lib.pkv_status_string(99) == b"PKV_ERR_UNKNOWN"


def _dims(P, nb=8, bs=16, hkv=2, d=64):
    return P.Dims(nb, bs, hkv, d)


FAKE = ctypes.c_void_p(0x1000)      # 16-byte aligned, never dereferenced
MISALIGNED = ctypes.c_void_p(0x1008)


def test_write_argument_checks(lib):
    import paged_kv_cache_212_gb300 as P
    d = _dims(P)
    w = lib.paged_kv_write
    # no-op sizes return OK without touching anything
    assert w(None, None, None, None, d, None, 4, None, 0, 1, None, None) == 0
    assert w(None, None, None, None, d, None, 4, None, 3, 0, None, None) == 0
    # null pointers / bad sizes
    assert w(None, FAKE, FAKE, FAKE, d, FAKE, 4, FAKE, 1, 1, None, None) == 1
    assert w(FAKE, FAKE, FAKE, FAKE, d, FAKE, 0, FAKE, 1, 1, None, None) == 1
    assert w(FAKE, FAKE, FAKE, FAKE, d, FAKE, 4, FAKE, -1, 1, None, None) == 1
    assert w(MISALIGNED, FAKE, FAKE, FAKE, d, FAKE, 4, FAKE, 1, 1, None, None) == 1
    # unsupported geometry
    assert w(FAKE, FAKE, FAKE, FAKE, _dims(P, d=96), FAKE, 4, FAKE, 1, 1, None, None) == 2
    assert w(FAKE, FAKE, FAKE, FAKE, _dims(P, bs=8), FAKE, 4, FAKE, 1, 1, None, None) == 2
    assert w(FAKE, FAKE, FAKE, FAKE, _dims(P, nb=-1), FAKE, 4, FAKE, 1, 1, None, None) == 1
    # more new tokens than a table row can hold
    assert w(FAKE, FAKE, FAKE, FAKE, d, FAKE, 2, FAKE, 1, 33, None, None) == 3
    wi = lib.paged_kv_write_int8
    assert wi(FAKE, FAKE, FAKE, FAKE, None, FAKE, d, FAKE, 4, FAKE, 1, 1, None, None) == 1


def test_decode_argument_checks(lib):
    import paged_kv_cache_212_gb300 as P
    d = _dims(P, hkv=2)
    f = lib.paged_decode_attention
    args = lambda **kw: [kw.get("q", FAKE), kw.get("hq", 8), FAKE, FAKE, kw.get("ks", None), kw.get("vs", None),
                         kw.get("dt", 0), kw.get("dims", d), FAKE, 4, FAKE, kw.get("n", 2), kw.get("sc", 0.125),
                         kw.get("split", 0), FAKE, None, kw.get("ws", FAKE), kw.get("wsb", 1 << 20), None,
                         None]
    assert f(*args(n=0)) == 0
    assert f(*args(hq=7)) == 1                      # Hq % Hkv != 0
    assert f(*args(hq=18 * 2)) == 2                 # G = 18 > 8
    assert f(*args(dt=3)) == 2
    assert f(*args(split=24)) == 2                  # not a multiple of 16
    assert f(*args(q=None)) == 1
    assert f(*args(q=MISALIGNED)) == 1
    assert f(*args(dt=1, dims=_dims(P, hkv=4))) == 1  # int8 without scales
    assert f(*args(dt=1, ks=FAKE, vs=FAKE)) == 2   # int8 needs Hkv % 4 == 0
    assert f(*args(ws=None)) == 4
    assert f(*args(wsb=64)) == 4
    assert f(*args(ws=ctypes.c_void_p(0x1010))) == 4  # not 256-byte aligned
    for sc in (0.0, -0.125, float("nan"), float("inf")):  # the scale must be finite and positive
        assert f(*args(sc=sc)) == 1, sc


def test_prefill_and_gather_argument_checks(lib):
    import paged_kv_cache_212_gb300 as P
    d = _dims(P, hkv=2)
    f = lib.paged_prefill_attention
    assert f(FAKE, 8, FAKE, FAKE, d, FAKE, 4, FAKE, 0, 16, 0.1, FAKE, None, None, None) == 0
    assert f(FAKE, 8, FAKE, FAKE, d, FAKE, 4, FAKE, 1, 0, 0.1, FAKE, None, None, None) == 0
    assert f(FAKE, 6, FAKE, FAKE, d, FAKE, 4, FAKE, 1, 16, 0.1, FAKE, None, None, None) == 2  # G = 3
    assert f(FAKE, 8, FAKE, FAKE, d, FAKE, 4, FAKE, 1, 65, 0.1, FAKE, None, None, None) == 3
    assert f(None, 8, FAKE, FAKE, d, FAKE, 4, FAKE, 1, 16, 0.1, FAKE, None, None, None) == 1
    for sc in (0.0, -0.1, float("nan")):
        assert f(FAKE, 8, FAKE, FAKE, d, FAKE, 4, FAKE, 1, 16, sc, FAKE, None, None, None) == 1, sc
    g = lib.paged_kv_gather
    assert g(FAKE, FAKE, d, FAKE, 4, FAKE, 0, 16, FAKE, FAKE, None, None) == 0
    assert g(FAKE, FAKE, d, FAKE, 4, FAKE, 2, 16, None, FAKE, None, None) == 1
    assert g(FAKE, FAKE, d, FAKE, 4, FAKE, 2, -1, FAKE, FAKE, None, None) == 1


def test_decode_workspace_sizing(lib):
    f = lib.pkv_decode_workspace_bytes
    assert f(4, 8, 64, 1000, 24) == 0             # split not a multiple of 16
    assert f(-1, 8, 64, 1000, 0) == 0
    small = f(64, 32, 128, 150_000, 512)
    auto = f(64, 32, 128, 150_000, 0)
    assert 0 < small < auto                       # auto covers the smallest automatic split
    # capacity grows with the number of splits: ceil(total / split) + n_seqs partial rows
    per_split = 8 + 32 * 8 + 32 * 128 * 4
    assert f(64, 32, 128, 150_000 + 512 * 100, 512) - small >= 100 * per_split - 4 * 256


def test_binding_declares_every_signature(lib):
    """Each exported call has argtypes and an int status return in the binding."""
    from paged_kv_cache_212_gb300 import EXPORTS
    for n in EXPORTS:
        fn = getattr(lib, n)
        assert fn.argtypes is not None, n
    for n in ("paged_kv_write", "paged_kv_write_int8", "paged_kv_gather", "paged_decode_attention",
              "paged_prefill_attention", "paged_decode_attention_noalloc", "paged_decode_step"):
        assert getattr(lib, n).restype is ctypes.c_int, n


def test_decode_step_argument_checks(lib):
    import paged_kv_cache_212_gb300 as P
    d = _dims(P, hkv=2)
    f = lib.paged_decode_step
    base = [FAKE, FAKE, FAKE, 1, FAKE, 8, FAKE, FAKE, None, None, 0, d, FAKE, 4, FAKE, 2, 0.125, 0, FAKE, None,
            FAKE, 1 << 20, None, None]
    args = list(base); args[15] = 0
    assert f(*args) == 0                           # no sequences: nothing to do
    args = list(base); args[0] = None
    assert f(*args) == 1                           # the write's checks apply
    args = list(base); args[3] = 65
    assert f(*args) == 3                           # more new rows than a table row holds
    args = list(base); args[5] = 7
    assert f(*args) == 1                           # the decode's checks apply
    args = list(base); args[20] = None
    assert f(*args) == 4


def test_pipeline_wait_limit_setter(lib):
    """pkv_set_pipeline_wait_ns (host state only): returns the previous limit;
    0 restores the 4 s default."""
    assert lib.pkv_set_pipeline_wait_ns(123) == 4_000_000_000
    assert lib.pkv_set_pipeline_wait_ns(0) == 123
    assert lib.pkv_set_pipeline_wait_ns(0) == 4_000_000_000

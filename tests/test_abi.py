"""The C-ABI library on a CPU-only machine: it loads, it exports every symbol the
public header declares, and argument errors come back as PA_ERR_* codes from
the host-side checks, before any CUDA call (so no GPU is needed)."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def lib(pa_lib_path):
    return ctypes.CDLL(str(pa_lib_path))


def _declared_functions():
    names = set()
    for h in sorted((ROOT / "include").glob("*.h")):
        text = re.sub(r"/\*.*?\*/", "", h.read_text(), flags=re.S)
        names |= set(re.findall(r"\b(pa_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_four_operations():
    names = _declared_functions()
    for op in ("pa_reshape_and_cache", "pa_decode", "pa_prefill_chunk", "pa_copy_blocks"):
        assert op in names


def test_headers_declare_the_kv_manager():
    names = _declared_functions()
    for op in ("pa_kvm_create", "pa_kvm_get_computed_blocks", "pa_kvm_allocate_slots",
               "pa_kvm_cache_blocks", "pa_kvm_free"):
        assert op in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, f"libpa.so lacks {missing}"


def test_status_strings_and_version(lib):
    lib.pa_status_string.restype = ctypes.c_char_p
    for code in (0, -1, -2, -3, -4, -5):
        assert lib.pa_status_string(code).startswith(b"PA_")
    assert lib.pa_status_string(12345) == b"unknown pa status code"
    assert lib.pa_version() >= 100


def test_workspace_size_is_host_arithmetic(lib):
    lib.pa_decode_workspace_size.restype = ctypes.c_size_t
    lib.pa_decode_workspace_size.argtypes = [ctypes.c_int] * 5
    assert lib.pa_decode_workspace_size(0, 32, 8, 128, 4096) == 0
    assert lib.pa_decode_workspace_size(8, 32, 8, 96, 4096) == 0      # unsupported head dim
    assert lib.pa_decode_workspace_size(8, 24, 8, 128, 4096) == 0     # G = 3
    small = lib.pa_decode_workspace_size(8, 32, 8, 128, 100)
    big = lib.pa_decode_workspace_size(256, 32, 8, 128, 32768)
    assert 0 < small < big
    assert big % 16 == 0


# Host-side validation: each call below must be rejected before anything runs.
FAKE = 1 << 20  # a 16-byte aligned, never-dereferenced address


def _decode(lib, **over):
    args = dict(out=FAKE, out_dtype=0, query=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, mbps=4, cl=FAKE,
                maxctx=100, S=2, Hq=32, Hkv=8, D=128, bs=32, NB=16, scale=0.088, kvdt=2,
                ws=FAKE, wsb=1 << 30, status=None, stream=None)
    args.update(over)
    f = lib.pa_decode
    vp, i, fl, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    f.argtypes = [vp, i, vp, vp, vp, vp, i, vp, i, i, i, i, i, i, i, fl, i, vp, sz, vp, vp]
    return f(*args.values())


@pytest.mark.parametrize("over,code", [
    (dict(D=96), -2), (dict(bs=64), -2), (dict(Hq=24), -2), (dict(Hq=30), -1),
    (dict(kvdt=7), -1), (dict(out_dtype=9), -1), (dict(S=-1), -1), (dict(query=None), -1),
    (dict(kc=FAKE + 4), -1), (dict(out=FAKE + 2), -1), (dict(cl=FAKE + 1), -1),
    (dict(scale=float("nan")), -1), (dict(maxctx=-5), -1),
    (dict(ws=None), -3), (dict(ws=FAKE + 8), -3), (dict(Hkv=6, Hq=12), -2),
])
def test_decode_rejects_bad_arguments(lib, over, code):
    assert _decode(lib, **over) == code


def test_decode_zero_sequences_is_a_noop(lib):
    assert _decode(lib, S=0, query=None, out=None) == 0


def test_reshape_copy_prefill_reject_bad_arguments(lib):
    vp, i, fl = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f = lib.pa_reshape_and_cache
    f.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, vp]
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8, 128, 12, 10, 2, None, None) == -2  # block size
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE + 4, 4, 8, 128, 16, 10, 2, None, None) == -1  # slots
    assert f(None, FAKE, FAKE, FAKE, FAKE, 4, 8, 128, 16, 10, 2, None, None) == -1
    assert f(None, None, None, None, None, 0, 8, 128, 16, 10, 2, None, None) == 0  # no tokens
    g = lib.pa_copy_blocks
    g.argtypes = [vp, vp, vp, i, i, i, i, i, i, vp, vp]
    assert g(FAKE, FAKE, None, 3, 8, 128, 16, 10, 2, None, None) == -1
    assert g(FAKE, FAKE, FAKE, -1, 8, 128, 16, 10, 2, None, None) == -1
    assert g(None, None, None, 0, 8, 128, 16, 10, 2, None, None) == 0
    h = lib.pa_prefill_chunk
    h.argtypes = [vp, i, vp, vp, i, i, vp, vp, vp, i, vp, i, i, i, i, i, i, i, fl, i, vp, vp]
    base = [FAKE, 0, FAKE, FAKE, 64, 64, FAKE, FAKE, FAKE, 8, FAKE, 256, 1, 32, 8, 128, 32, 16,
            0.088, 2, None, None]
    bad_dtype = list(base)
    bad_dtype[19] = 0  # fp32 prefill is not built
    assert h(*bad_dtype) == -2
    no_qsl = list(base)
    no_qsl[3] = None
    assert h(*no_qsl) == -1


def _decode_write(lib, **over):
    args = dict(out=FAKE, out_dtype=0, query=FAKE, key=FAKE, value=FAKE, slots=FAKE, kc=FAKE, vc=FAKE, bt=FAKE,
                mbps=4, cl=FAKE, maxctx=100, S=2, Hq=32, Hkv=8, D=128, bs=32, NB=16, scale=0.088, kvdt=2,
                ws=FAKE, wsb=1 << 30, status=None, stream=None)
    args.update(over)
    f = lib.pa_decode_write
    vp, i, fl, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    f.argtypes = [vp, i, vp, vp, vp, vp, vp, vp, vp, i, vp, i, i, i, i, i, i, i, fl, i, vp, sz, vp, vp]
    return f(*args.values())


@pytest.mark.parametrize("over,code", [
    (dict(key=None), -1), (dict(value=None), -1), (dict(slots=None), -1), (dict(key=FAKE + 8), -1),
    (dict(slots=FAKE + 4), -1), (dict(D=96), -2), (dict(ws=None), -3), (dict(query=None), -1),
])
def test_decode_write_rejects_bad_arguments(lib, over, code):
    assert _decode_write(lib, **over) == code


def test_decode_write_and_prefill_with_nothing_to_do_are_noops(lib):
    assert _decode_write(lib, S=0, query=None, out=None, key=None, value=None, slots=None) == 0
    vp, i, fl = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    h = lib.pa_prefill_chunk
    h.argtypes = [vp, i, vp, vp, i, i, vp, vp, vp, i, vp, i, i, i, i, i, i, i, fl, i, vp, vp]
    # no sequences, and no query tokens: nothing is read or launched
    assert h(None, 0, None, None, 0, 0, FAKE, FAKE, FAKE, 8, FAKE, 256, 0, 32, 8, 128, 32, 16, 0.088, 2,
             None, None) == 0

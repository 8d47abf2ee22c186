"""The C-ABI library builds, loads without a GPU, exports every entry point
include/pa.h declares, and rejects bad arguments on the host before touching
CUDA (no compute calls here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_193_gb300 import build, _lib
    build.build()
    return _lib.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(pa_[a-z0-9_]+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_entry_points():
    names = declared_functions()
    for want in ("pa_slot_mapping", "pa_cache_append", "pa_decode", "pa_decode_partitions",
                 "pa_decode_reduce", "pa_decode_workspace_size", "pa_decode_max_partitions",
                 "pa_device_errors", "pa_status_string", "pa_last_error"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    from paged_kv_cache_193_gb300 import _lib
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"{name} has no ctypes signature in the binding"


def test_status_strings(lib):
    for st in range(5):
        assert lib.pa_status_string(st)
    assert lib.pa_status_string(99) == b"unknown status"


def test_workspace_formula(lib):
    # P = ceil(MB * B / PS); bytes = S * Hq * P * (D + 2) * 4
    assert lib.pa_decode_max_partitions(2048, 16, 512) == 64
    assert lib.pa_decode_max_partitions(8193, 16, 512) == 257
    assert lib.pa_decode_max_partitions(128, 16, 0) == 1
    assert lib.pa_decode_workspace_size(64, 64, 128, 2048, 16, 512) == 64 * 64 * 64 * 130 * 4
    assert lib.pa_decode_workspace_size(4, 8, 64, 16, 16, 0) == 0


FAKE = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: calls fail validation first


def _decode(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, mb=16, cl=FAKE, S=4, Hq=8, Hkv=2, D=64, NB=64, B=16,
             dt=0, kvs=1.0, sm=0.125, ps=0, ws=None, wsb=0, out=FAKE)
    a.update(kw)
    return lib.pa_decode(a["q"], a["k"], a["v"], a["bt"], a["mb"], a["cl"], a["S"], a["Hq"],
                         a["Hkv"], a["D"], a["NB"], a["B"], a["dt"], a["kvs"], a["sm"], a["ps"],
                         a["ws"], a["wsb"], a["out"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), 1),
    (dict(q=ctypes.c_void_p((1 << 20) + 4)), 1),
    (dict(Hkv=3), 1),
    (dict(Hq=64, Hkv=2), 2),
    (dict(D=96), 2),
    (dict(B=8), 2),
    (dict(dt=7), 2),
    (dict(ps=24), 2),
    (dict(ps=32), 3),
    (dict(ps=32, ws=FAKE, wsb=100), 3),
    (dict(dt=1, kvs=0.0), 1),
    (dict(sm=float("inf")), 1),
    (dict(NB=-1), 1),
    (dict(S=70000), 2),
    (dict(NB=1 << 27), 2),
])
def test_decode_rejects_on_host(lib, kw, status):
    assert _decode(lib, **kw) == status
    assert lib.pa_last_error()


def test_empty_batch_is_a_no_op(lib):
    assert _decode(lib, S=0, q=None, out=None) == 0


def test_append_rejects_on_host(lib):
    assert lib.pa_cache_append(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 64, 2, 96, 16, 0, 1.0, None) == 2
    assert lib.pa_cache_append(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 64, 2, 64, 16, 1, -1.0, None) == 1
    assert lib.pa_cache_append(None, FAKE, FAKE, 4, FAKE, FAKE, 64, 2, 64, 16, 0, 1.0, None) == 1
    assert lib.pa_cache_append(FAKE, FAKE, FAKE, 0, FAKE, FAKE, 64, 2, 64, 16, 0, 1.0, None) == 0


def test_reduce_and_slots_reject_on_host(lib):
    assert lib.pa_decode_reduce(FAKE, 10, FAKE, 4, 8, 64, 16, 16, 32, FAKE, None) == 3
    assert lib.pa_decode_reduce(FAKE, 1 << 30, FAKE, 4, 8, 96, 16, 16, 32, FAKE, None) == 2
    assert lib.pa_decode_reduce(FAKE, 1 << 30, FAKE, 4, 8, 64, 16, 16, 0, FAKE, None) == 1
    assert lib.pa_slot_mapping(None, 16, FAKE, 4, 16, FAKE, None) == 1
    assert lib.pa_slot_mapping(FAKE, 16, FAKE, 0, 16, FAKE, None) == 0


def test_binding_fails_loudly_without_library(tmp_path):
    from paged_kv_cache_193_gb300 import _lib
    with pytest.raises(ImportError):
        _lib.load(str(tmp_path / "missing.so"))

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


def _prefill(lib, fn="pa_prefill", **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, mb=16, cl=FAKE, qs=FAKE, S=4, T=64, mq=32, Hq=8, Hkv=2,
             D=128, NB=64, B=16, dt=0, kvs=1.0, sm=0.088, out=FAKE)
    a.update(kw)
    return getattr(lib, fn)(a["q"], a["k"], a["v"], a["bt"], a["mb"], a["cl"], a["qs"], a["S"], a["T"],
                            a["mq"], a["Hq"], a["Hkv"], a["D"], a["NB"], a["B"], a["dt"], a["kvs"],
                            a["sm"], a["out"], None)


@pytest.mark.parametrize("fn", ["pa_prefill", "pa_prefill_mma"])
@pytest.mark.parametrize("kw,status", [
    (dict(Hkv=3), 1),                               # query heads not a multiple of KV heads
    (dict(Hq=6, Hkv=2), 2),                         # group of 3
    (dict(Hq=64, Hkv=2), 2),                        # group of 32
    (dict(D=96), 2),
    (dict(B=8), 2),
    (dict(dt=7), 1),                                # no such cache type
    (dict(dt=1, D=64), 2),                          # E4M3 caches: head_dim 128 only
    (dict(NB=0), 1),
    (dict(T=-1), 1),
    (dict(S=70000), 2),
    (dict(NB=1 << 27), 2),                          # pool rows past 2^31
    (dict(sm=float("nan")), 1),
    (dict(sm=0.0), 2),                              # the prefill kernels need a positive scale
    (dict(sm=-0.088), 2),
    (dict(q=None), 1),
    (dict(out=ctypes.c_void_p((1 << 20) + 8)), 1),  # not 16-byte aligned
])
def test_prefill_rejects_on_host(lib, fn, kw, status):
    assert _prefill(lib, fn, **kw) == status
    assert lib.pa_last_error()


@pytest.mark.parametrize("kw,tc_status,mma_status", [
    (dict(dt=1, kvs=0.0), 1, 2),                    # E4M3 needs a positive, finite scale ...
    (dict(dt=1, kvs=float("inf")), 1, 2),
    (dict(dt=1, kvs=-1.0), 1, 2),                   # ... and the warp-level MMA kernel reads bf16 only
])
def test_prefill_e4m3_checks_on_host(lib, kw, tc_status, mma_status):
    assert _prefill(lib, "pa_prefill", **kw) == tc_status
    assert _prefill(lib, "pa_prefill_mma", **kw) == mma_status


@pytest.mark.parametrize("kw", [dict(T=0), dict(S=0), dict(mq=0)])
def test_empty_prefill_is_a_no_op(lib, kw):
    assert _prefill(lib, q=None, out=None, **kw) == 0


def test_chunk_slots_reject_on_host(lib):
    assert lib.pa_chunk_slot_mapping(FAKE, 0, FAKE, FAKE, 4, 16, FAKE, None) == 1
    assert lib.pa_chunk_slot_mapping(FAKE, 16, FAKE, FAKE, 4, 0, FAKE, None) == 1
    assert lib.pa_chunk_slot_mapping(FAKE, 16, FAKE, FAKE, -1, 16, FAKE, None) == 1
    assert lib.pa_chunk_slot_mapping(None, 16, FAKE, FAKE, 4, 16, FAKE, None) == 1
    assert lib.pa_chunk_slot_mapping(FAKE, 16, FAKE, FAKE, 0, 16, FAKE, None) == 0


def _step(lib, **kw):
    a = dict(q=FAKE, kn=FAKE, vn=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, mb=16, cl=FAKE, S=4, Hq=8, Hkv=2,
             D=64, NB=64, B=16, dt=0, kvs=1.0, sm=0.125, ps=0, ws=None, wsb=0, slots=None, out=FAKE)
    a.update(kw)
    return lib.pa_decode_step(a["q"], a["kn"], a["vn"], a["kc"], a["vc"], a["bt"], a["mb"], a["cl"],
                              a["S"], a["Hq"], a["Hkv"], a["D"], a["NB"], a["B"], a["dt"], a["kvs"],
                              a["sm"], a["ps"], a["ws"], a["wsb"], a["slots"], a["out"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(kn=None), 1),
    (dict(vn=ctypes.c_void_p((1 << 20) + 4)), 1),
    (dict(out=None), 1),
    (dict(ps=32), 3),                               # split without a workspace
    (dict(D=96), 2),
    (dict(dt=1, kvs=-1.0), 1),
])
def test_step_rejects_on_host(lib, kw, status):
    assert _step(lib, **kw) == status
    assert lib.pa_last_error()


def test_empty_step_is_a_no_op(lib):
    assert _step(lib, S=0, q=None, kn=None, vn=None, out=None) == 0


def _step_scaled(lib, fn, qsc=None, **kw):
    a = dict(q=FAKE, kn=FAKE, vn=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, mb=16, cl=FAKE, S=4, Hq=8, Hkv=2,
             D=64, NB=64, B=16, ks=FAKE, vs=FAKE, sm=0.125, ps=0, ws=None, wsb=0, slots=None, out=FAKE)
    a.update(kw)
    head = [a["q"], a["kn"], a["vn"], a["kc"], a["vc"], a["bt"], a["mb"], a["cl"], a["S"], a["Hq"],
            a["Hkv"], a["D"], a["NB"], a["B"], a["ks"], a["vs"]]
    tail = [a["sm"], a["ps"], a["ws"], a["wsb"], a["slots"], a["out"], None]
    return getattr(lib, fn)(*head, *([] if qsc is None else [qsc]), *tail)


@pytest.mark.parametrize("fn,qsc", [("pa_decode_step_scaled", None), ("pa_decode_step_fp8_qk", 0.05)])
@pytest.mark.parametrize("kw,status", [
    (dict(ks=None), 1),                             # scale arrays are required
    (dict(vn=None), 1),                             # K and V new rows come together
    (dict(out=ctypes.c_void_p((1 << 20) + 8)), 1),
    (dict(ps=32), 3),
    (dict(B=8), 2),
])
def test_scaled_steps_reject_on_host(lib, fn, qsc, kw, status):
    assert _step_scaled(lib, fn, qsc, **kw) == status
    assert lib.pa_last_error()


@pytest.mark.parametrize("qsc", [0.0, -1.0, float("inf"), float("nan")])
def test_fp8_qk_rejects_bad_query_scale(lib, qsc):
    assert _step_scaled(lib, "pa_decode_step_fp8_qk", qsc) == 1
    assert b"q_scale" in lib.pa_last_error()


def test_empty_scaled_steps_are_no_ops(lib):
    assert _step_scaled(lib, "pa_decode_step_scaled", None, S=0, q=None, out=None) == 0
    assert _step_scaled(lib, "pa_decode_step_fp8_qk", 0.05, S=0, q=None, out=None) == 0


def test_scaled_append_rejects_on_host(lib):
    assert lib.pa_cache_append_scaled(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 64, 2, 64, 16, None, FAKE, None) == 1
    assert lib.pa_cache_append_scaled(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 64, 2, 96, 16, FAKE, FAKE, None) == 2
    assert lib.pa_cache_append_scaled(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 64, 2, 64, 8, FAKE, FAKE, None) == 2
    assert lib.pa_cache_append_scaled(None, FAKE, FAKE, 4, FAKE, FAKE, 64, 2, 64, 16, FAKE, FAKE, None) == 1
    assert lib.pa_cache_append_scaled(FAKE, FAKE, FAKE, 0, FAKE, FAKE, 64, 2, 64, 16, FAKE, FAKE, None) == 0


def _alloc(lib, **kw):
    a = dict(bt=FAKE, mb=16, cl=FAKE, S=4, B=16, adv=1, free=FAKE, fc=FAKE, rc=FAKE, NB=64, kc=FAKE,
             vc=FAKE, Hkv=2, D=64, dt=0, cow=FAKE)
    a.update(kw)
    return lib.pa_block_alloc(a["bt"], a["mb"], a["cl"], a["S"], a["B"], a["adv"], a["free"], a["fc"],
                              a["rc"], a["NB"], a["kc"], a["vc"], a["Hkv"], a["D"], a["dt"], a["cow"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(NB=0), 1),
    (dict(mb=0), 1),
    (dict(S=-1), 1),
    (dict(S=16385), 2),
    (dict(D=96), 2),
    (dict(B=8), 2),
    (dict(dt=7), 2),
    (dict(free=None), 1),
    (dict(cow=None), 1),
    (dict(kc=ctypes.c_void_p((1 << 20) + 4)), 1),
])
def test_block_alloc_rejects_on_host(lib, kw, status):
    assert _alloc(lib, **kw) == status
    assert lib.pa_last_error()


def test_empty_block_alloc_is_a_no_op(lib):
    assert _alloc(lib, S=0, bt=None, free=None) == 0


def _alloc_chunk(lib, **kw):
    a = dict(bt=FAKE, mb=8, cl=FAKE, qs=FAKE, S=4, B=16, free=FAKE, fc=FAKE, rc=FAKE, NB=64, kc=FAKE,
             vc=FAKE, Hkv=2, D=64, dt=0, cow=FAKE)
    a.update(kw)
    return lib.pa_block_alloc_chunk(a["bt"], a["mb"], a["cl"], a["qs"], a["S"], a["B"], a["free"], a["fc"],
                                    a["rc"], a["NB"], a["kc"], a["vc"], a["Hkv"], a["D"], a["dt"], a["cow"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(NB=0), 1),
    (dict(mb=0), 1),
    (dict(S=-1), 1),
    (dict(S=16385), 2),
    (dict(D=96), 2),
    (dict(B=8), 2),
    (dict(dt=7), 2),
    (dict(qs=None), 1),
    (dict(free=None), 1),
    (dict(cow=None), 1),
    (dict(kc=ctypes.c_void_p((1 << 20) + 4)), 1),
])
def test_block_alloc_chunk_rejects_on_host(lib, kw, status):
    assert _alloc_chunk(lib, **kw) == status
    assert lib.pa_last_error()


def test_empty_block_alloc_chunk_is_a_no_op(lib):
    assert _alloc_chunk(lib, S=0, bt=None, qs=None, free=None) == 0



def test_prefill_scaled_checks_on_host(lib):
    a = [FAKE, FAKE, FAKE, FAKE, 16, FAKE, FAKE, 4, 64, 32, 8, 2, 128, 64, 16, FAKE, FAKE, 0.088, FAKE, None]
    bad = list(a)
    bad[15] = None                                       # no K scales
    assert lib.pa_prefill_scaled(*bad) == 1 and lib.pa_last_error()
    bad = list(a)
    bad[12] = 64                                         # E4M3 caches: head_dim 128 only
    assert lib.pa_prefill_scaled(*bad) == 2 and lib.pa_last_error()
    bad = list(a)
    bad[10], bad[11] = 6, 2                              # group of 3
    assert lib.pa_prefill_scaled(*bad) == 2
    empty = list(a)
    empty[8] = 0                                         # no chunk rows: nothing to do
    assert lib.pa_prefill_scaled(*empty) == 0

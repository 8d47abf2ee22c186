"""The Python binding's host-side checks, without a GPU: arguments that are
not CUDA tensors, or have the wrong dtype, rank or layout, are refused before
any call reaches the library, and a failing status becomes a
PagedAttentionError that carries the library's message."""
import pytest
import torch

from paged_kv_cache_193_gb300 import api


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from paged_kv_cache_193_gb300 import build
    build.build()


def _host_tables():
    return torch.zeros(4, 8, dtype=torch.int32), torch.ones(4, dtype=torch.int32)


def test_host_tensors_are_refused():
    bt, cl = _host_tables()
    with pytest.raises(ValueError, match="CUDA tensor"):
        api.slot_mapping(bt, cl, 16)
    q = torch.zeros(4, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        api.decode(q, q, q, bt, cl)


def test_non_tensors_are_refused():
    with pytest.raises(TypeError, match="torch.Tensor"):
        api.slot_mapping([[0]], torch.ones(1, dtype=torch.int32), 16)


@pytest.mark.parametrize("t,err,match", [
    (torch.zeros(4, 8, dtype=torch.int64), TypeError, "dtype"),
    (torch.zeros(4, 8, 2, dtype=torch.int32), ValueError, "dimensions"),
    (torch.zeros(8, 4, dtype=torch.int32).t(), ValueError, "contiguous"),
])
def test_need_refuses_wrong_dtype_rank_and_layout(t, err, match, monkeypatch):
    # the device check comes first; pretend the tensor lives on the GPU to
    # reach the later checks
    monkeypatch.setattr(torch.Tensor, "device", property(lambda self: torch.device("cuda", 0)))
    with pytest.raises(err, match=match):
        api._need(t, "block_tables", (torch.int32,), 2)


def test_failing_status_raises_with_the_library_message():
    lib = api._lib_handle()
    st = lib.pa_cache_append(None, None, None, 4, None, None, 64, 2, 96, 16, 0, 1.0, None)
    assert st == 2  # head_dim 96 is not supported
    with pytest.raises(api.PagedAttentionError, match="96"):
        api._check(st)
    api._check(0)  # PA_OK passes silently


def test_prefill_and_chunk_allocation_refuse_host_tensors():
    bt, cl = _host_tables()
    qs = torch.zeros(5, dtype=torch.int32)
    q = torch.zeros(4, 8, 128, dtype=torch.bfloat16)
    kc = torch.zeros(8, 2, 16, 128, dtype=torch.uint8)
    sc = torch.ones(2, dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        api.prefill_scaled(q, kc, kc, bt, cl, qs, 4, sc, sc)
    with pytest.raises(ValueError, match="CUDA tensor"):
        api.prefill(q, kc, kc, bt, cl, qs, 4, kv_scale=0.5)
    pool = api.DeviceBlockPool.__new__(api.DeviceBlockPool)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pool.allocate_chunk(bt, cl, qs, kc, kc)

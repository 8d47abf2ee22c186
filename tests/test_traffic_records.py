"""The committed DRAM-traffic records that bench.py puts in its roofline
line: well-formed, each citing a committed profile summary, and found by
the benchmark's lookup when the kernel source digest matches (a digest that
no longer matches makes the lookup return None, never a stale figure)."""
import json
import os
import sys
from types import SimpleNamespace

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


@pytest.mark.parametrize("name", ["decode_traffic.json", "prefill_traffic.json"])
def test_records_are_well_formed(name):
    with open(os.path.join(ROOT, "profiles", name)) as f:
        rec = json.load(f)
    assert rec
    for key, e in rec.items():
        assert isinstance(e["dram_bytes_per_launch"], int) and e["dram_bytes_per_launch"] > 0, key
        assert len(e["source_digest"]) == 16, key
        assert os.path.exists(os.path.join(ROOT, e["profile"])), (key, e["profile"])
        assert e["how"].startswith("ncu"), key


def test_prefill_lookup_follows_the_digest(monkeypatch):
    import bench
    sh = SimpleNamespace(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16)
    with open(os.path.join(ROOT, "profiles", "prefill_traffic.json")) as f:
        want = json.load(f)["S16/C512/H32/KV8/D128/B16"]
    monkeypatch.setattr(bench, "source_digest", lambda sources=None: want["source_digest"])
    assert bench.recorded_prefill_traffic(sh, 512, 16) == want["dram_bytes_per_launch"]
    assert bench.recorded_prefill_traffic(sh, 256, 16) is None  # another workload shape
    monkeypatch.setattr(bench, "source_digest", lambda sources=None: "0" * 16)
    assert bench.recorded_prefill_traffic(sh, 512, 16) is None  # the kernel changed since

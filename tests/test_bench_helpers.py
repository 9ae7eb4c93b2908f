"""bench.py host helpers (no GPU): the L2 rule per workload and the digest
that keeps a committed DRAM-traffic record valid."""
import importlib.util
import shutil
from pathlib import Path

import pytest

from kv_cache_quantization_store_gb300 import workloads as W

ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", ROOT / "bench.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name,slot,flush", [("c0", 62, True), ("c1", 118, True), ("c2", 196, False),
                                             ("c3", 102, False), ("c4", 262, False)])
def test_l2_flush_only_where_inputs_fit_in_l2(bench, name, slot, flush):
    assert bench.needs_l2_flush(W.named(name), slot) is flush


def test_traffic_digest_ignores_comments_not_code(bench, tmp_path, monkeypatch):
    src = ROOT / "kv_cache_quantization_store_gb300" / "csrc"
    dst = tmp_path / "kv_cache_quantization_store_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in src.glob("tq_decode*"):
        shutil.copy(f, dst / f.name)
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    base = bench.decode_source_digest()
    target = dst / "tq_decode.cu"
    text = target.read_text()
    target.write_text("// an added comment line\n" + text.replace("\n", "\n  ", 3) + "/* trailing */\n")
    assert bench.decode_source_digest() == base
    target.write_text(text.replace("kCombineMaxWarps = 8", "kCombineMaxWarps = 4", 1))
    assert bench.decode_source_digest() != base

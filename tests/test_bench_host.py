"""bench.py's host logic for the roofline's `traffic` field: the stored ncu
byte counts are reported only while the code of the kernel (its source file
and the headers it includes) is the code they were taken on.  Edits of
comments or layout keep them; any edit of the code drops them to null."""
import json
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

CSRC = os.path.join("vocab_sharded_lm_gb300", "csrc")


@pytest.fixture()
def tree(tmp_path, monkeypatch):
    """A copy of the kernel sources under a temporary root that bench.py reads."""
    shutil.copytree(os.path.join(ROOT, CSRC), tmp_path / CSRC)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def _edit(root, name, old, new):
    p = root / CSRC / name
    text = p.read_text()
    assert old in text
    p.write_text(text.replace(old, new, 1))


def test_hash_ignores_comments_and_layout(tree):
    h0 = bench._kernel_source_hash("stream_fused_kernel")
    _edit(tree, "vpce_fused.cu", "namespace vpce {", "// a new comment line\n/* and a block\n   comment */\nnamespace   vpce\n{")
    assert bench._kernel_source_hash("stream_fused_kernel") == h0


def test_hash_follows_code_of_file_and_shared_headers(tree):
    h0 = {k: bench._kernel_source_hash(k) for k in bench._KERNEL_FILES}
    _edit(tree, "vpce_fused.cu", "constexpr int kSSlots = 3;", "constexpr int kSSlots = 4;")
    h1 = {k: bench._kernel_source_hash(k) for k in bench._KERNEL_FILES}
    assert h1["stream_fused_kernel"] != h0["stream_fused_kernel"]
    assert all(h1[k] == h0[k] for k in h0 if k != "stream_fused_kernel")
    # a header every kernel includes
    _edit(tree, "vpce_device.cuh", "namespace vpce {", "namespace vpce {\nconstexpr int kUnused = 1;")
    h2 = {k: bench._kernel_source_hash(k) for k in bench._KERNEL_FILES}
    assert all(h2[k] != h1[k] for k in h1)


def test_traffic_reported_only_for_matching_code(tree):
    entry = {"dram_bytes_per_launch": 123, "read": 100, "write": 23,
             "source_hash": bench._kernel_source_hash("backward_kernel")}
    (tree / "profiles" / "ncu_traffic.json").write_text(json.dumps({"backward_kernel": {"wl": entry}}))
    assert bench._ncu_traffic("backward_kernel", "wl") == 123
    assert bench._ncu_traffic("backward_kernel", "other") is None
    assert bench._ncu_traffic("stream_fused_kernel", "wl") is None
    _edit(tree, "vpce_backward.cu", "kc % kStages", "kc % unsigned(kStages)")
    assert bench._ncu_traffic("backward_kernel", "wl") is None


def test_stored_traffic_is_consistent():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        d = json.load(f)
    for kernel, workloads in d.items():
        if kernel.startswith("_"):
            continue
        assert kernel in bench._KERNEL_FILES
        for name, e in workloads.items():
            assert len(e["source_hash"]) == 16
            if "dram_bytes_per_launch" in e:
                assert e["dram_bytes_per_launch"] == e["read"] + e["write"] > 0

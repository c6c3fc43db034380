"""bench.py's use of the committed DRAM counters (CPU only).

roofline.traffic must come from an ncu capture of the kernels as they are: the
counters carry a hash of the kernel sources, a formatting change keeps them, any
other edit voids them (bench then reports null).  Run on a copy of the sources.
"""
import json
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.fixture
def tree(tmp_path, monkeypatch):
    src = os.path.join(ROOT, "bwd_gemm_epilogue_gb300", "csrc")
    dst = tmp_path / "bwd_gemm_epilogue_gb300" / "csrc"
    shutil.copytree(src, dst, ignore=shutil.ignore_patterns("*.o", "*.so"))
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def _write_counters(root, bytes_per_launch=123456789):
    data = {"source_hash": bench.kernel_source_hash(),
            "kernels": {"bwd_gemms": {"dram_bytes_per_launch": bytes_per_launch}}}
    (root / "profiles" / "traffic.json").write_text(json.dumps(data))


def _kernel_file(root):
    return root / "bwd_gemm_epilogue_gb300" / "csrc" / "gemm_kernel.cuh"


def test_counters_are_reported_for_the_sources_they_were_taken_with(tree):
    _write_counters(tree)
    assert bench.measured_traffic("bwd_gemms") == 123456789
    assert bench.measured_traffic("bwd_gemms", workload="decode") is None
    assert bench.measured_traffic("no_such_kernel") is None


def test_formatting_change_keeps_the_counters(tree):
    _write_counters(tree)
    f = _kernel_file(tree)
    text = f.read_text()
    f.write_text(text.replace("\n    ", "\n        ").replace(" = ", "  =  ") + "\n\n")
    assert bench.measured_traffic("bwd_gemms") == 123456789


def test_code_edit_voids_the_counters(tree):
    _write_counters(tree)
    f = _kernel_file(tree)
    text = f.read_text()
    assert "SRC_TABLE = 2" in text
    f.write_text(text.replace("SRC_TABLE = 2", "SRC_TABLE = 4", 1))
    assert bench.measured_traffic("bwd_gemms") is None


def test_renaming_a_file_voids_the_counters(tree):
    _write_counters(tree)
    f = _kernel_file(tree)
    f.rename(f.with_name("gemm_kernel2.cuh"))
    assert bench.measured_traffic("bwd_gemms") is None

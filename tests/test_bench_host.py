"""Host logic of bench.py (CPU): the source hash that keeps the ncu traffic
record tied to the kernel sources it was taken on, the record lookup, and
the description of the GEMM tile shapes."""

import json
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_code_only_drops_comments_and_blank_lines():
    src = "int a; // note\n/* block\n comment */\n\nint b;   \n"
    assert bench._code_only(src) == "int a;\nint b;"


@pytest.fixture
def fake_root(tmp_path, monkeypatch):
    csrc = tmp_path / "top_kl_loss_tcgen05_b300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("__global__ void k() {}\n")
    (csrc / "h.h").write_text("#define X 1\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def test_hash_ignores_comments_but_not_code(fake_root):
    csrc = fake_root / "top_kl_loss_tcgen05_b300" / "csrc"
    h0 = bench.kernel_src_hash(["k.cu"])
    (csrc / "k.cu").write_text("// a comment\n__global__ void k() {}  // why\n")
    assert bench.kernel_src_hash(["k.cu"]) == h0
    (csrc / "h.h").write_text("#define X 2\n")  # not in the list
    assert bench.kernel_src_hash(["k.cu"]) == h0
    assert bench.kernel_src_hash() != h0  # all files
    (csrc / "k.cu").write_text("__global__ void k() { int x = 1; }\n")
    assert bench.kernel_src_hash(["k.cu"]) != h0


def test_traffic_record_only_while_the_sources_match(fake_root):
    rec = {"grad_dH_dW": {"llama3b": {"src_files": ["k.cu"], "src_sha": bench.kernel_src_hash(["k.cu"]),
                                      "dram_bytes_per_launch": 123}}}
    (fake_root / "profiles" / "ncu_traffic.json").write_text(json.dumps(rec))
    assert bench.ncu_traffic("grad_dH_dW", "llama3b") == 123
    assert bench.ncu_traffic("grad_dH_dW", "gptoss20b") is None
    assert bench.ncu_traffic("topk_cache", "topk") is None
    (fake_root / "top_kl_loss_tcgen05_b300" / "csrc" / "k.cu").write_text("__global__ void k() { return; }\n")
    assert bench.ncu_traffic("grad_dH_dW", "llama3b") is None


def test_committed_traffic_record_lists_existing_sources():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        d = json.load(f)
    csrc = os.path.join(ROOT, "top_kl_loss_tcgen05_b300", "csrc")
    for kernel, per in d.items():
        if kernel.startswith("_"):
            continue
        for wl, e in per.items():
            assert e["src_files"] and all(os.path.exists(os.path.join(csrc, f)) for f in e["src_files"])
            assert e["dram_bytes_per_launch"] >= e["algorithmic_bytes_per_launch"] * 0.9


def test_gemm_tiles_description(monkeypatch):
    monkeypatch.delenv("KD_GEMM_WIDE", raising=False)
    monkeypatch.setenv("KD_GEMM_CTA2", "0")
    assert bench.gemm_tiles_desc() == "128x256 per CTA"
    monkeypatch.setenv("KD_GEMM_CTA2", "1")
    assert "dz recompute" in bench.gemm_tiles_desc()
    monkeypatch.setenv("KD_GEMM_WIDE", "1")
    assert bench.gemm_tiles_desc().startswith("256x512") and "every GEMM" in bench.gemm_tiles_desc()


def test_max_over_ranks_single_process():
    assert bench.max_over_ranks(3.5, 1) == 3.5

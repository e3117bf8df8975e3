"""Host logic of bench.py (CPU): the source hash that keeps the ncu traffic
record tied to the kernel sources it was taken on, the record lookup, and
the description of the GEMM tile shapes."""

import json
import os
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


def test_gemm_tiles_description():
    from top_kl_loss_tcgen05_b300 import _native

    try:
        assert bench.gemm_tiles_desc().startswith("256x512")  # the defaults
        _native.set_gemm_tiles(0, -1)
        assert bench.gemm_tiles_desc() == "128x256 per CTA"
        _native.set_gemm_tiles(1, 0)
        assert bench.gemm_tiles_desc().startswith("256x256") and "every GEMM" in bench.gemm_tiles_desc()
        _native.set_gemm_tiles(1, 1)
        assert bench.gemm_tiles_desc().startswith("256x512") and "every GEMM" in bench.gemm_tiles_desc()
    finally:
        _native.set_gemm_tiles(-1, -1)


def test_default_group_is_the_library_rule():
    """bench's description of the rows per GEMM launch follows the group the
    library picks: the default workspace equals the explicit-group one."""
    from top_kl_loss_tcgen05_b300 import _native

    L = _native.lib()
    for name in ("tiny", "llama3b", "gptoss20b", "long"):
        c = bench.synth.CONFIGS[name]
        G = bench.default_group(c["chunk"])
        assert L.kd_fused_kl_workspace_size(c["d"], c["V"], c["K"], c["chunk"]) == \
            L.kd_fused_kl_workspace_size_ex(c["d"], c["V"], c["K"], c["chunk"], G)
    for chunk in (1, 100, 1024, 1500, 2048, 3000, 4096, 10000):
        G = bench.default_group(chunk)
        assert L.kd_fused_kl_workspace_size(256, 4096, 16, chunk) == \
            L.kd_fused_kl_workspace_size_ex(256, 4096, 16, chunk, G)


def test_roofline_fields_from_a_profile():
    """The dominant kernel's achieved rate is its per-launch algorithmic flops
    over its mean launch time, reported against the sustained and burst peaks
    and clock-normalised."""
    T, d, V, steps = 4096, 2880, 201088, 2
    prof = {"grad_dH_dW": (2, 2 * 3.0), "logits_dz": (2, 2 * 1.5), "logits_fwd_lse_gather": (2, 2 * 1.4),
            "teacher_prep": (2, 0.02)}
    peaks = {"bf16_tflops_sustained": 1400.0, "bf16_tflops": 1800.0, "clocks_under_load": {"sm_mhz_median": 1200.0}}
    roof, kernels, launches = bench.fused_roofline(prof, steps, T, d, V, peaks, "measured", {"sm_mhz": 1800.0},
                                                   "long")
    assert roof["kernel"] == "grad_dH_dW" and launches == 8
    achieved = 4.0 * T * d * V / 3.0e-3 / 1e12
    assert abs(roof["achieved"] - achieved) < 1e-6 * achieved
    assert abs(roof["frac"] - achieved / 1400.0) < 1e-9
    assert abs(roof["frac_burst"] - achieved / 1800.0) < 1e-9
    assert abs(roof["frac_clock_normalised"] - achieved / (1400.0 * 1800.0 / 1200.0)) < 1e-9
    assert abs(sum(k["share"] for k in kernels.values()) - 1.0) < 1e-9


def test_max_over_ranks_single_process():
    assert bench.max_over_ranks(3.5, 1) == 3.5


@pytest.mark.parametrize("a,b,cap", [(0.0, 0.01, 4096), (5.0, 0.01, 4096), (0.5, 0.2, 4096), (0.0, 1e-5, 300)])
def test_oracle_sample_sizing_never_overshoots(monkeypatch, a, b, cap):
    """size_sample picks rows whose oracle time stays within the budget for
    any per-call cost a >= 0 and per-row cost b (time = a + b r), and never
    more rows than the sample holds."""
    calls = []

    def fake(cw, rows):
        calls.append(rows)
        return a + b * rows

    monkeypatch.setattr(bench, "oracle_sample", fake)
    budget = 6.0
    rows = bench.size_sample({"ids": [0] * cap}, budget)
    assert 2 <= rows <= cap
    if a < budget:
        assert a + b * rows <= budget * 1.0001
    if a + b * cap <= budget / 3:
        assert rows == cap
    assert sum(a + b * r for r in calls) < 4 * budget + 10 * a  # probing stays bounded


def test_workload_description_names_a_truncated_run():
    """A --rows capture run says it covers only the first positions; the
    full workload's description is the plain shape."""
    assert bench.describe("long") == "long: T=262144 d=2880 V=201088 K=100 chunk=4096"
    d = bench.describe("long", 8192)
    assert d.startswith("long: T=8192 d=2880 V=201088 K=100 chunk=4096") and "first 8192 of its 262144" in d
    assert bench.describe("tiny", 10**9) == bench.describe("tiny")

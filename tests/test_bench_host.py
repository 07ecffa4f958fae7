"""Host logic of bench.py that needs no GPU: the key that ties the committed
DRAM-traffic record to the kernel sources, and the lookup it gates."""
import json
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

KERNELS = ("bwd.cu", "fwd.cu", "ptx.cuh")


def _copy_tree(tmp_path):
    """A copy of the files the key covers, laid out as in the repository."""
    csrc = tmp_path / "causal_gqa_flashattention_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in KERNELS:
        shutil.copy(os.path.join(ROOT, "causal_gqa_flashattention_gb300", "csrc", f), csrc / f)
    (tmp_path / "profiles").mkdir()
    return csrc


def test_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    csrc = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_file_hash()
    assert h0 == bench.kernel_file_hash()  # stable
    fwd = csrc / "fwd.cu"
    src = fwd.read_text()
    # a comment line, a trailing comment and a blank line leave it unchanged
    fwd.write_text("// a note\n\n" + src.replace("namespace nea {", "namespace nea {  // x", 1))
    assert bench.kernel_file_hash() == h0
    # a change of code does not
    fwd.write_text(src.replace("kRescaleLog2 = 8.0f", "kRescaleLog2 = 7.0f", 1))
    assert bench.kernel_file_hash() != h0


def test_traffic_only_for_matching_sources(tmp_path, monkeypatch):
    csrc = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("bwd_main", "gpt2s_bf16") is None  # no record at all
    rec = {"kernel_hash": bench.kernel_file_hash(), "workload_key": "gpt2s_bf16",
           "per_launch_bytes": {"bwd_main": 123}}
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    assert bench.traffic_for("bwd_main", "gpt2s_bf16") == 123
    assert bench.traffic_for("fwd", "gpt2s_bf16") is None
    bwd = csrc / "bwd.cu"
    bwd.write_text(bwd.read_text() + "\nint unused_symbol_for_the_test;\n")
    assert bench.traffic_for("bwd_main", "gpt2s_bf16") is None  # counters taken on other code


def test_traffic_only_for_the_workload_it_was_taken_on(tmp_path, monkeypatch):
    _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"kernel_hash": bench.kernel_file_hash(), "workload_key": "gpt2s_bf16",
           "per_launch_bytes": {"bwd_main": 123}}
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    assert bench.traffic_for("bwd_main", "gpt2s_bf16") == 123
    for other in ("long_bf16", "wide_bf16", "tiny_f32", "gpt2s_f32"):
        assert bench.traffic_for("bwd_main", other) is None
    del rec["workload_key"]  # a record that does not say which workload it measured
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    assert bench.traffic_for("bwd_main", "gpt2s_bf16") is None


def test_gpus_flag_is_honoured():
    # launched by torchrun: the flag must agree with the launcher
    assert bench.check_gpus(4, 4, 8) == "run"
    assert "launcher started 2" in bench.check_gpus(4, 2, 8)
    # launched directly: one GPU runs here, more GPUs start local ranks
    assert bench.check_gpus(1, None, 1) == "run"
    assert bench.check_gpus(8, None, 8) == "spawn"
    assert "only 1 GPU" in bench.check_gpus(2, None, 1)
    assert "at least 1" in bench.check_gpus(0, None, 8)

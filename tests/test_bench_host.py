"""Host logic of bench.py that needs no GPU: the kernel-source hash that keys
the committed ncu traffic figures, and their lookup."""
import json
import os
import shutil

import bench


def test_code_only_strips_comments_and_keeps_literals():
    src = 'int a = 1; // note\n/* block\n comment */ const char* s = "x // y /* z */";\nchar c = \'/\';'
    assert bench.code_only(src) == 'int a = 1; const char* s = "x // y /* z */"; char c = \'/\';'
    assert bench.code_only("a  \n\t b") == "a b"
    assert bench.code_only('s = "a\\"//b"; // c') == 's = "a\\"//b";'


def _tree(tmp_path):
    csrc = tmp_path / "lsd_radix_sort_key_gb300" / "csrc"
    shutil.copytree(os.path.join(bench.ROOT, "lsd_radix_sort_key_gb300", "csrc"), csrc,
                    ignore=shutil.ignore_patterns("obj", "*.o"))
    return csrc


def test_source_hash_follows_code_not_comments(tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    kern = csrc / "rs_kernels.cuh"
    kern.write_text(kern.read_text() + "\n// a new comment\n/* and another */\n")
    assert bench.kernel_source_hash() == h0
    api = csrc / "rs_api.cu"  # the host entry layer is not device code
    api.write_text(api.read_text() + "\nstatic int unused_host_symbol = 0;\n")
    assert bench.kernel_source_hash() == h0
    kern.write_text(kern.read_text() + "\nnamespace rs { constexpr int kUnused = 1; }\n")
    assert bench.kernel_source_hash() != h0


def test_traffic_lookup_needs_the_same_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps(
        {"downsweep:w": {"dram_bytes_per_launch": 123, "source_hash": "abc"}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc")
    assert bench.ncu_traffic("downsweep", "w") == 123
    assert bench.ncu_traffic("upsweep", "w") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "def")
    assert bench.ncu_traffic("downsweep", "w") is None


def test_committed_traffic_records_are_well_formed():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        data = json.load(f)
    entries = {k: v for k, v in data.items() if not k.startswith("_")}
    assert "downsweep:u32_uniform_2p28" in entries
    for key, v in entries.items():
        kind, workload = key.split(":")
        assert kind and workload
        assert isinstance(v["dram_bytes_per_launch"], int) and v["dram_bytes_per_launch"] > 0
        assert len(v["source_hash"]) == 16


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the CPU oracle timed as the reference
    arm) prints one JSON line with the contract's keys; a 2^16-key workload
    keeps it quick."""
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "u32_uniform_2p16", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=bench.ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 2
    assert line["config"]["workload"] == "u32_uniform_2p16"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_cpu_baseline_reports_host_and_extra_sorts():
    import synth
    w = synth.WORKLOADS["u32_uniform_2p16"]
    cb = bench.cpu_baseline(w, w.key_type, w.begin_bit, w.end_bit, w.log2n, budget_s=0.2)
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] > 0
    host = cb["host"]
    assert host["cores_online"] >= 1 and host["hardware_concurrency"] >= 1
    kinds = [o["kind"] for o in cb["others"]]
    assert kinds == ["std::stable_sort", "one_bit_split", "parallel_lsd"]
    assert all(o["value"] > 0 for o in cb["others"])
    assert [o["cores"] for o in cb["others"][:2]] == [1, 1] and cb["others"][2]["cores"] >= 1

"""Host-side logic of the benchmark (CPU): mode strings, the algorithmic byte counts behind
the roofline, and the launch counts behind its `gpu_launches` claim."""
import pytest

import bench
import workloads


def test_parse_mode():
    assert bench.parse_mode("q8") == ("q8", {})
    assert bench.parse_mode("q8/bs256/p99/sr/approx") == (
        "q8", {"block_size": 256, "percentile": 99.0, "stochastic_rounding": True, "approx_update": True})
    assert bench.parse_mode("bf16m/approx") == ("bf16m", {"approx_update": True})
    for bad in ("q4", "bf16m/bs256", "fp32/sr", "q8/xyz"):
        with pytest.raises(SystemExit):
            bench.parse_mode(bad)


def test_algorithmic_bytes_per_param():
    # p read + write 8, g 4 (bf16 2), m and v read + write; 8-bit scales: 4 bytes read and
    # written per block and moment
    n = 2048 * 1000
    assert bench.algorithmic_bytes("fp32", [n], "f32") == 28 * n
    assert bench.algorithmic_bytes("bf16m", [n], "f32") == 20 * n
    assert bench.algorithmic_bytes("q8", [n], "f32") == 16 * n + 16 * 1000
    assert bench.algorithmic_bytes("q8v", [n], "f32") == 22 * n + 8 * 1000
    assert bench.algorithmic_bytes("q8", [n], "bf16") == 14 * n + 16 * 1000
    assert bench.algorithmic_bytes("fp32", [n], "f32", zero_grads=True) == 32 * n
    # a partial last block still has its scales; another block size scales the overhead
    assert bench.algorithmic_bytes("q8", [2049], "f32") == 16 * 2049 + 16 * 2
    assert bench.algorithmic_bytes("q8", [n], "f32", block_size=256) == 16 * n + 16 * (n // 256)


def test_launches_per_call():
    assert bench.launches_per_call([]) == 0
    assert bench.launches_per_call([0, 0]) == 0
    assert bench.launches_per_call([5] * 8) == 1
    assert bench.launches_per_call([5] * 9) == 1            # the 440-entry parameter block
    assert bench.launches_per_call([5] * 440) == 1
    assert bench.launches_per_call([5] * 441) == 2
    assert bench.launches_per_call([5] * 8 + [0] * 3) == 1  # empty tensors take no slot
    assert bench.launches_per_call(workloads.WORKLOADS["vit_base"].sizes) == 1
    assert bench.launches_per_call(workloads.WORKLOADS["gpt_1p3b"].sizes) == 1


def test_from_host_launches():
    # one chunk: the plain call
    assert bench.from_host_launches([1 << 24], 1, 2048) == 1
    # 8 chunks of one 16.7M tensor: 8 slices, one launch each
    assert bench.from_host_launches([1 << 24], 8, 2048) == 8
    # a chunk never splits below one cut unit (4 blocks of 2048)
    assert bench.from_host_launches([8192], 8, 2048) == 1
    # whole small tensors share a chunk (a chunk is at least one cut unit): one chunk, one launch
    assert bench.from_host_launches([100] * 16, 2, 2048) == 1
    # no cut past 4 * INT_MAX elements: a 2^34-element tensor in 8 chunks of 2^31 gives
    # cuts at 2^31, 2^32 and 3 * 2^31, then the rest as one slice
    assert bench.from_host_launches([1 << 34], 8, 2048) == 4
    assert bench.from_host_launches([1 << 32], 8, 2048) == 8


def test_workload_sizes_match_the_stated_counts():
    w = workloads.WORKLOADS
    assert len(w["vit_base"].sizes) == 148 and sum(w["vit_base"].sizes) == 86_564_352
    assert len(w["gpt_1p3b"].sizes) == 292 and sum(w["gpt_1p3b"].sizes) == 1_315_819_520
    assert w["flat_16m"].sizes == [16_777_216]
    assert w["flat_1g_heavy"].sizes == [1 << 30]


def test_clock_sampler_sees_samples_while_it_runs(tmp_path, monkeypatch):
    # a stand-in for nvidia-smi that, like it, buffers its output fully unless it writes to a
    # terminal: the sampler must see its lines while it runs, not only when it exits
    import os
    import sys
    import time
    fake = tmp_path / "nvidia-smi"
    fake.write_text(
        f"#!{sys.executable}\n"
        "import time\n"
        "for i in range(200):\n"
        "    print('GPU-1, %d, 2070, 500.0, Not Active, Not Active, Not Active, %s'\n"
        "          % (2070 - i % 2, 'Active' if i == 3 else 'Not Active'))\n"
        "    time.sleep(0.05)\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    c = bench.ClockSampler("GPU-1")
    c.start()
    time.sleep(1.0)
    got = c.stop()
    assert got is not None and got["samples"] >= 5
    assert got["sm_max_mhz"] == 2070.0 and 2069.0 <= got["sm_mhz"] <= 2070.0
    assert got["reasons"] == ["sw_power_cap"]


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))
    c = bench.ClockSampler(None)
    c.start()
    assert c.stop() is None


def test_both_arms_report_the_same_config(monkeypatch, capsys):
    """The reference arm (the CPU oracle) prints the very `config` dict the GPU arm prints for
    the same workload and mode, so the two lines describe one workload."""
    monkeypatch.setattr(bench, "oracle_sample_rate", lambda w, spec, budget, threads=1: (1e-3, "stub sample"))
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3"])
    bench.main()
    import json
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    w = workloads.WORKLOADS["gpt_1p3b"]
    assert line["impl"] == "reference"
    assert line["config"] == bench.workload_config(w, "q8", False, 2, 3)
    assert line["config"]["workload"] == "gpt_1p3b" and line["config"]["params"] == 1_315_819_520


def test_grad_sets_stay_within_budget():
    for name, w in workloads.WORKLOADS.items():
        n = bench.n_grad_sets(w, 20, 5)
        per = sum(w.sizes) * (4 if w.grad_dtype == "f32" else 2)
        assert 2 <= n <= 8
        assert n == 2 or n * per <= bench.GRAD_SET_BUDGET, name


def test_kernel_hash_ignores_comments_not_code():
    """The stored ncu traffic stays attached to a kernel through comment edits only."""
    base = {"k.cu": 'int f(int x) {  // twice\n  return 2 * x; /* doubled */ }\nconst char* s = "a // b";\n'}
    same = {"k.cu": 'int f(int x) {\n  // a new remark\n  return 2 * x;   }\nconst char* s = "a // b";\n'}
    code = {"k.cu": 'int f(int x) {  // twice\n  return 3 * x; /* doubled */ }\nconst char* s = "a // b";\n'}
    lit = {"k.cu": 'int f(int x) {  // twice\n  return 2 * x; /* doubled */ }\nconst char* s = "a / b";\n'}
    h = bench.kernel_source_hash(base)
    assert bench.kernel_source_hash(same) == h
    assert bench.kernel_source_hash(code) != h
    assert bench.kernel_source_hash(lit) != h

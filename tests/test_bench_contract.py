"""bench.py on the CPU: model size and flops per token against the pages'
figures, the guard that drops stale DRAM-traffic counters, and the JSON line
of the reference arm (the oracle timed on host cores).

The 1558M parameter count, 1 557 686 400 with the vocabulary padded to 50304,
is the one "Karpathy reproduces GPT-2 (1.6B) in llm.c" shows in the training
log printed after its launch command; 124 475 904 is the same formula at the
124M shape."""
import importlib.util
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_parameter_counts_match_the_pages_and_the_oracle():
    from oracle.pyoracle import param_count, padded_vocab
    b = _bench()
    w = b.WORKLOADS
    assert b.n_params(w["1558M"]["L"], w["1558M"]["C"], w["1558M"]["V"], w["1558M"]["T"]) == 1557686400
    assert b.n_params(w["124M"]["L"], w["124M"]["C"], w["124M"]["V"], w["124M"]["T"]) == 124475904
    for k in ("124M", "350M", "1558M"):
        L, C, V, T = (w[k][x] for x in ("L", "C", "V", "T"))
        assert b.n_params(L, C, V, T) == param_count(L, C, padded_vocab(V), T)


def test_flops_per_token_is_6N_plus_6LCT():
    b = _bench()
    w = b.WORKLOADS
    assert b.flops_per_token(w["124M"]) == 6 * 124475904 + 6 * 12 * 768 * 1024 == 803478528
    assert b.flops_per_token(w["1558M"]) == 6 * 1557686400 + 6 * 48 * 1600 * 1024 == 9817977600


def test_stale_traffic_counters_are_dropped(tmp_path, monkeypatch):
    b = _bench()
    csrc = tmp_path / "scratch_gpt_step_train_b300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k_attn_tc.cu").write_text("// kernel v1\n")
    (csrc / "k_misc.cu").write_text("// other kernels v1\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(b, "ROOT", os.fspath(tmp_path))
    sha = b.kernel_sources_hash()
    (tmp_path / "profiles" / "dram_traffic_gpt2_124M.txt").write_text(
        f"# counters\n# kernel_sources_sha256 {sha}\nattention_bwd 270392320\nmatmul_qkv_fwd 52000000\n")
    assert b.load_traffic("124M") == {"attention_bwd": 270392320.0, "matmul_qkv_fwd": 52000000.0}
    (csrc / "k_misc.cu").write_text("// other kernels v2\n")  # not a recorded kernel
    assert b.load_traffic("124M") == {"attention_bwd": 270392320.0, "matmul_qkv_fwd": 52000000.0}
    (csrc / "k_attn_tc.cu").write_text("// kernel v2\n")  # the kernels changed after the capture
    assert b.load_traffic("124M") is None
    assert b.load_traffic("350M") is None  # no capture at all


@pytest.mark.slow
def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([x for x in r.stdout.splitlines() if x.startswith("{")][-1])
    assert line["impl"] == "reference"
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["warmup"] >= 3 and line["steps"] == 1
    assert line["value"] > 0 and line["e2e"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert line["dtype"] == "f64" and line["data"] == "synthetic"


def test_cpu_baselines_skip_a_sample_the_host_cannot_hold(monkeypatch):
    """the 1558M oracle sample holds ~50 GB of fp64 state; with less host
    memory it is reported as skipped, with the reason, not run"""
    b = _bench()
    w = b.WORKLOADS
    need = b.oracle_bytes(w["1558M"], b.CPU_SAMPLE_1558M)
    assert 4 * 8 * 1.55e9 < need < 4 * 8 * 1.6e9 + 8e9
    calls = []

    def fake_rate(wl, sample, steps=1, warmup=0, threads=None):
        calls.append((wl["C"], sample["T"], threads))
        return 100.0, threads or 8, [1.0]
    monkeypatch.setattr(b, "cpu_oracle_step_rate", fake_rate)
    monkeypatch.setattr(b, "mem_available", lambda: 16 << 30)
    cb = b.cpu_baselines()
    assert calls == [(768, 256, None), (768, 32, 1)]
    assert cb["kind"] == "oracle" and cb["value"] == 100.0 and cb["cores"] == 8
    assert [("skipped" in r) for r in cb["runs"]] == [False, False, True]
    assert cb["runs"][1]["cores"] == 1


def test_secondary_workload_list():
    b = _bench()
    assert b.parse_secondary("1558M:3,350M:30") == [("1558M", 3), ("350M", 30)]
    assert b.parse_secondary("350M") == [("350M", 3)]
    assert b.parse_secondary("") == [] and b.parse_secondary(None) == []
    with pytest.raises(SystemExit):
        b.parse_secondary("7B:1")

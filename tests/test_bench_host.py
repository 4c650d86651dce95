"""Host-side logic of bench.py that needs no GPU: the oracle pool behind the
reported core count (single-threaded BLAS in each of one worker per core), the DRAM-traffic record that is used
only while the kernel sources are unchanged, and the algorithmic work counts."""

import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_oracle_blas_is_single_threaded_per_worker():
    pytest.importorskip("threadpoolctl")
    code = ("import bench, numpy, threadpoolctl, json; "
            "print(json.dumps([p['num_threads'] for p in threadpoolctl.threadpool_info() "
            "if p.get('user_api') == 'blas']))")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                         check=True, env={k: v for k, v in os.environ.items()
                                          if k not in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS",
                                                       "MKL_NUM_THREADS")}).stdout
    threads = json.loads(out.strip().splitlines()[-1])
    assert threads, "numpy reports no BLAS library"
    assert all(t == bench.ORACLE_BLAS_THREADS == 1 for t in threads)


def _fake_tree(tmp_path, src_text):
    csrc = tmp_path / "position_independent_kv_paged_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text(src_text)
    (tmp_path / "profiles").mkdir()
    return tmp_path


def test_traffic_record_used_only_for_unchanged_sources(tmp_path, monkeypatch):
    root = _fake_tree(tmp_path, "kernel v1")
    monkeypatch.setattr(bench, "ROOT", str(root))
    sha = bench.kernel_sources_sha256(["k.cu"])
    rec = {"w": {"sources": ["k.cu"], "source_sha256": sha, "traffic": 1234}}
    (root / "profiles" / "traffic.txt").write_text(json.dumps(rec))
    assert bench.kernel_traffic(["k.cu"], "w") == 1234
    assert bench.kernel_traffic(["k.cu"], "other") is None
    (root / "position_independent_kv_paged_gb300" / "csrc" / "k.cu").write_text("kernel v2")
    assert bench.kernel_traffic(["k.cu"], "w") is None
    assert bench.kernel_traffic(["missing.cu"], "w") is None


def test_committed_traffic_record_names_existing_sources():
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        pytest.skip("no traffic record")
    for name, rec in json.load(open(path)).items():
        assert rec["traffic"] == rec["dram_bytes_read"] + rec["dram_bytes_write"], name
        for f in rec["sources"]:
            assert os.path.exists(os.path.join(ROOT, "position_independent_kv_paged_gb300", "csrc", f)), f
        assert "--clock-control none" in rec["command"]


class _P:
    def __init__(self, cu_q_lens, kv_lens):
        self.cu_q_lens = np.asarray(cu_q_lens)
        self.kv_lens = np.asarray(kv_lens)
        self.batch = len(kv_lens)


class _W:
    def __init__(self, p, Hq, d):
        self.prefill, self.Hq, self.d = p, Hq, d


def test_prefill_flops_count_only_the_causal_key_set():
    # one request: 3 queries over 5 keys (2 cached): rows see 3, 4, 5 keys
    w = _W(_P([0, 3], [5]), Hq=2, d=4)
    assert bench.prefill_flops(w) == 4 * 2 * 4 * (3 + 4 + 5)
    # brute force over a ragged batch, with an empty chunk
    rng = np.random.default_rng(0)
    q = rng.integers(0, 40, 6)
    q[2] = 0
    kv = q + rng.integers(0, 100, 6)
    cu = np.concatenate([[0], np.cumsum(q)])
    want = 0
    for ql, kl in zip(q, kv):
        for i in range(ql):
            want += kl - ql + i + 1
    assert bench.prefill_flops(_W(_P(cu, kv), Hq=7, d=128)) == 4 * 7 * 128 * want


def test_whole_job_value_scales_with_ranks():
    assert bench.whole_job_gbs(10**9, 1, 1.0) == pytest.approx(1000.0)
    assert bench.whole_job_gbs(10**9, 4, 2.0) == pytest.approx(2000.0)


REF_CMD = [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"]


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run(REF_CMD, cwd=ROOT, capture_output=True, text=True, check=True, timeout=600).stdout
    lines = [ln for ln in out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["steps"] == 1 and d["warmup"] == 0 and d["value"] > 0 and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["value"] == d["value"] and cb["kind"] == "oracle" and cb["cores"] == (os.cpu_count() or 1)
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run(REF_CMD, cwd=ROOT, capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_only_legs_name_known_workloads_and_calls():
    # every --only leg (the commands the profiles are captured from) maps to a
    # generator and a call the bench's cases provide
    import workloads as W
    gens = {"rag_decode", "rag_decode_private", "long_decode", "rag_prefill", "mixed_batch"}
    for leg, (wname, kind, call) in bench.ONLY_LEGS.items():
        assert wname in gens, leg
        assert kind in ("decode", "prefill", "mixed"), leg
        if kind != "mixed":
            assert hasattr(bench.DecodeCase if kind == "decode" else bench.PrefillCase, call), leg
    assert callable(W.rag_decode) and callable(W.mixed_batch)
    out = subprocess.run([sys.executable, "bench.py", "--help"], cwd=ROOT, capture_output=True, text=True,
                         check=True).stdout
    assert "--only" in out

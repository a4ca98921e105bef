"""bench.py's host helpers, without a GPU: the byte counts behind every GB/s
figure, the peak lookup, the source-hash gate on recorded ncu traffic, and
the argument checks of the command line."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_algorithmic_bytes_match_the_scope_formula():
    # (n + 3) m H 2 + 2 H: n partials and the residual read, out and
    # residual_out written, the weight read once
    assert bench.algo_bytes(8, 8192, 6144) == 1_107_308_544
    assert bench.algo_bytes(2, 4, 1024) == 43_008
    assert bench.algo_bytes(8, 1, 7168) == 172_032
    for n, m, H in ((1, 1, 8), (16, 3, 131072), (4, 2048, 7168)):
        assert bench.algo_bytes(n, m, H) == ((n + 3) * m + 1) * H * 2


def test_two_stage_moves_the_temporary_twice_more():
    n, m, H = 4, 2048, 7168
    assert bench.actual_bytes(n, m, H, False) == bench.algo_bytes(n, m, H)
    assert bench.actual_bytes(n, m, H, True) == (n + 5) * m * H * 2 + H * 2


def test_peak_comes_from_the_measured_file_or_the_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks() == (bench.FALLBACK_HBM_GBS, "of fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6690.5}))
    assert bench.peaks() == (6690.5, "of measured")


def test_recorded_traffic_is_dropped_once_the_kernel_sources_change(tmp_path, monkeypatch):
    csrc = tmp_path / "allreduce_sum_residual_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    for name in ("common.cuh", "stream_epilogue.cuh"):
        (csrc / name).write_text(f"// {name}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.source_hash("k_stream_epilogue")
    rec = {"k_stream_epilogue@prefill": {"source_hash": h, "dram_bytes_per_launch": 1084702208}}
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(rec))
    assert bench.ncu_traffic("k_stream_epilogue", "prefill") == 1084702208.0
    assert bench.ncu_traffic("k_stream_epilogue", "decode") is None      # no capture
    (csrc / "stream_epilogue.cuh").write_text("// changed\n")
    assert bench.source_hash("k_stream_epilogue") != h
    assert bench.ncu_traffic("k_stream_epilogue", "prefill") is None     # stale


def test_committed_traffic_record_matches_the_current_prefill_kernel(arlib):
    """The prefill traffic figure the bench reports is only valid for the
    kernel it was captured from (the one the plan picks for the prefill
    workload); the record must carry that kernel's current source hash."""
    p = arlib.ar_get_plan(8, 8192, 6144, 0, sm_count=152)
    kernel = ("k_reduce_flat" if p["mode"] == 2 else
              "k_stream_epilogue" if p["kernel"] == arlib.AR_KERNEL_STREAM else "k_fused_epilogue")
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        rec = json.load(f)
    e = rec[f"{kernel}@prefill"]
    assert e["source_hash"] == bench.source_hash(kernel)
    # the captured launch is the one the plan makes (the device adds the
    # prefetch one wave ahead to the host plan's own-row prefetch)
    for k in bench.PLAN_KEYS:
        if k != "prefetch":
            assert e["plan"][k] == p[k], k
    assert bench.ncu_traffic(kernel, "prefill", e["plan"]) == e["dram_bytes_per_launch"]
    assert bench.ncu_traffic(kernel, "prefill", dict(e["plan"], vpt=e["plan"]["vpt"] * 2)) is None
    assert 0.9 * bench.algo_bytes(8, 8192, 6144) < e["dram_bytes_per_launch"] < \
        1.1 * bench.algo_bytes(8, 8192, 6144)


def test_warmup_below_three_is_refused():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_every_kernel_candidate_names_a_forced_shape():
    for name, shape in bench.KERNEL_CANDIDATES.items():
        kernel, cluster, vpt = shape
        assert kernel in ("stream", "register", "register_late")
        assert (vpt == 0) == (kernel == "stream")
        assert name.endswith(str(vpt)) or kernel == "stream"


def test_cpu_baseline_times_one_thread_and_all_threads():
    """The CPU baseline reports the oracle single-threaded and over every host
    thread, each the fastest of 3 passes, with the CPU model."""
    import oracle
    import synth
    from oracle import build as oracle_build
    oracle_build.build()
    w = synth.TINY
    inp = synth.make_inputs(w, 64)
    cb = bench.cpu_baseline(inp, w.n, w.H, w.eps, False, budget_s=0.3)
    assert cb["kind"] == "oracle" and cb["unit"] == "GB/s" and cb["value"] > 0
    assert cb["cores"] == oracle.host_threads() and cb["cpu_model"]
    st = cb["single_thread"]
    assert st["cores"] == 1 and st["value"] > 0 and "1 thread" in st["sample"]
    assert "fastest of 3" in cb["sample"] and "fastest of 3" in st["sample"]
    assert abs(cb["speedup_all_threads"] - cb["value"] / st["value"]) <= 0.01 * cb["speedup_all_threads"] + 0.01
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()


def test_ar_mode_environment_picks_the_default_path(monkeypatch):
    import bench
    monkeypatch.delenv("AR_MODE", raising=False)
    assert bench.env_mode() == "auto"
    for v, want in (("1", "one_stage"), ("two_stage", "two_stage"), ("0", "auto"), (" AUTO ", "auto")):
        monkeypatch.setenv("AR_MODE", v)
        assert bench.env_mode() == want
    monkeypatch.setenv("AR_MODE", "3")
    with pytest.raises(SystemExit):
        bench.env_mode()

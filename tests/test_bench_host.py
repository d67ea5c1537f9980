"""bench.py's host-side bookkeeping, without a GPU: the stored ncu traffic is reported only for the
kernel sources it was captured from, the committed traffic table is well formed, and a tensor-core
GEMM is measured against the burst or the sustained bf16 peak by the clocks of its own timing loop."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_stored_traffic_follows_the_sources(monkeypatch):
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        entries = json.load(f)
    e = entries[0]
    # the entry's own sources: its bytes
    monkeypatch.setattr(bench, "sources_sha", lambda paths: e["source_sha256"])
    assert bench.stored_traffic(e["kernel"], e["workload"], ["any"]) == e["bytes_per_launch"]
    # changed sources: nothing (the counters no longer describe the kernel)
    monkeypatch.setattr(bench, "sources_sha", lambda paths: "0" * 64)
    assert bench.stored_traffic(e["kernel"], e["workload"], ["any"]) is None
    # another workload or kernel: nothing
    monkeypatch.setattr(bench, "sources_sha", lambda paths: e["source_sha256"])
    assert bench.stored_traffic(e["kernel"], "no_such_workload", ["any"]) is None
    assert bench.stored_traffic("no_such_kernel", e["workload"], ["any"]) is None


def test_traffic_table_is_well_formed():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        entries = json.load(f)
    assert entries
    seen = set()
    for e in entries:
        assert set(e) >= {"kernel", "workload", "bytes_per_launch", "source_sha256", "from"}
        assert e["bytes_per_launch"] > 0 and len(e["source_sha256"]) == 64
        assert os.path.exists(os.path.join(ROOT, e["from"].split(" ")[0].rstrip(",")))
        key = (e["kernel"], e["workload"])
        assert key not in seen  # one capture per kernel and workload
        seen.add(key)


def test_sources_sha_depends_on_content(tmp_path):
    a, b = tmp_path / "a.cu", tmp_path / "b.cu"
    a.write_text("x")
    b.write_text("y")
    assert bench.sources_sha([str(a)]) != bench.sources_sha([str(b)])
    assert bench.sources_sha([str(a)]) == bench.sources_sha([str(a)])


def clock_record(sm, reasons, window="timed region", samples=3):
    return {"sm_mhz": sm, "sm_max_mhz": 2070.0, "reasons": reasons, "samples": samples, "window": window}


def test_power_limited_reads_the_loops_own_samples():
    assert bench.power_limited(clock_record(1695.0, ["sw_power_cap"]))
    assert bench.power_limited(clock_record(1800.0, []))  # well below the maximum with no reason given
    assert not bench.power_limited(clock_record(2070.0, []))
    assert not bench.power_limited(clock_record(1990.0, []))
    assert not bench.power_limited(clock_record(1695.0, ["sw_power_cap"], samples=0))
    assert not bench.power_limited(clock_record(1695.0, ["sw_power_cap"], window="whole GPU phase"))
    assert not bench.power_limited(None)


def test_tensor_roofline_peak_follows_the_timing_loop_clocks():
    import sparse_mixture_experts_moe_gb300 as moe
    from inputgen import workloads
    w = workloads.get("skew_e128")
    peaks = {"hbm_gbs": 6784.5, "bf16_tflops": 1927.9, "bf16_tflops_sustained": 1711.9}
    kern_ms = {"expert_up": 1.99, "expert_down": 2.03}
    flops = 2.0 * w.T * w.k * w.d * w.F
    capped = {n: clock_record(1695.0, ["sw_power_cap"]) for n in kern_ms}
    free = {n: clock_record(2070.0, []) for n in kern_ms}
    for clk, peak in ((capped, 1711.9), (free, 1927.9), (None, 1927.9)):
        r = bench.dominant_roofline(w, kern_ms, 128, moe.PATH_TENSOR_T, 0, peaks, "measured", clk)
        assert r["kernel"] == "ffn_tct_kernel (expert_down)" and r["bound"] == "tensor"
        assert r["peak"] == peak
        achieved = flops / 2.03e-3 / 1e12
        assert abs(r["achieved"] - achieved) < 1e-9 * achieved
        assert abs(r["frac"] - achieved / peak) < 1e-12
        assert abs(r["frac_of_burst"] - achieved / 1927.9) < 1e-12
        assert abs(r["frac_of_sustained"] - achieved / 1711.9) < 1e-12


def test_moved_routings_keep_the_work_on_other_experts():
    import numpy as np
    E = 128
    counts = np.zeros(E, np.int64)
    counts[[17, 90]] = 1                      # one token, top-2
    rs = bench.moved_routings(counts, reps=200)
    assert len(rs) == E // 2 - 1
    prev = {17, 90}
    for o in rs:
        assert o.dtype == np.int32 and o.shape == (E + 1,) and o[0] == 0 and o[-1] == counts.sum()
        c = np.diff(o)
        assert (c >= 0).all() and sorted(c[c > 0].tolist()) == [1, 1]   # the same rows per expert
        now = set(np.nonzero(c)[0].tolist())
        assert not (now & prev)               # neighbouring launches read different experts
        prev = now
    counts = np.zeros(E, np.int64)
    counts[[3, 4, 9]] = [5, 2, 7]             # ragged rows move with their order kept
    o = bench.moved_routings(counts, reps=4)[0]
    assert np.diff(o)[3:6].tolist() == [5, 2, 7]
    assert bench.moved_routings(np.ones(8, np.int64), reps=10) == []   # every expert touched: nothing to move to


def test_streaming_roofline_counts_the_touched_bytes():
    """Quantised and bf16 weight streaming: bytes per launch = the touched experts' codes (or weights)
    and block scales, plus the rows read and written, over the launch time."""
    import sparse_mixture_experts_moe_gb300 as moe
    from inputgen import workloads
    w = workloads.get("decode_t1")                     # T=1, d = d_ff = 8192, E=128, top-2
    peaks = {"hbm_gbs": 6784.5, "bf16_tflops": 1927.9, "bf16_tflops_sustained": 1711.9}
    kern_ms = {"expert_up": 0.0206, "expert_down": 0.0205}
    A, K, N = w.T * w.k, w.d, w.F
    for bits in (4, 8):
        r = bench.dominant_roofline(w, kern_ms, 2, moe.PATH_AUTO, bits, peaks, "measured")
        assert r["bound"] == "hbm" and r["kernel"] == f"ffn_stream_q{bits}_kernel (expert_up)"
        codes = K * N * bits // 8 + (K // 64) * (N // 64) * 8
        want = 2 * codes + A * K * 2 + A * N * 2    # two experts; x rows in, h rows out (bf16)
        assert r["alg_bytes_per_launch"] == want
        assert abs(r["achieved"] - want / 0.0206e-3 / 1e9) < 1e-6 * r["achieved"]
        assert abs(r["frac"] - r["achieved"] / 6784.5) < 1e-12
    r = bench.dominant_roofline(w, kern_ms, 2, moe.PATH_AUTO, 0, peaks, "measured")
    assert r["kernel"] == "ffn_stream_tma_kernel (expert_up)"
    assert r["alg_bytes_per_launch"] == 2 * K * N * 2 + A * K * 2 + A * N * 2

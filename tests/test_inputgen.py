"""Seeded input generator: published SplitMix64 vector, slicing, moments, bf16 rounding, workload table."""
import json
import os

import numpy as np
import torch

import inputgen as ig
from inputgen import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_published_vector():
    with open(os.path.join(GOLDEN, "page_facts.json")) as f:
        v = json.load(f)["splitmix64_vector"]
    # Output n of SplitMix64 started at state s is mix64(s + (n+1)*GAMMA): the counter form used here.
    got = [ig.mix64_int(v["seed"] + (n + 1) * ig.GAMMA) for n in range(5)]
    assert got == [int(o) for o in v["outputs"]]


def test_slices_are_consistent():
    key = ig.stream_key(0, ig.STREAM_W1)
    full = ig.normal_f32(0, 5000, key, 0.125)
    assert np.array_equal(full[1234:1234 + 777], ig.normal_f32(1234, 777, key, 0.125))


def test_moments_and_support():
    v = ig.normal_f32(0, 1 << 20, ig.stream_key(3, ig.STREAM_X), 1.0).astype(np.float64)
    assert abs(v.mean()) < 5e-3
    assert abs(v.var() - 1.0) < 1e-2
    assert np.abs(v).max() < 6.0
    # Irwin-Hall(12) fourth moment is 3 - 1.2/12 = 2.9
    assert abs(np.mean(v ** 4) - 2.9) < 0.05


def test_streams_and_attempts_differ():
    keys = {ig.stream_key(s, st, a) for s in range(3) for st in range(1, 5) for a in range(3)}
    assert len(keys) == 36
    a = ig.normal_f32(0, 64, ig.stream_key(0, ig.STREAM_X, 0), 1.0)
    b = ig.normal_f32(0, 64, ig.stream_key(0, ig.STREAM_X, 1), 1.0)
    assert not np.array_equal(a, b)


def test_bf16_rounding_matches_torch():
    v = ig.normal_f32(0, 100000, ig.stream_key(1, ig.STREAM_X), 1.0)
    # add exact ties (low 16 bits = 0x8000) to exercise round-half-to-even
    ties = (np.arange(1, 200, dtype=np.uint32) << 16 | 0x8000).astype(np.uint32).view(np.float32)
    v = np.concatenate([v, ties, -ties])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ig.f32_to_bf16_bits(v), ref)
    back = ig.bf16_bits_to_f64(ref)
    assert np.array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).double().numpy())


def test_sigma_and_skew_bias():
    assert ig.sigma_for_fan_in(4096) == np.float32(1 / 64)
    b = ig.skew_bias(128, 0.5)
    assert b[0] == 0.0 and np.all(np.diff(b) < 0)
    assert abs(float(b[127]) - 0.5 * -1.2 * np.log(128.0)) < 1e-6


def test_skew_scale_matches_calibration_output():
    with open(os.path.join(GOLDEN, "skew_bias_scale.json")) as f:
        cal = json.load(f)
    assert workloads.SKEW_BIAS_SCALE == cal["c"]
    assert abs(cal["share_at_c"] - 0.38) < 0.01
    w = workloads.get("skew_e128")
    assert (w.T, w.d, w.F, w.E, w.k) == (cal["workload"]["T"], 4096, 8192, 128, 2)


def test_workload_table():
    w = workloads.WORKLOADS
    assert (w["tiny_fp32"].T, w["tiny_fp32"].d, w["tiny_fp32"].E, w["tiny_fp32"].F) == (64, 128, 8, 256)
    assert w["tiny_fp32"].dtype == ig.DTYPE_F32
    assert (w["e16_bf16"].T, w["e16_bf16"].d, w["e16_bf16"].F, w["e16_bf16"].E) == (4096, 1024, 4096, 16)
    assert (w["prefill_e128"].T, w["prefill_e128"].d, w["prefill_e128"].F) == (8192, 4096, 8192)
    assert [w[f"decode_t{t}"].T for t in (1, 8, 64)] == [1, 8, 64]
    assert all(x.k == 2 for x in w.values())

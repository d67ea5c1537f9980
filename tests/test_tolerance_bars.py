"""Which GPU parity cases check a bf16 layer's output against a bar above the stated 2e-2, and by how much.

The GPU parity tests compare a bf16 layer's fp32 output with the oracle at 2e-2 of the output RMS,
except where rounding h to bf16 once (a documented step of the bf16 path) already costs more than
that on the shape; there the bar is 1.1x that rounding's own error plus 2e-3
(``moe_cases.output_tolerance``). This test computes every such case's bar with the oracle, on the
CPU, and pins: the list of cases whose bar is raised and each raised bar at most 3e-2. (The
full-size workloads are too large for the CPU here; their test pins its own list by the same rule.)
"""
import numpy as np
import pytest

import inputgen as ig
import oracle
from inputgen import workloads
from moe_cases import MAX_RAISED_TOL, STATED_TOL_BF16, make_case, output_tolerance
import test_gpu_parity as par
import test_gpu_small_batch as small

BF16 = ig.DTYPE_BF16

# The cases whose bar is raised, by the ids used below, with the raised bar rounded up to 1e-3.
# A change of a kernel cannot move these (they depend on the oracle and the inputs only); a change
# of the cases or of the inputs shows up here.
RAISED = {
    "forward:17": 0.027,      # T=300, d=64, d_ff=64, E=1024, k=8 (pair GEMM)
    "forward:20": 0.027,      # the same shape on the transposed pair GEMM
    "capacity:0": 0.027,      # T=640, d=256, d_ff=512, E=16, capacity factor 1
    "capacity:1": 0.027,      # the same on the pair GEMM
    "capacity:4": 0.030,      # T=640, d=256, d_ff=1024, E=16, capacity factor 0.5 (SIMT)
    "hist:1": 0.021,          # T=1000, d=256, d_ff=128, E=256
    "hist:2": 0.023,          # T=2049, d=64, d_ff=128, E=16, capacity factor 1.1
    "hist:3": 0.024,          # T=777, d=256, d_ff=128, E=8, capacity factor 0.6
    "layer_capacity": 0.024,  # T=512, d=256, d_ff=256, E=16, capacity factor 1.25
}


def _cases():
    """(id, make_case kwargs, oracle kwargs) of every bf16 layer case that uses output_tolerance."""
    out = []
    for i, cfg in enumerate(par.FORWARD_CASES):
        cfg = {k: v for k, v in cfg.items() if k != "path"}
        if cfg["dt"] == BF16:
            out.append((f"forward:{i}", cfg, {}))
    for i, cfg in enumerate(par.CAPACITY_FORWARD_CASES):
        cfg = dict(cfg)
        cfg.pop("path")
        cf = cfg.pop("cf")
        if cfg["dt"] == BF16:
            C = oracle.capacity(cfg["T"], cfg["k"], cfg["E"], cf)
            out.append((f"capacity:{i}", dict(cfg, bias=par._skewed(cfg["E"])), {"cap": C}))
    for i, h in enumerate(par.HIST_CASES):
        T, d, E = h["T"], h["d"], h["E"]
        C = oracle.capacity(T, 2, E, h["cap_factor"]) if h["cap_factor"] > 0 else None
        out.append((f"hist:{i}", dict(T=T, d=d, F=128, E=E, k=2, dt=BF16, bias=par._skewed(E, boost=h.get("boost", 2.5))),
                    {"cap": C}))
    out.append(("layer_capacity", dict(T=512, d=256, F=256, E=16, k=2, dt=BF16, bias=par._skewed(16)),
                {"cap": oracle.capacity(512, 2, 16, 1.25)}))
    ids = ["t1", "t8", "k_eq_e", "e1024", "d136", "e6", "cap", "cap_t2", "bias", "t1_ragged", "t1_k8"]
    assert len(ids) == len(small.CASES)
    for name, cfg in zip(ids, small.CASES):
        cfg = dict(cfg)
        cf = cfg.pop("cf", 0.0)
        bias = cfg.pop("bias", False)
        E = cfg["E"]
        C = oracle.capacity(cfg["T"], cfg["k"], E, cf) if cf > 0 else None
        kw = dict(cfg, dt=BF16, bias=np.linspace(-1.0, 1.0, E, dtype=np.float32) if bias else None)
        for renorm in (False, True):
            out.append((f"small:{name}:{'renorm' if renorm else 'raw'}", kw, {"cap": C, "renormalise": renorm}))
    return out


def test_raised_bars_are_listed_and_bounded():
    raised = {}
    for cid, cfg, okw in _cases():
        c = make_case(host_only=True, **cfg)
        ref = oracle.forward(c.x64, c.wr64, c.w1_host(), c.w2_host(), c.k, c.br64,
                             renormalise=okw.get("renormalise", False), cap=okw.get("cap"))
        bar, was_raised = output_tolerance(c, ref, okw.get("cap"))
        assert bar >= STATED_TOL_BF16
        assert was_raised == (bar > STATED_TOL_BF16)
        if was_raised:
            raised[cid] = bar
    assert set(raised) == set(RAISED), sorted(raised.items())
    for cid, bar in raised.items():
        assert bar <= MAX_RAISED_TOL, (cid, bar)
        assert bar <= RAISED[cid], (cid, bar)


def test_no_benchmark_workload_shape_among_the_small_raised_cases():
    """The small cases with a raised bar are test shapes, none with a benchmark workload's shape; the
    full-size test decides its own raised bars by the same rule and pins them separately."""
    shapes = {(w.d, w.F, w.E, w.k) for w in workloads.WORKLOADS.values()}
    for cid, cfg, _ in _cases():
        if cid in RAISED:
            assert (cfg["d"], cfg["F"], cfg["E"], cfg["k"]) not in shapes, cid
    import test_gpu_fullsize as full
    assert full.FULL_SIZE_RAISED <= set(workloads.WORKLOADS)
    assert full.EMULATION_TOL <= 1e-2


@pytest.mark.parametrize("cid", sorted(RAISED))
def test_raised_bar_is_within_bound(cid):
    assert STATED_TOL_BF16 < RAISED[cid] <= MAX_RAISED_TOL

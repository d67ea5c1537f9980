"""Seeded random layers within the C ABI's limits, each against the fp64 oracle.

160 configurations come from one fixed seed: tokens, model width d, hidden width d_ff (any
multiples of 8), expert count, k, element type, for bf16 a kernel family (every family runs every
valid bf16 shape), and for some an expert capacity (the assignments past it dropped) or renormalised
gates. Each runs moe_forward with its outputs and workspace inside guard bands. Forty more layers
run moe_forward_q on INT4 or INT8 weights against the oracle on its own quantisation of them, and
forty run with an expert capacity that reroutes the assignments past it. Forty routers are checked
with their routing statistics, and twenty layers replayed as CUDA graphs against their direct calls. Routing
indices and counts must equal the oracle's, and the fp32 output must lie within the tolerance rule of
the fixed parity cases: 1e-4 of the RMS for fp32 layers; 2e-2 for bf16, or a bar raised by the one
documented rounding of h. A random shape can raise that bar further than the fixed cases do (d_ff = 8
leaves 8 rounded values per row), so each bf16 output is also held to 1e-2 of the oracle run with h
rounded once. The bf16 output must be the fp32 output rounded once.
"""
import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
import sparse_mixture_experts_moe_gb300 as moe
from moe_cases import (Guarded, guarded_workspace, make_case, oracle_h_rounded, output_tolerance, rel_rms_err,
                        to_f64, torch_dtype)

EMULATION_TOL = 1e-2  # a bf16 output against the oracle with h rounded once to bf16


def check_output(c, out, ref, cap=None):
    """fp32 output of a layer against the oracle (the tolerance rule), and for bf16 layers against the
    oracle with h rounded once."""
    got = to_f64(out)
    bar, _ = output_tolerance(c, ref, cap=cap)
    assert rel_rms_err(got, ref["out"]) < bar, (rel_rms_err(got, ref["out"]), bar)
    if c.dt == BF16:
        assert rel_rms_err(got, oracle_h_rounded(c, ref, cap)) < EMULATION_TOL

BF16, F32 = ig.DTYPE_BF16, ig.DTYPE_F32
PATHS = {moe.PATH_AUTO: "auto", moe.PATH_TENSOR: "tc", moe.PATH_STREAM: "stream", moe.PATH_SIMT: "simt",
         moe.PATH_TENSOR_PAIR: "pair", moe.PATH_TENSOR_T: "tct"}


def draw_cases(n=160, seed=20261203):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        dt = BF16 if rng.random() < 0.8 else F32
        T = int(rng.choice([1, 2, 3, 7, 8, 9, 31, 64, 100, 257, 513, 700]))
        d = 8 * int(rng.integers(1, 49))  # 8 .. 384
        F = 8 * int(rng.integers(1, 49))
        E = int(rng.choice([1, 2, 3, 5, 8, 16, 24, 40, 64, 100, 128, 256]))
        k = int(rng.integers(1, min(E, 8) + 1))
        path = int(rng.choice(list(PATHS))) if dt == BF16 else int(rng.choice([moe.PATH_AUTO, moe.PATH_SIMT]))
        cf = float(rng.choice([0.5, 1.0, 1.25])) if rng.random() < 0.2 else 0.0
        renorm = bool(rng.random() < 0.2)
        cases.append(dict(T=T, d=d, F=F, E=E, k=k, dt=dt, path=path, cf=cf, renorm=renorm))
    return cases


CASES = draw_cases()


@pytest.mark.gpu
def run(c, path, out_dt, cap, renorm):
    """moe_forward with its outputs and workspace inside guard bands; the bands are checked."""
    g = dict(out=Guarded((c.T, c.d), torch_dtype(out_dt)), idx=Guarded((c.T, c.k), torch.int32),
             counts=Guarded(c.E, torch.int32))
    ws = guarded_workspace(c)
    moe.forward(c.x, c.w_r, c.b_r, c.w1, c.w2, c.T, c.d, c.F, c.E, c.k, c.dt, g["out"].t, ws.t,
                topk_idx=g["idx"].t, counts=g["counts"].t, path=path, out_dt=out_dt, capacity=cap,
                renormalise=renorm)
    st, detail = moe.get_device_status(ws.t)
    assert st == moe.MOE_OK, (moe.status_string(st), detail)
    assert all(b.intact() for b in g.values()) and ws.intact()
    return g["out"].t, g["idx"].t.cpu().numpy(), g["counts"].t.cpu().numpy()


def case_id(c):
    tags = ["bf16" if c["dt"] == BF16 else "f32", PATHS[c["path"]]]
    tags += [f"cf{c['cf']}"] if c["cf"] else []
    tags += ["renorm"] if c["renorm"] else []
    return "T{T}_d{d}_F{F}_E{E}_k{k}_".format(**c) + "_".join(tags)


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", CASES, ids=case_id)
def test_random_layer(cfg):
    cfg = dict(cfg)
    path, cf, renorm = cfg.pop("path"), cfg.pop("cf"), cfg.pop("renorm")
    c = make_case(**cfg)
    cap = moe.capacity(c.T, c.k, c.E, cf) if cf else 0
    out, idx, counts = run(c, path, F32, cap, renorm)
    ref = oracle.forward(c.x64, c.wr64, c.w1_host(), c.w2_host(), c.k, c.br64, renormalise=renorm,
                         cap=cap if cap else None)
    assert np.array_equal(idx, ref["idx"])
    routed = oracle.dispatch(ref["idx"], c.E)["counts"]
    assert np.array_equal(counts, np.minimum(routed, cap) if cap else routed)  # kept rows per expert
    check_output(c, out, ref, cap=cap if cap else None)
    if c.dt == BF16:
        out_bf, _, _ = run(c, path, BF16, cap, renorm)
        assert torch.equal(out_bf.view(torch.int16), out.to(torch.bfloat16).view(torch.int16))


def test_draw_covers_the_families():  # host only: the draw exercises every kernel family and both types
    drawn = {(c["dt"], c["path"]) for c in CASES}
    assert {p for dt, p in drawn if dt == BF16} == set(PATHS)
    assert any(dt == F32 for dt, _ in drawn)


def draw_quantised_cases(n=40, seed=20261204):
    """Layers with block-quantised expert weights: d and d_ff multiples of 64, INT4 or INT8."""
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        T = int(rng.choice([1, 2, 3, 8, 9, 33, 64, 130, 300]))
        d = 64 * int(rng.integers(1, 9))  # 64 .. 512
        F = 64 * int(rng.integers(1, 9))
        E = int(rng.choice([1, 2, 5, 8, 16, 40, 64, 128]))
        k = int(rng.integers(1, min(E, 8) + 1))
        cases.append(dict(T=T, d=d, F=F, E=E, k=k, bits=int(rng.choice([4, 8]))))
    return cases


Q_CASES = draw_quantised_cases()


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", Q_CASES, ids=lambda c: "T{T}_d{d}_F{F}_E{E}_k{k}_int{bits}".format(**c))
def test_random_quantised_layer(cfg):
    """moe_forward_q against the oracle run on the oracle's own quantisation of the same weights."""
    from test_gpu_quant import q_case, q_tolerance
    c, q1, q2, w1h, w2h = q_case(**cfg)
    out = Guarded((c.T, c.d), torch.float32)
    idx = Guarded((c.T, c.k), torch.int32)
    ws = guarded_workspace(c)
    moe.forward_q(c.x, c.w_r, c.b_r, q1, q2, c.T, c.d, c.F, c.E, c.k, cfg["bits"], out.t, ws.t, topk_idx=idx.t,
                  out_dt=F32)
    st, detail = moe.get_device_status(ws.t)
    assert st == moe.MOE_OK, (moe.status_string(st), detail)
    assert out.intact() and idx.intact() and ws.intact()
    ref = oracle.forward(c.x64, c.wr64, w1h, w2h, c.k, c.br64)
    assert np.array_equal(idx.t.cpu().numpy(), ref["idx"])
    assert rel_rms_err(to_f64(out.t), ref["out"]) < q_tolerance(c, ref, w1h, w2h)


def draw_reroute_cases(n=40, seed=20261205):
    """Layers whose expert capacity reroutes the assignments past it (MOE_CAPACITY_REROUTE) within each
    token's min(E, 8) best experts; a few experts are made popular so that their queues fill."""
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        dt = BF16 if rng.random() < 0.8 else F32
        E = int(rng.choice([2, 3, 8, 16, 24, 64, 128]))
        k = int(rng.integers(1, min(E, 8) + 1))
        path = int(rng.choice(list(PATHS))) if dt == BF16 else moe.PATH_SIMT
        cases.append(dict(T=int(rng.choice([5, 64, 200, 513])), d=8 * int(rng.integers(1, 33)),
                          F=8 * int(rng.integers(1, 33)), E=E, k=k, dt=dt, path=path,
                          cf=float(rng.choice([0.5, 0.75, 1.0, 1.25])), hot=int(rng.integers(1, 4)),
                          seed=int(rng.integers(0, 1000))))
    return cases


R_CASES = draw_reroute_cases()


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", R_CASES, ids=lambda c: "T{T}_d{d}_F{F}_E{E}_k{k}_cf{cf}_{0}_{1}".format(
    "bf16" if c["dt"] == BF16 else "f32", PATHS[c["path"]], **c))
def test_random_reroute_layer(cfg):
    """moe_forward with MOE_CAPACITY_REROUTE against oracle.forward(cap, reroute): the expert that took
    each slot (-1 when dropped) bit for bit, counts, gates within 1e-5, the output within the bar, and
    exact zeros for tokens whose every assignment was dropped."""
    cfg = dict(cfg)
    path, cf, hot = cfg.pop("path"), cfg.pop("cf"), cfg.pop("hot")
    E = cfg["E"]
    R = min(E, 8)
    bias = np.zeros(E, np.float32)
    bias[:hot] = 2.5
    c = make_case(bias=bias, gap_k=R, **cfg)
    cap = oracle.capacity(c.T, c.k, E, cf)
    out = Guarded((c.T, c.d), torch.float32)
    g = dict(idx=Guarded((c.T, c.k), torch.int32), gate=Guarded((c.T, c.k), torch.float32),
             counts=Guarded(E, torch.int32))
    ws = guarded_workspace(c)
    moe.forward(c.x, c.w_r, c.b_r, c.w1, c.w2, c.T, c.d, c.F, E, c.k, c.dt, out.t, ws.t, topk_idx=g["idx"].t,
                topk_gate=g["gate"].t, counts=g["counts"].t, path=path, out_dt=F32, capacity=cap, reroute=True)
    st, detail = moe.get_device_status(ws.t)
    assert st == moe.MOE_OK, (moe.status_string(st), detail)
    assert out.intact() and ws.intact() and all(b.intact() for b in g.values())
    ref = oracle.forward(c.x64, c.wr64, c.w1_host(), c.w2_host(), c.k, c.br64, cap=cap, reroute=R)
    assert np.array_equal(g["idx"].t.cpu().numpy(), ref["idx"])
    assert np.max(np.abs(g["gate"].t.cpu().numpy() - ref["gate"])) < 1e-5
    assert np.array_equal(g["counts"].t.cpu().numpy(), oracle.dispatch(ref["idx"], E)["counts"])
    check_output(c, out.t, ref)
    gone = ~(ref["idx"] >= 0).any(axis=1)
    assert np.all(to_f64(out.t)[gone] == 0.0)


def draw_router_cases(n=40, seed=20261206):
    """Routers with their statistics: every router kernel (tensor-core tiles, the split-K cluster for
    one deep tile, the CUDA-core kernel for fp32 or other E, the one-launch small batch)."""
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        dt = BF16 if rng.random() < 0.75 else F32
        E = int(rng.choice([1, 3, 8, 16, 24, 64, 100, 128, 200, 256, 512, 1024]))
        cases.append(dict(T=int(rng.choice([1, 2, 5, 8, 9, 64, 128, 129, 700, 2049])),
                          d=8 * int(rng.integers(1, 129)), E=E, k=int(rng.integers(1, min(E, 8) + 1)), dt=dt,
                          renorm=bool(rng.random() < 0.3), skew=bool(rng.random() < 0.5)))
    return cases


ROUTER_CASES = draw_router_cases()


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", ROUTER_CASES, ids=lambda c: "T{T}_d{d}_E{E}_k{k}_{0}{1}".format(
    "bf16" if c["dt"] == BF16 else "f32", "_renorm" if c["renorm"] else "", **c))
def test_random_router_with_stats(cfg):
    """moe_router_topk_stats: indices bit for bit, gates within 1e-5, the statistics against
    oracle.routing_stats, and a second call bit-identical (the cross-CTA sums run in a fixed order)."""
    from test_gpu_parity import check_stats
    cfg = dict(cfg)
    renorm, skew = cfg.pop("renorm"), cfg.pop("skew")
    E = cfg["E"]
    bias = (np.log(np.arange(1, E + 1, dtype=np.float64) ** -1.2) * 0.5).astype(np.float32) if skew else None
    c = make_case(F=8, bias=bias, **cfg)
    ws = guarded_workspace(c)
    idx = Guarded((c.T, c.k), torch.int32)
    gate = Guarded((c.T, c.k), torch.float32)
    stats = Guarded(moe.router_stats_len(E), torch.float32)
    moe.router_topk_stats(c.x, c.w_r, c.b_r, c.T, c.d, E, c.k, c.dt, idx.t, gate.t, stats.t, ws.t,
                          renormalise=renorm)
    st, detail = moe.get_device_status(ws.t)
    assert st == moe.MOE_OK, (moe.status_string(st), detail)
    assert idx.intact() and gate.intact() and stats.intact() and ws.intact()
    logits = oracle.router_logits(c.x64, c.wr64, c.br64)
    ridx = oracle.topk_select(logits, c.k)
    assert np.array_equal(idx.t.cpu().numpy(), ridx)
    want = oracle.gates_renormalised(logits, ridx) if renorm else oracle.gates_of(oracle.softmax(logits), ridx)
    assert np.max(np.abs(gate.t.cpu().numpy() - want)) < 1e-5
    check_stats(stats.t, logits, ridx, c.T, E, c.k)
    again = torch.empty_like(stats.t)
    moe.router_topk_stats(c.x, c.w_r, c.b_r, c.T, c.d, E, c.k, c.dt, idx.t, gate.t, again, ws.t,
                          renormalise=renorm)
    assert torch.equal(again.view(torch.int32), stats.t.view(torch.int32))


def draw_graph_cases(n=20, seed=20261207):
    rng = np.random.default_rng(seed)
    return [dict(T=int(rng.choice([1, 4, 8, 40, 300])), d=8 * int(rng.integers(1, 49)), F=8 * int(rng.integers(1, 49)),
                 E=int(rng.choice([2, 8, 16, 64])), k=2, dt=BF16 if rng.random() < 0.8 else F32,
                 bits=int(rng.choice([0, 0, 4, 8]))) for _ in range(n)]


GRAPH_CASES = draw_graph_cases()


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", GRAPH_CASES, ids=lambda c: "T{T}_d{d}_F{F}_E{E}_{0}_bits{bits}".format(
    "bf16" if c["dt"] == BF16 else "f32", **c))
def test_random_layer_graph_replay(cfg):
    """MoELayer.graph(): a replay gives the direct call's output bit for bit, and the next replay picks
    up new contents of the input buffer."""
    cfg = dict(cfg)
    bits = cfg.pop("bits")
    if bits and (cfg["dt"] != BF16 or cfg["d"] % 64 or cfg["F"] % 64):
        cfg.update(dt=BF16, d=64 * max(1, cfg["d"] // 64), F=64 * max(1, cfg["F"] // 64))  # quantised: bf16, blocks of 64
    c = make_case(**cfg)
    layer = moe.MoELayer(c.w_r, c.w1, c.w2, k=c.k, b_r=c.b_r, weight_bits=bits or None)
    x_buf = c.x.clone()
    out_buf = torch.empty_like(c.x)
    g = layer.graph(x_buf, out_buf)
    for scale in (1.0, -0.5):
        x_new = (c.x.float() * scale).to(c.x.dtype)
        x_buf.copy_(x_new)
        g.launch()
        torch.cuda.synchronize()
        want = layer(x_new)
        torch.cuda.synchronize()
        assert torch.equal(out_buf.view(torch.int16 if out_buf.dtype == torch.bfloat16 else torch.int32),
                           want.view(torch.int16 if want.dtype == torch.bfloat16 else torch.int32))
    assert layer.device_status()[0] == moe.MOE_OK

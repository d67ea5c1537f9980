"""Capacity with rerouting (aicoding/6a320eef §3.2; csdn/6a919c0d §3.2) against the oracle.

moe_dispatch_reroute is fed each token's ranking from the oracle; the expert that takes each slot,
its gate and every dispatch output are compared bit for bit with oracle.reroute_assignments and
oracle.dispatch. The layer with MOE_CAPACITY_REROUTE is compared with oracle.forward(cap, reroute):
routing bit-exact, gates within 1e-5, the output within the usual bar. Inputs are re-drawn until
every token's top-(R+1) logits are 1e-3 apart, so the whole ranking the rerouting walks is decided
far above fp32 rounding.
"""
import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
import sparse_mixture_experts_moe_gb300 as moe
from moe_cases import Guarded, guarded_workspace, make_case, output_tolerance, rel_rms_err, to_f64, torch_dtype

pytestmark = pytest.mark.gpu

BF16, F32 = ig.DTYPE_BF16, ig.DTYPE_F32
DEV = "cuda"


def _hot(E, hot=3, boost=2.5):
    b = np.zeros(E, np.float32)
    b[:hot] = boost  # a few popular experts: their queues fill and tokens are rerouted
    return b


def _ranking(c, R):
    logits = oracle.router_logits(c.x64, c.wr64, c.br64)
    ri = oracle.topk_select(logits, R)
    return ri, oracle.gates_of(oracle.softmax(logits), ri)


DISPATCH_CASES = [
    dict(T=1000, d=64, E=16, k=2, R=8, cf=1.0, dt=BF16),      # 8 chunks, many reroutes
    dict(T=1000, d=64, E=16, k=2, R=3, cf=0.6, dt=BF16),      # one candidate beyond the two chosen: drops too
    dict(T=300, d=40, E=8, k=1, R=8, cf=1.0, dt=F32),         # one slot, the whole ranking
    dict(T=257, d=32, E=64, k=4, R=8, cf=1.25, dt=BF16),      # k = 4, ragged last chunk
    dict(T=50, d=16, E=8, k=8, R=8, cf=0.5, dt=BF16),         # R = k: nothing beyond, the drop rule
    dict(T=37, d=8, E=4, k=2, R=4, cf=0.2, dt=BF16),          # capacity 4 over 74 assignments
    dict(T=4000, d=16, E=128, k=2, R=8, cf=1.0, dt=BF16),     # E = 128, 32 chunks
]


@pytest.mark.parametrize("cfg", DISPATCH_CASES, ids=lambda c: "T{T}_E{E}_k{k}_R{R}_cf{cf}".format(**c))
def test_dispatch_reroute(cfg):
    cfg = dict(cfg)
    R, cf = cfg.pop("R"), cfg.pop("cf")
    c = make_case(F=8, bias=_hot(cfg["E"]), gap_k=R, **cfg)
    ri, rp = _ranking(c, R)
    C = oracle.capacity(c.T, c.k, c.E, cf)
    A = c.A
    g = dict(final_idx=Guarded((c.T, c.k), torch.int32), final_gate=Guarded((c.T, c.k), torch.float32),
             counts=Guarded(c.E, torch.int32), offsets=Guarded(c.E + 1, torch.int32),
             perm_token=Guarded(A, torch.int32), row_of=Guarded((c.T, c.k), torch.int32),
             row_gate=Guarded(A, torch.float32), x_perm=Guarded((A, c.d), torch_dtype(c.dt)))
    ws = guarded_workspace(c)
    moe.dispatch_reroute(c.x, torch.from_numpy(ri.astype(np.int32)).to(DEV),
                         torch.from_numpy(rp.astype(np.float32)).to(DEV), c.T, c.d, c.E, c.k, R, c.dt, C,
                         *(g[n].t for n in ("final_idx", "final_gate", "counts", "offsets", "perm_token", "row_of",
                                            "row_gate", "x_perm")), ws.t)
    st, detail = moe.get_device_status(ws.t)
    assert st == moe.MOE_OK, (st, detail)
    for n, b in g.items():
        assert b.intact(), n
    assert ws.intact()
    fi, fg = oracle.reroute_assignments(ri, rp.astype(np.float32), c.k, c.E, C)
    assert (fi != ri[:, :c.k]).any()  # the case does reroute or drop
    assert np.array_equal(g["final_idx"].t.cpu().numpy(), fi)
    assert np.array_equal(g["final_gate"].t.cpu().numpy(), fg.astype(np.float32))
    ref = oracle.dispatch(fi, c.E, fg.astype(np.float32))
    rows = int(ref["offsets"][-1])
    for n in ("counts", "offsets", "row_of"):
        assert np.array_equal(g[n].t.cpu().numpy(), ref[n]), n
    assert np.array_equal(g["perm_token"].t.cpu().numpy()[:rows], ref["perm_token"][:rows])
    assert np.array_equal(g["row_gate"].t.cpu().numpy()[:rows], ref["row_gate"][:rows].astype(np.float32))
    perm = torch.from_numpy(ref["perm_token"][:rows]).to(DEV)
    assert torch.equal(g["x_perm"].t[:rows], c.x[perm])
    assert np.all(g["counts"].t.cpu().numpy() <= C)


def test_dispatch_reroute_flags_out_of_range_index():
    c = make_case(T=200, d=16, F=8, E=16, k=2, dt=BF16, gap_k=4)
    ri, rp = _ranking(c, 4)
    ri[77, 1] = 16  # out of range
    out = {n: torch.empty(s, dtype=t, device=DEV) for n, s, t in [
        ("fi", (200, 2), torch.int32), ("fg", (200, 2), torch.float32), ("counts", 16, torch.int32),
        ("offsets", 17, torch.int32), ("perm", 400, torch.int32), ("row_of", (200, 2), torch.int32),
        ("row_gate", 400, torch.float32), ("x_perm", (400, 16), torch.bfloat16)]}
    ws = guarded_workspace(c)
    moe.dispatch_reroute(c.x, torch.from_numpy(ri.astype(np.int32)).to(DEV),
                         torch.from_numpy(rp.astype(np.float32)).to(DEV), 200, 16, 16, 2, 4, BF16, 1000,
                         *out.values(), ws.t)
    st, detail = moe.get_device_status(ws.t)
    assert st == moe.MOE_ERR_DEVICE_CHECK and detail == 77 * 2 + 1
    assert out["fi"][77, 1].item() == -1 and out["row_of"][77, 1].item() == -1
    assert out["counts"].sum().item() == 399


FORWARD_CASES = [
    dict(T=640, d=256, F=512, E=16, k=2, dt=BF16, path=moe.PATH_AUTO, cf=1.0),
    dict(T=640, d=256, F=512, E=16, k=2, dt=BF16, path=moe.PATH_TENSOR_T, cf=0.75),
    dict(T=200, d=128, F=256, E=8, k=2, dt=F32, path=moe.PATH_AUTO, cf=1.0),
    dict(T=8, d=512, F=512, E=16, k=2, dt=BF16, path=moe.PATH_AUTO, cf=1.0),     # a decode batch: streaming
    dict(T=300, d=64, F=64, E=1024, k=8, dt=BF16, path=moe.PATH_AUTO, cf=1.0),  # R = k = 8: drops only
]


@pytest.mark.parametrize("cfg", FORWARD_CASES, ids=["auto", "tensor_t", "simt_f32", "decode", "e1024_k8"])
def test_forward_reroute(cfg):
    cfg = dict(cfg)
    path, cf = cfg.pop("path"), cfg.pop("cf")
    E = cfg["E"]
    R = min(E, 8)
    c = make_case(bias=_hot(E), gap_k=R, **cfg)
    C = oracle.capacity(c.T, c.k, E, cf)
    out = Guarded((c.T, c.d), torch.float32)
    idx = torch.empty((c.T, c.k), dtype=torch.int32, device=DEV)
    gate = torch.empty((c.T, c.k), dtype=torch.float32, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    ws = guarded_workspace(c)
    moe.forward(c.x, c.w_r, c.b_r, c.w1, c.w2, c.T, c.d, c.F, E, c.k, c.dt, out.t, ws.t, topk_idx=idx,
                topk_gate=gate, counts=counts, path=path, out_dt=F32, capacity=C, reroute=True)
    st, detail = moe.get_device_status(ws.t)
    assert st == moe.MOE_OK, (st, detail)
    assert out.intact() and ws.intact()
    ref = oracle.forward(c.x64, c.wr64, c.w1_host(), c.w2_host(), c.k, c.br64, cap=C, reroute=R)
    assert (ref["idx"] != oracle.topk_select(ref["logits"], c.k)).any()  # something was rerouted or dropped
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert np.max(np.abs(gate.cpu().numpy() - ref["gate"])) < 1e-5
    assert np.array_equal(counts.cpu().numpy(), oracle.dispatch(ref["idx"], E)["counts"])
    assert rel_rms_err(to_f64(out.t), ref["out"]) < output_tolerance(c, ref)[0]
    gone = ~(ref["idx"] >= 0).any(axis=1)
    assert np.all(to_f64(out.t)[gone] == 0.0)


@pytest.mark.parametrize("bits", [4, 8])
def test_forward_q_reroute(bits):
    c = make_case(T=64, d=512, F=512, E=16, k=2, dt=BF16, bias=_hot(16), gap_k=8)
    C = oracle.capacity(64, 2, 16, 1.0)
    q1, q2 = moe.quantize(c.w1, bits), moe.quantize(c.w2, bits)
    out = torch.empty((64, 512), dtype=torch.float32, device=DEV)
    idx = torch.empty((64, 2), dtype=torch.int32, device=DEV)
    ws = guarded_workspace(c)
    moe.forward_q(c.x, c.w_r, c.b_r, q1, q2, 64, 512, 512, 16, 2, bits, out, ws.t, topk_idx=idx, out_dt=F32,
                  capacity=C, reroute=True)
    assert moe.get_device_status(ws.t)[0] == moe.MOE_OK
    logits = oracle.router_logits(c.x64, c.wr64, c.br64)
    ri = oracle.topk_select(logits, 8)
    fi, _ = oracle.reroute_assignments(ri, oracle.gates_of(oracle.softmax(logits), ri), 2, 16, C)
    assert (fi != ri[:, :2]).any()
    assert np.array_equal(idx.cpu().numpy(), fi)

"""CUDA-graph replay of the layer (moe_forward_graph_create / moe_graph_launch) against the direct
call and the fp64 oracle: bit-identical outputs, new input contents picked up on every launch."""
import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
import sparse_mixture_experts_moe_gb300 as moe
from moe_cases import make_case, rel_rms_err, to_f64, workspace_for

pytestmark = pytest.mark.gpu

DEV = "cuda"
BF16, F32 = ig.DTYPE_BF16, ig.DTYPE_F32


@pytest.mark.parametrize("cfg", [dict(T=640, d=256, F=512, E=16, k=2, dt=BF16, path=moe.PATH_AUTO),
                                 dict(T=8, d=1024, F=1024, E=32, k=2, dt=BF16, path=moe.PATH_AUTO),
                                 dict(T=1, d=2048, F=1024, E=64, k=2, dt=BF16, path=moe.PATH_AUTO),
                                 dict(T=64, d=128, F=256, E=8, k=2, dt=F32, path=moe.PATH_AUTO),
                                 dict(T=300, d=256, F=256, E=16, k=2, dt=BF16, path=moe.PATH_TENSOR_PAIR)],
                         ids=["tensor", "stream", "stream_t1", "simt_f32", "pair"])
def test_graph_matches_direct_call(cfg):
    cfg = dict(cfg)
    path = cfg.pop("path")
    c = make_case(**cfg)
    ws = workspace_for(c)
    out_direct = torch.empty((c.T, c.d), dtype=torch.float32, device=DEV)
    moe.forward(c.x, c.w_r, c.b_r, c.w1, c.w2, c.T, c.d, c.F, c.E, c.k, c.dt, out_direct, ws, path=path,
                out_dt=F32)
    out = torch.full((c.T, c.d), float("nan"), dtype=torch.float32, device=DEV)
    idx = torch.empty((c.T, c.k), dtype=torch.int32, device=DEV)
    g = moe.ForwardGraph(c.x, c.w_r, c.b_r, c.w1, c.w2, c.T, c.d, c.F, c.E, c.k, c.dt, out, ws, topk_idx=idx,
                         path=path, out_dt=F32)
    torch.cuda.synchronize()
    assert torch.isnan(out).all()  # creating the graph runs nothing
    for _ in range(3):
        g.launch()
    assert moe.get_device_status(ws)[0] == moe.MOE_OK
    assert torch.equal(out.view(torch.int32), out_direct.view(torch.int32))
    ref = oracle.forward(c.x64, c.wr64, c.w1_host(), c.w2_host(), c.k, c.br64)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    # new contents of the same input buffer (the tokens in reverse order): the next replay routes
    # and computes them
    c.x.copy_(torch.flip(c.x, dims=[0]))
    g.launch()
    ref2 = oracle.forward(c.x64[::-1].copy(), c.wr64, c.w1_host(), c.w2_host(), c.k, c.br64)
    assert np.array_equal(idx.cpu().numpy(), ref2["idx"])
    tol = 1e-4 if c.dt == F32 else 2e-2
    assert rel_rms_err(to_f64(out), ref2["out"]) < tol
    g.close()


def test_layer_graph_with_capacity_and_stats():
    c = make_case(T=512, d=256, F=256, E=16, k=2, dt=BF16)
    layer = moe.MoELayer(c.w_r, c.w1, c.w2, k=2, b_r=c.b_r, capacity_factor=1.0)
    out = torch.empty((c.T, c.d), dtype=torch.float32, device=DEV)
    stats = torch.empty(moe.router_stats_len(16), dtype=torch.float32, device=DEV)
    g = layer.graph(c.x, out, router_stats=stats)
    g.launch()
    want = torch.empty_like(out)
    want_stats = torch.empty_like(stats)
    layer(c.x, out=want, router_stats=want_stats)
    assert layer.device_status()[0] == moe.MOE_OK
    assert torch.equal(out.view(torch.int32), want.view(torch.int32))
    assert torch.equal(stats.view(torch.int32), want_stats.view(torch.int32))


def test_graph_zero_tokens_and_bad_args():
    c = make_case(T=0, d=64, F=64, E=4, k=2, dt=BF16)
    ws = torch.empty(moe.workspace_bytes(0, 64, 64, 4, 2, BF16), dtype=torch.uint8, device=DEV)
    moe.workspace_init(ws)
    out = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    g = moe.ForwardGraph(c.x, c.w_r, None, c.w1, c.w2, 0, 64, 64, 4, 2, BF16, out, ws)
    g.launch()
    torch.cuda.synchronize()
    with pytest.raises(moe.MoeError):
        moe.ForwardGraph(c.x, c.w_r, None, c.w1, c.w2, 0, 64, 64, 4, 9, BF16, out, ws)  # k > E: the library refuses


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("T", [1, 8])
def test_graph_quantised_forward(T, bits):
    """moe_forward_q recorded into a graph (moe_graph_capture_*, as bench.py replays it) gives the
    direct call's output bit for bit, and the next replay picks up new input contents."""
    c = make_case(T=T, d=1024, F=1024, E=32, k=2, dt=BF16)
    q1, q2 = moe.quantize(c.w1, bits), moe.quantize(c.w2, bits)
    ws = workspace_for(c)
    want = torch.empty((c.T, c.d), dtype=torch.float32, device=DEV)
    moe.forward_q(c.x, c.w_r, c.b_r, q1, q2, c.T, c.d, c.F, c.E, c.k, bits, want, ws, out_dt=F32)
    out = torch.full((c.T, c.d), float("nan"), dtype=torch.float32, device=DEV)
    with moe.GraphCapture(keep=(c.x, c.w_r, c.b_r, q1, q2, out, ws)) as cap:
        moe.forward_q(c.x, c.w_r, c.b_r, q1, q2, c.T, c.d, c.F, c.E, c.k, bits, out, ws, out_dt=F32,
                      stream=cap.stream)
    torch.cuda.synchronize()
    assert torch.isnan(out).all()  # recording runs nothing
    g = cap.graph
    for _ in range(2):
        g.launch()
    torch.cuda.synchronize()
    assert moe.get_device_status(ws)[0] == moe.MOE_OK
    assert torch.equal(out.view(torch.int32), want.view(torch.int32))
    c.x.copy_(torch.flip(c.x, dims=[0]))
    want2 = torch.empty_like(want)
    moe.forward_q(c.x, c.w_r, c.b_r, q1, q2, c.T, c.d, c.F, c.E, c.k, bits, want2, ws, out_dt=F32)
    g.launch()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int32), want2.view(torch.int32))
    g.close()

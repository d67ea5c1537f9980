"""GPU path vs the fp64 oracle, through the C ABI, at sizes the oracle finishes in seconds.

Bars (stated by the layer's specification): routing indices, counts, offsets and the
permutation bit-exact; outputs within max relative-to-RMS error 1e-4 (fp32) and
2e-2 (bf16). Shapes span several 128x256 tensor-core tiles with ragged row and
column tails, several dispatch chunks, and the degenerate cases of the method.
Each step is also checked on its own, fed by inputs that do not come from the
GPU path (oracle routing, or generator tensors for h and y_perm).
"""
import numpy as np
import pytest
import torch

import inputgen as ig
from inputgen import workloads
import oracle
import sparse_mixture_experts_moe_gb300 as moe
from moe_cases import (Guarded, device_tensor, guarded_workspace, make_case, output_tolerance, rel_rms_err,
                        to_f64, torch_dtype, workspace_for)

pytestmark = pytest.mark.gpu

BF16, F32 = ig.DTYPE_BF16, ig.DTYPE_F32
TOL = {F32: 1e-4, BF16: 2e-2}
DEV = "cuda"


def assert_rounded_once(got, ref, dt):
    """got is ref (fp64) rounded once to dt after fp32 arithmetic.

    bf16 keeps 8 significant bits, so one round-to-nearest moves a value by at most
    2^-8 of its magnitude (a rounding that flips near a midpoint adds a little); fp32
    accumulation and erff add far less than 1e-4 of the tensor's RMS.
    """
    rms = float(np.sqrt(np.mean(ref * ref)))
    rel = 2.0 ** -8 if dt == BF16 else 2.0 ** -22
    excess = np.abs(got - ref) - (rel * np.abs(ref) + 1e-4 * rms)
    assert np.all(excess <= 0), f"max excess {excess.max():.3e} (rms {rms:.3e})"


def run_router(c):
    idx = torch.empty((c.T, c.k), dtype=torch.int32, device=DEV)
    gate = torch.empty((c.T, c.k), dtype=torch.float32, device=DEV)
    moe.router_topk(c.x, c.w_r, c.b_r, c.T, c.d, c.E, c.k, c.dt, idx, gate)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), gate.cpu().numpy()


def oracle_routing(c):
    logits = oracle.router_logits(c.x64, c.wr64, c.br64)
    p = oracle.softmax(logits)
    idx = oracle.topk_select(logits, c.k)
    return idx, oracle.gates_of(p, idx)


ROUTER_CASES = [
    dict(T=64, d=128, F=256, E=8, k=2, dt=F32),            # the tiny fp32 layer
    dict(T=300, d=320, F=64, E=16, k=2, dt=BF16),
    dict(T=257, d=256, F=64, E=128, k=2, dt=BF16),
    dict(T=33, d=64, F=64, E=1024, k=8, dt=BF16),          # largest E and k
    dict(T=50, d=96, F=64, E=2, k=2, dt=F32),              # E = k
    dict(T=70, d=64, F=64, E=5, k=1, dt=BF16),
    dict(T=1, d=8, F=8, E=3, k=2, dt=F32),
    dict(T=1, d=2048, F=64, E=64, k=2, dt=BF16),           # one token, deep d: split over a cluster
    dict(T=128, d=1024, F=64, E=128, k=4, dt=BF16),        # the split path's largest batch
    dict(T=129, d=1024, F=64, E=128, k=2, dt=BF16),        # one token more: two plain CTAs
    dict(T=40, d=4096, F=64, E=256, k=2, dt=BF16),         # E = 256 keeps the plain kernel
    dict(T=1000, d=1024, F=64, E=16, k=2, dt=BF16),        # eight split clusters, ragged last tile
    dict(T=300, d=2048, F=64, E=128, k=3, dt=BF16),
]


@pytest.mark.parametrize("cfg", ROUTER_CASES, ids=lambda c: "T{T}_d{d}_E{E}_k{k}_{dt}".format(**c))
def test_router_topk(cfg):
    c = make_case(**cfg)
    idx, gate = run_router(c)
    ridx, rgate = oracle_routing(c)
    assert np.array_equal(idx, ridx)
    assert np.max(np.abs(gate - rgate)) < 1e-5
    assert np.all(gate.sum(axis=1) <= 1.0 + 1e-6)


@pytest.mark.parametrize("T,d", [(400, 256), (64, 4096)], ids=["plain", "split"])
def test_router_skew_bias(T, d):
    c = make_case(T=T, d=d, F=64, E=128, k=2, dt=BF16, bias_scale=workloads.SKEW_BIAS_SCALE)
    idx, gate = run_router(c)
    ridx, rgate = oracle_routing(c)
    assert np.array_equal(idx, ridx)
    assert np.max(np.abs(gate - rgate)) < 1e-5


DISPATCH_CASES = [
    dict(T=1000, d=64, E=128, k=2, dt=BF16),   # 8 chunks, ragged last chunk
    dict(T=300, d=40, E=1024, k=8, dt=F32),    # 10 chunks, E = 1024
    dict(T=3, d=8, E=4, k=2, dt=BF16),
    dict(T=513, d=128, E=16, k=2, dt=F32),
]


def run_dispatch(c, idx, gate, capacity=0):
    """moe_dispatch with every output (and the workspace) inside guard bands; the bands are checked."""
    A, E = c.A, c.E
    g = dict(counts=Guarded(E, torch.int32), offsets=Guarded(E + 1, torch.int32),
             perm_token=Guarded(A, torch.int32), row_of=Guarded((c.T, c.k), torch.int32),
             row_gate=Guarded(A, torch.float32), x_perm=Guarded((A, c.d), torch_dtype(c.dt)))
    out = {name: b.t for name, b in g.items()}
    ws = guarded_workspace(c)
    ti = torch.from_numpy(idx.astype(np.int32)).to(DEV)
    tg = torch.from_numpy(gate.astype(np.float32)).to(DEV)
    moe.dispatch(c.x, ti, tg, c.T, c.d, E, c.k, c.dt, out["counts"], out["offsets"], out["perm_token"],
                 out["row_of"], out["row_gate"], out["x_perm"], ws.t, capacity=capacity)
    st, detail = moe.get_device_status(ws.t)
    for name, b in g.items():
        assert b.intact(), f"dispatch wrote outside {name}"
    assert ws.intact(), "dispatch wrote outside its workspace"
    return out, st, detail


@pytest.mark.parametrize("cfg", DISPATCH_CASES, ids=lambda c: "T{T}_E{E}_k{k}".format(**c))
def test_dispatch(cfg):
    c = make_case(F=64, **cfg)
    ridx, rgate = oracle_routing(c)
    out, st, _ = run_dispatch(c, ridx, rgate)
    assert st == moe.MOE_OK
    ref = oracle.dispatch(ridx, c.E, rgate.astype(np.float32))
    assert np.array_equal(out["counts"].cpu().numpy(), ref["counts"])
    assert np.array_equal(out["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(out["perm_token"].cpu().numpy(), ref["perm_token"])
    assert np.array_equal(out["row_of"].cpu().numpy(), ref["row_of"])
    assert np.array_equal(out["row_gate"].cpu().numpy(), ref["row_gate"].astype(np.float32))
    assert np.array_equal(to_f64(out["x_perm"]), c.x64[ref["perm_token"]])


def _skewed(E, hot=3, boost=2.5):
    b = np.zeros(E, np.float32)
    b[:hot] = boost  # a few popular experts, so a capacity factor of 1 drops assignments
    return b


@pytest.mark.parametrize("cfg,cf", [(dict(T=1000, d=64, E=16, k=2, dt=BF16), 1.0),
                                    (dict(T=1000, d=64, E=16, k=2, dt=BF16), 1.25),
                                    (dict(T=300, d=40, E=1024, k=8, dt=F32), 1.0),
                                    (dict(T=513, d=128, E=16, k=2, dt=F32), 100.0),   # nothing dropped
                                    (dict(T=37, d=8, E=4, k=2, dt=BF16), 0.05)],      # capacity 1
                         ids=["e16_cf1", "e16_cf1.25", "e1024_cf1", "no_drop", "cap1"])
def test_dispatch_capacity(cfg, cf):
    c = make_case(F=64, bias=_skewed(cfg["E"]), **cfg)
    ridx, rgate = oracle_routing(c)
    C = oracle.capacity(c.T, c.k, c.E, cf)
    assert moe.capacity(c.T, c.k, c.E, cf) == C
    out, st, _ = run_dispatch(c, ridx, rgate, capacity=C)
    assert st == moe.MOE_OK
    ref = oracle.dispatch(ridx, c.E, rgate.astype(np.float32), cap=C)
    if cf <= 1.0:
        assert ref["offsets"][-1] < c.A  # the case does drop assignments
    rows = int(ref["offsets"][-1])
    assert np.array_equal(out["counts"].cpu().numpy(), ref["counts"])
    assert np.array_equal(out["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(out["row_of"].cpu().numpy(), ref["row_of"])
    assert np.array_equal(out["perm_token"].cpu().numpy()[:rows], ref["perm_token"][:rows])
    assert np.array_equal(out["row_gate"].cpu().numpy()[:rows], ref["row_gate"][:rows].astype(np.float32))
    assert np.array_equal(to_f64(out["x_perm"])[:rows], c.x64[ref["perm_token"][:rows]])


def test_dispatch_rejects_negative_capacity():
    c = make_case(T=16, d=64, F=64, E=4, k=2, dt=BF16)
    ridx, rgate = oracle_routing(c)
    with pytest.raises(moe.MoeError) as e:
        run_dispatch(c, ridx, rgate, capacity=-1)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG


def test_dispatch_flags_out_of_range_index():
    c = make_case(T=200, d=64, F=64, E=16, k=2, dt=BF16)
    ridx, rgate = oracle_routing(c)
    bad = ridx.copy()
    bad[77, 1] = 16  # out of range
    out, st, detail = run_dispatch(c, bad, rgate)
    assert st == moe.MOE_ERR_DEVICE_CHECK and detail == 77 * 2 + 1
    row_of = out["row_of"].cpu().numpy()
    assert row_of[77, 1] == -1
    assert out["counts"].cpu().numpy().sum() == c.A - 1
    # the context is still usable and the status was cleared
    out2, st2, _ = run_dispatch(c, ridx, rgate)
    assert st2 == moe.MOE_OK


# ----------------------------------------------------------------------------- expert FFN halves

FFN_CASES = [
    # (T, d, F, E, k, dt, path)
    (600, 320, 704, 6, 2, BF16, moe.PATH_TENSOR),   # 2 row tiles per expert + tails, N tail 704 = 2.75 x 256
    (700, 256, 512, 3, 2, BF16, moe.PATH_TENSOR),   # ~467 rows per expert: 4 row tiles
    (96, 64, 128, 8, 2, BF16, moe.PATH_TENSOR),     # K = 64: one k-block, N < 256
    (600, 320, 704, 6, 2, BF16, moe.PATH_SIMT),
    (12, 512, 384, 16, 2, BF16, moe.PATH_STREAM),
    (64, 1024, 512, 8, 2, BF16, moe.PATH_STREAM),   # up to 8+ rows per expert: several passes
    (64, 128, 256, 8, 2, F32, moe.PATH_SIMT),
    (1100, 320, 704, 3, 2, BF16, moe.PATH_TENSOR_PAIR),  # ~733 rows/expert: 3 pair tiles + tails, N tail
    (600, 320, 704, 6, 2, BF16, moe.PATH_TENSOR_PAIR),   # ~200 rows/expert: one partly empty pair tile each
    (96, 64, 128, 8, 2, BF16, moe.PATH_TENSOR_PAIR),     # K = 64, N < 256, most rows of the pair idle
    (1100, 320, 704, 3, 2, BF16, moe.PATH_TENSOR_T),     # ~733 rows/expert: 3 row tiles, feature tail 704
    (600, 320, 704, 6, 2, BF16, moe.PATH_TENSOR_T),      # ~200 rows/expert: one tile of N = rows rounded to 16
    (96, 64, 128, 8, 2, BF16, moe.PATH_TENSOR_T),        # K = 64, 24 rows per expert, 128 features
    (37, 128, 264, 5, 2, BF16, moe.PATH_TENSOR_T),       # odd row counts (N = 16 tiles), F = 264 not a multiple of 64
    (2048, 256, 4096, 8, 2, BF16, moe.PATH_TENSOR_T),    # enough items for 256-row tiles (up), 128-row (down)
]


def _ffn_inputs(c):
    ridx, rgate = oracle_routing(c)
    dp = oracle.dispatch(ridx, c.E, rgate.astype(np.float32))
    x_perm = c.x[torch.from_numpy(dp["perm_token"]).to(DEV)].contiguous()
    offsets = torch.from_numpy(dp["offsets"].astype(np.int32)).to(DEV)
    row_gate = torch.from_numpy(dp["row_gate"].astype(np.float32)).to(DEV)
    return dp, x_perm, offsets, row_gate


@pytest.mark.parametrize("cfg", FFN_CASES, ids=lambda c: "T{}_d{}_F{}_E{}_dt{}_path{}".format(*c[:4], c[5], c[6]))
def test_expert_up(cfg):
    T, d, F, E, k, dt, path = cfg
    c = make_case(T=T, d=d, F=F, E=E, k=k, dt=dt)
    dp, x_perm, offsets, _ = _ffn_inputs(c)
    hg = Guarded((c.A, F), torch_dtype(dt), fill=0)
    h = hg.t
    ws = guarded_workspace(c)
    moe.expert_up(x_perm, c.w1, offsets, T, d, F, E, k, dt, h, ws.t, path=path)
    st, _ = moe.get_device_status(ws.t)
    assert st == moe.MOE_OK
    assert hg.intact() and ws.intact(), "the up-projection wrote outside h or its workspace"
    ref = oracle.expert_rows_up(c.x64[dp["perm_token"]], dp["offsets"], c.w1_host())
    assert_rounded_once(to_f64(h), ref, dt)


@pytest.mark.parametrize("cfg", FFN_CASES, ids=lambda c: "T{}_d{}_F{}_E{}_dt{}_path{}".format(*c[:4], c[5], c[6]))
def test_expert_down(cfg):
    T, d, F, E, k, dt, path = cfg
    c = make_case(T=T, d=d, F=F, E=E, k=k, dt=dt)
    dp, _, offsets, row_gate = _ffn_inputs(c)
    # h from the generator (stream 5), not from the GPU's up-projection
    h = device_tensor((c.A, F), 0, 5, 1.0, dt, DEV)
    yg = Guarded((c.A, d), torch.float32, fill=0)
    y = yg.t
    ws = guarded_workspace(c)
    moe.expert_down(h, c.w2, offsets, row_gate, T, d, F, E, k, dt, y, ws.t, path=path)
    st, _ = moe.get_device_status(ws.t)
    assert st == moe.MOE_OK
    assert yg.intact() and ws.intact(), "the down-projection wrote outside y_perm or its workspace"
    ref = oracle.expert_rows_down(to_f64(h), dp["offsets"], dp["row_gate"], c.w2_host())
    # y_perm is fp32 (no rounding to bf16): only fp32 accumulation error remains
    assert rel_rms_err(to_f64(y), ref) < 1e-4


@pytest.mark.parametrize("T,F", [(1500, 512), (700, 256)])
def test_expert_gemms_mixed_routing(T, F):
    """The pair GEMM on a skewed batch (experts with more than 256 rows and experts with a few rows in
    the same launch): items come from the workspace counter through the item ring, heavy and light
    experts interleaved; h and y_perm against the oracle as in test_expert_up / test_expert_down."""
    d, E, k = 256, 16, 2
    c = make_case(T=T, d=d, F=F, E=E, k=k, dt=BF16, bias=_skewed(E))
    dp, x_perm, offsets, row_gate = _ffn_inputs(c)
    cnt = np.diff(dp["offsets"])
    assert (cnt > 256).any() and ((cnt > 0) & (cnt <= 256)).any()  # both classes present
    hg = Guarded((c.A, F), torch.bfloat16, fill=0)
    ws = guarded_workspace(c)
    for _ in range(2):  # the second launch also checks that the counter was set back to zero
        moe.expert_up(x_perm, c.w1, offsets, T, d, F, E, k, BF16, hg.t, ws.t, path=moe.PATH_TENSOR_T)
        assert moe.get_device_status(ws.t)[0] == moe.MOE_OK
        assert hg.intact() and ws.intact()
        ref = oracle.expert_rows_up(c.x64[dp["perm_token"]], dp["offsets"], c.w1_host())
        assert_rounded_once(to_f64(hg.t), ref, BF16)
    yg = Guarded((c.A, d), torch.float32, fill=0)
    moe.expert_down(hg.t, c.w2, offsets, row_gate, T, d, F, E, k, BF16, yg.t, ws.t, path=moe.PATH_TENSOR_T)
    assert moe.get_device_status(ws.t)[0] == moe.MOE_OK
    assert yg.intact() and ws.intact()
    yref = oracle.expert_rows_down(to_f64(hg.t), dp["offsets"], dp["row_gate"], c.w2_host())
    assert rel_rms_err(to_f64(yg.t), yref) < 1e-4
    hdr = ws.t[:32].view(torch.int32).cpu().numpy()
    assert hdr[4] == 0 and hdr[5] == 0  # item counter and finished pairs back at zero


@pytest.mark.parametrize("d,F", [(256, 512), (192, 320)])
def test_expert_gemms_given_row_counts(d, F):
    """The pair GEMM on given per-expert row counts: heavy experts with full 256-row tiles and ragged
    last tiles (600 = 256 + 256 + 88, 777 = 3 x 256 + 9, 300 = 256 + 44), an exact multiple (1024), a
    light expert and an empty one, in one launch (both classes: the counter and the item ring).
    x_perm is the case's token rows in order (k = 1); h and y_perm against the oracle."""
    counts = np.array([600, 1024, 300, 40, 0, 777])
    E, A = len(counts), int(counts.sum())
    c = make_case(T=A, d=d, F=F, E=E, k=1, dt=BF16)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    offsets = torch.from_numpy(offs).to(DEV)
    gate = np.random.default_rng(7).uniform(0.0, 1.0, A).astype(np.float32)
    row_gate = torch.from_numpy(gate).to(DEV)
    ws = guarded_workspace(c)
    hg = Guarded((A, F), torch.bfloat16, fill=0)
    moe.expert_up(c.x, c.w1, offsets, A, d, F, E, 1, BF16, hg.t, ws.t, path=moe.PATH_TENSOR_T)
    assert moe.get_device_status(ws.t)[0] == moe.MOE_OK
    assert hg.intact() and ws.intact()
    assert_rounded_once(to_f64(hg.t), oracle.expert_rows_up(c.x64, offs, c.w1_host()), BF16)
    yg = Guarded((A, d), torch.float32, fill=0)
    moe.expert_down(hg.t, c.w2, offsets, row_gate, A, d, F, E, 1, BF16, yg.t, ws.t, path=moe.PATH_TENSOR_T)
    assert moe.get_device_status(ws.t)[0] == moe.MOE_OK
    assert yg.intact() and ws.intact()
    yref = oracle.expert_rows_down(to_f64(hg.t), offs, gate, c.w2_host())
    assert rel_rms_err(to_f64(yg.t), yref) < 1e-4


@pytest.mark.parametrize("dt", [BF16, F32])
def test_combine(dt):
    T, d, k = 333, 136, 3
    c = make_case(T=T, d=d, F=64, E=7, k=k, dt=dt)
    ridx, rgate = oracle_routing(c)
    dp = oracle.dispatch(ridx, c.E, rgate)
    y = device_tensor((T * k, d), 0, 6, 1.0, F32, DEV)   # y_perm is fp32 for every dt
    og = Guarded((T, d), torch_dtype(dt))
    out = og.t
    moe.combine(y, torch.from_numpy(dp["row_of"].astype(np.int32)).to(DEV), T, d, k, dt, out)
    assert og.intact(), "combine wrote outside its output"
    y64 = to_f64(y)
    ref = oracle.combine(y64, dp["row_of"])
    got = to_f64(out)
    # fp32 sum of k terms (each addition within 2^-24 of the running sum, bounded by sum |y_j|),
    # then one rounding to dt (bf16: at most 2^-8 |value|; fp32: 2^-24 |value|)
    abs_sum = sum(np.abs(y64[dp["row_of"][:, j]]) for j in range(k))
    rel = 2.0 ** -8 if dt == BF16 else 2.0 ** -23
    assert np.all(np.abs(got - ref) <= rel * np.abs(ref) + k * 2.0 ** -23 * abs_sum)


# ----------------------------------------------------------------------------- whole layer

FORWARD_CASES = [
    dict(T=64, d=128, F=256, E=8, k=2, dt=F32, path=moe.PATH_AUTO),          # the tiny fp32 layer
    dict(T=640, d=256, F=512, E=16, k=2, dt=BF16, path=moe.PATH_AUTO),       # tensor-core path
    dict(T=640, d=256, F=512, E=16, k=2, dt=BF16, path=moe.PATH_SIMT),
    dict(T=600, d=320, F=704, E=6, k=2, dt=BF16, path=moe.PATH_TENSOR),
    dict(T=384, d=512, F=1024, E=128, k=2, dt=BF16, path=moe.PATH_TENSOR),   # many nearly empty experts
    dict(T=8, d=1024, F=1024, E=128, k=2, dt=BF16, path=moe.PATH_AUTO),      # decode-shaped: streaming path
    dict(T=64, d=512, F=512, E=32, k=2, dt=BF16, path=moe.PATH_STREAM),
    dict(T=8, d=512, F=512, E=32, k=2, dt=BF16, path=moe.PATH_TENSOR),       # decode shape on the tensor path
    dict(T=1, d=256, F=256, E=16, k=2, dt=BF16, path=moe.PATH_AUTO),         # one token
    dict(T=77, d=64, F=96, E=2, k=2, dt=F32, path=moe.PATH_AUTO),            # E = k
    dict(T=50, d=64, F=64, E=1, k=1, dt=F32, path=moe.PATH_AUTO),            # a single dense expert
    dict(T=93, d=8, F=8, E=4, k=1, dt=BF16, path=moe.PATH_TENSOR),           # smallest d, F
    dict(T=4, d=8, F=8, E=8, k=2, dt=BF16, path=moe.PATH_STREAM),            # smallest d, F streamed: boxes
                                                                               # mostly past the matrix edges
    dict(T=3, d=64, F=72, E=1, k=1, dt=BF16, path=moe.PATH_STREAM),          # one expert, streamed
    dict(T=40, d=64, F=64, E=1024, k=8, dt=BF16, path=moe.PATH_AUTO),        # largest E and k
    dict(T=2048, d=256, F=512, E=8, k=2, dt=BF16, path=moe.PATH_TENSOR_PAIR),  # 1024 rows/expert: 4 pair tiles
    dict(T=640, d=256, F=512, E=16, k=2, dt=BF16, path=moe.PATH_TENSOR_PAIR),
    dict(T=300, d=64, F=64, E=1024, k=8, dt=BF16, path=moe.PATH_TENSOR_PAIR),  # E = 1024: five stages
    dict(T=2048, d=256, F=512, E=8, k=2, dt=BF16, path=moe.PATH_TENSOR_T),     # 512 rows/expert: 2 full row tiles
    dict(T=640, d=256, F=512, E=16, k=2, dt=BF16, path=moe.PATH_TENSOR_T),
    dict(T=300, d=64, F=64, E=1024, k=8, dt=BF16, path=moe.PATH_TENSOR_T),     # E = 1024: six stages
]


def run_forward(c, path=moe.PATH_AUTO, out_dt=None):
    """moe_forward with its outputs and workspace inside guard bands; the bands are checked."""
    out_dt = c.dt if out_dt is None else out_dt
    g = dict(out=Guarded((c.T, c.d), torch_dtype(out_dt)), idx=Guarded((c.T, c.k), torch.int32),
             gate=Guarded((c.T, c.k), torch.float32), counts=Guarded(c.E, torch.int32))
    out, idx, gate, counts = (g[n].t for n in ("out", "idx", "gate", "counts"))
    ws = guarded_workspace(c)
    moe.forward(c.x, c.w_r, c.b_r, c.w1, c.w2, c.T, c.d, c.F, c.E, c.k, c.dt, out, ws.t, topk_idx=idx,
                topk_gate=gate, counts=counts, path=path, out_dt=out_dt)
    st, detail = moe.get_device_status(ws.t)
    assert st == moe.MOE_OK, (st, detail)
    for name, b in g.items():
        assert b.intact(), f"the forward pass wrote outside {name}"
    assert ws.intact(), "the forward pass wrote outside its workspace"
    return out, idx.cpu().numpy(), gate.cpu().numpy(), counts.cpu().numpy()


@pytest.mark.parametrize("cfg", FORWARD_CASES,
                         ids=lambda c: "T{T}_d{d}_F{F}_E{E}_k{k}_dt{dt}_path{path}".format(**c))
def test_forward(cfg):
    cfg = dict(cfg)
    path = cfg.pop("path")
    c = make_case(**cfg)
    out, idx, gate, counts = run_forward(c, path, out_dt=F32)
    ref = oracle.forward(c.x64, c.wr64, c.w1_host(), c.w2_host(), c.k, c.br64)
    assert np.array_equal(idx, ref["idx"])
    assert np.array_equal(counts, oracle.dispatch(ref["idx"], c.E)["counts"])
    assert np.max(np.abs(gate - ref["gate"])) < 1e-5
    assert rel_rms_err(to_f64(out), ref["out"]) < output_tolerance(c, ref)[0]
    if c.dt == BF16:
        check_bf16_output(c, path, out, ref["out"])


def check_bf16_output(c, path, out_f32, ref):
    """The bf16 output is the fp32 output rounded once to nearest even, so it is within that
    rounding (at most 2^-8 of each value) of the fp32 output's own distance to the oracle."""
    out_bf, _, _, _ = run_forward(c, path, out_dt=BF16)
    assert torch.equal(out_bf.view(torch.int16), out_f32.to(torch.bfloat16).view(torch.int16))
    f32 = to_f64(out_f32)
    assert np.all(np.abs(to_f64(out_bf) - ref) <= np.abs(f32 - ref) + 2.0 ** -8 * np.abs(f32))


def test_forward_all_tokens_to_one_expert():
    b = np.zeros(8, np.float32)
    b[3] = 50.0  # expert 3 is every token's first choice; the rest of the ranking is the plain router's
    c = make_case(T=300, d=128, F=256, E=8, k=2, dt=BF16, bias=b)
    out, idx, gate, counts = run_forward(c, out_dt=F32)
    ref = oracle.forward(c.x64, c.wr64, c.w1_host(), c.w2_host(), 2, c.br64)
    assert counts[3] == c.T
    assert np.all(idx[:, 0] == 3)
    assert np.array_equal(idx, ref["idx"])
    assert rel_rms_err(to_f64(out), ref["out"]) < TOL[BF16]


@pytest.mark.parametrize("cfg", [dict(T=300, d=320, F=64, E=16, k=2, dt=BF16), dict(T=64, d=4096, F=64, E=128, k=4, dt=BF16),
                                 dict(T=70, d=64, F=64, E=5, k=3, dt=F32), dict(T=33, d=64, F=64, E=1024, k=8, dt=BF16)],
                         ids=["tc", "split", "simt_f32", "simt_e1024"])
def test_router_renormalised_gates(cfg):
    c = make_case(**cfg)
    idx = torch.empty((c.T, c.k), dtype=torch.int32, device=DEV)
    gate = torch.empty((c.T, c.k), dtype=torch.float32, device=DEV)
    moe.router_topk(c.x, c.w_r, c.b_r, c.T, c.d, c.E, c.k, c.dt, idx, gate, renormalise=True)
    logits = oracle.router_logits(c.x64, c.wr64, c.br64)
    ridx = oracle.topk_select(logits, c.k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    g = gate.cpu().numpy()
    assert np.max(np.abs(g - oracle.gates_renormalised(logits, ridx))) < 1e-5
    assert np.allclose(g.sum(axis=1), 1.0, atol=1e-5)


@pytest.mark.parametrize("path", [moe.PATH_AUTO, moe.PATH_STREAM])
def test_forward_renormalised_gates(path):
    c = make_case(T=256 if path == moe.PATH_AUTO else 16, d=512, F=512, E=16, k=2, dt=BF16)
    out = torch.empty((c.T, c.d), dtype=torch.float32, device=DEV)
    ws = workspace_for(c)
    moe.forward(c.x, c.w_r, None, c.w1, c.w2, c.T, c.d, c.F, c.E, c.k, c.dt, out, ws, path=path, out_dt=F32,
                renormalise=True)
    assert moe.get_device_status(ws)[0] == moe.MOE_OK
    ref = oracle.forward(c.x64, c.wr64, c.w1_host(), c.w2_host(), c.k, renormalise=True)
    assert rel_rms_err(to_f64(out), ref["out"]) < TOL[BF16]


CAPACITY_FORWARD_CASES = [
    dict(T=640, d=256, F=512, E=16, k=2, dt=BF16, path=moe.PATH_AUTO, cf=1.0),
    dict(T=640, d=256, F=512, E=16, k=2, dt=BF16, path=moe.PATH_TENSOR_PAIR, cf=1.0),
    dict(T=24, d=512, F=512, E=16, k=2, dt=BF16, path=moe.PATH_STREAM, cf=1.0),
    dict(T=200, d=128, F=256, E=8, k=2, dt=F32, path=moe.PATH_AUTO, cf=1.25),
    dict(T=640, d=256, F=1024, E=16, k=2, dt=BF16, path=moe.PATH_SIMT, cf=0.5),
]


@pytest.mark.parametrize("cfg", CAPACITY_FORWARD_CASES, ids=["tensor", "pair", "stream", "simt_f32", "simt_half"])
def test_forward_capacity(cfg):
    cfg = dict(cfg)
    path, cf = cfg.pop("path"), cfg.pop("cf")
    c = make_case(bias=_skewed(cfg["E"]), **cfg)
    C = oracle.capacity(c.T, c.k, c.E, cf)
    out = torch.empty((c.T, c.d), dtype=torch.float32, device=DEV)
    counts = torch.empty(c.E, dtype=torch.int32, device=DEV)
    ws = workspace_for(c)
    moe.forward(c.x, c.w_r, c.b_r, c.w1, c.w2, c.T, c.d, c.F, c.E, c.k, c.dt, out, ws, counts=counts, path=path,
                out_dt=F32, capacity=C)
    st, detail = moe.get_device_status(ws)
    assert st == moe.MOE_OK, (st, detail)
    ref = oracle.forward(c.x64, c.wr64, c.w1_host(), c.w2_host(), c.k, c.br64, cap=C)
    assert not ref["keep"].all()  # some assignments are dropped
    assert np.array_equal(counts.cpu().numpy(), oracle.dispatch(ref["idx"], c.E, cap=C)["counts"])
    assert np.all(counts.cpu().numpy() <= C)
    got = to_f64(out)
    assert rel_rms_err(got, ref["out"]) < output_tolerance(c, ref, cap=C)[0]
    # a token with every assignment dropped gets an exact zero
    gone = ~ref["keep"].any(axis=1)
    assert np.all(got[gone] == 0.0)


STATS_CASES = [
    dict(T=1000, d=256, E=16, k=2, dt=BF16),      # tensor-core router, 8 CTAs
    dict(T=64, d=4096, E=128, k=4, dt=BF16),      # split-K cluster router
    dict(T=300, d=64, E=24, k=3, dt=F32),         # CUDA-core router, 10 CTAs
    dict(T=100, d=64, E=1024, k=8, dt=BF16),      # CUDA-core router, E = 1024
    dict(T=1, d=128, E=64, k=2, dt=BF16),         # one token
]


def check_stats(got, logits, idx, T, E, k):
    ref = oracle.routing_stats(logits, idx)
    g = got.cpu().numpy().astype(np.float64)
    assert g.shape == (moe.router_stats_len(E),)
    assert np.allclose(g[:E], ref["soft_load"], rtol=1e-4, atol=1e-7)
    assert np.array_equal(got.cpu().numpy()[E:2 * E], ref["hard_load"].astype(np.float32))
    assert abs(g[2 * E] - ref["balance"]) <= 1e-6 * ref["balance"] + 1e-9
    assert abs(g[2 * E + 1] - ref["entropy"]) <= 1e-4 * ref["entropy"] + 1e-6


@pytest.mark.parametrize("cfg", STATS_CASES, ids=["tc", "split", "simt_f32", "simt_e1024", "one_token"])
@pytest.mark.parametrize("renormalise", [False, True], ids=["raw", "renorm"])
def test_router_stats(cfg, renormalise):
    ws = None
    for seed, bias in [(0, None), (5, _skewed(cfg["E"]))]:  # the second call also checks the ticket reset
        c = make_case(F=64, seed=seed, bias=bias, **cfg)
        if ws is None:
            ws = workspace_for(c)
        idx = torch.empty((c.T, c.k), dtype=torch.int32, device=DEV)
        gate = torch.empty((c.T, c.k), dtype=torch.float32, device=DEV)
        stats = torch.full((moe.router_stats_len(c.E),), float("nan"), dtype=torch.float32, device=DEV)
        moe.router_topk_stats(c.x, c.w_r, c.b_r, c.T, c.d, c.E, c.k, c.dt, idx, gate, stats, ws,
                              renormalise=renormalise)
        assert moe.get_device_status(ws)[0] == moe.MOE_OK
        logits = oracle.router_logits(c.x64, c.wr64, c.br64)
        ridx = oracle.topk_select(logits, c.k)
        assert np.array_equal(idx.cpu().numpy(), ridx)
        want = oracle.gates_renormalised(logits, ridx) if renormalise else oracle.gates_of(oracle.softmax(logits), ridx)
        assert np.max(np.abs(gate.cpu().numpy() - want)) < 1e-5
        check_stats(stats, logits, ridx, c.T, c.E, c.k)
        again = torch.empty_like(stats)
        moe.router_topk_stats(c.x, c.w_r, c.b_r, c.T, c.d, c.E, c.k, c.dt, idx, gate, again, ws,
                              renormalise=renormalise)
        assert torch.equal(again.view(torch.int32), stats.view(torch.int32))  # fixed reduction order


def test_forward_writes_router_stats():
    c = make_case(T=640, d=256, F=512, E=16, k=2, dt=BF16, bias=_skewed(16, boost=0.5))
    out = torch.empty((c.T, c.d), dtype=torch.float32, device=DEV)
    stats = torch.empty(moe.router_stats_len(c.E), dtype=torch.float32, device=DEV)
    ws = workspace_for(c)
    moe.forward(c.x, c.w_r, c.b_r, c.w1, c.w2, c.T, c.d, c.F, c.E, c.k, c.dt, out, ws, out_dt=F32, router_stats=stats)
    assert moe.get_device_status(ws)[0] == moe.MOE_OK
    logits = oracle.router_logits(c.x64, c.wr64, c.br64)
    check_stats(stats, logits, oracle.topk_select(logits, c.k), c.T, c.E, c.k)
    ref = oracle.forward(c.x64, c.wr64, c.w1_host(), c.w2_host(), c.k, c.br64)
    assert rel_rms_err(to_f64(out), ref["out"]) < TOL[BF16]


HIST_CASES = [
    dict(T=100, d=2048, E=64, cap_factor=0.0),     # split-K cluster router: ranks add into rank 0's counts
    dict(T=1000, d=256, E=256, cap_factor=0.0, boost=0.0),  # E = 256: one chunk group per expert
    dict(T=2049, d=64, E=16, cap_factor=1.1),      # 17 chunks, a 1-token tail tile, capacity drops
    dict(T=777, d=256, E=8, cap_factor=0.6),       # most assignments dropped
]


@pytest.mark.parametrize("cfg", HIST_CASES, ids=["split", "e256", "tail_cap", "cap_small"])
def test_forward_router_histogram_dispatch(cfg):
    """Top-2 bf16 forward: the router's per-tile histograms feed the one-kernel dispatch. Counts,
    indices and output against the oracle, with router statistics written in the same call."""
    T, d, E = cfg["T"], cfg["d"], cfg["E"]
    c = make_case(T=T, d=d, F=128, E=E, k=2, dt=BF16, bias=_skewed(E, boost=cfg.get("boost", 2.5)))
    C = oracle.capacity(T, 2, E, cfg["cap_factor"]) if cfg["cap_factor"] > 0 else 0
    out = torch.empty((T, d), dtype=torch.float32, device=DEV)
    idx = torch.empty((T, 2), dtype=torch.int32, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    stats = torch.empty(moe.router_stats_len(E), dtype=torch.float32, device=DEV)
    ws = workspace_for(c)
    moe.forward(c.x, c.w_r, c.b_r, c.w1, c.w2, T, d, c.F, E, 2, BF16, out, ws, topk_idx=idx, counts=counts,
                out_dt=F32, capacity=C, router_stats=stats)
    assert moe.get_device_status(ws)[0] == moe.MOE_OK
    ref = oracle.forward(c.x64, c.wr64, c.w1_host(), c.w2_host(), 2, c.br64, cap=C if C else None)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert np.array_equal(counts.cpu().numpy(), oracle.dispatch(ref["idx"], E, cap=C if C else None)["counts"])
    check_stats(stats, ref["logits"], ref["idx"], T, E, 2)
    assert rel_rms_err(to_f64(out), ref["out"]) < output_tolerance(c, ref, cap=C if C else None)[0]


def test_router_stats_rejects_small_workspace():
    c = make_case(T=256, d=64, F=64, E=16, k=2, dt=BF16)
    idx = torch.empty((c.T, c.k), dtype=torch.int32, device=DEV)
    gate = torch.empty((c.T, c.k), dtype=torch.float32, device=DEV)
    stats = torch.empty(moe.router_stats_len(c.E), dtype=torch.float32, device=DEV)
    ws = torch.zeros(512, dtype=torch.uint8, device=DEV)
    with pytest.raises(moe.MoeError) as e:
        moe.router_topk_stats(c.x, c.w_r, None, c.T, c.d, c.E, c.k, c.dt, idx, gate, stats, ws)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG


def test_layer_object_capacity_and_stats():
    c = make_case(T=512, d=256, F=256, E=16, k=2, dt=BF16, bias=_skewed(16))
    layer = moe.MoELayer(c.w_r, c.w1, c.w2, k=2, b_r=c.b_r, capacity_factor=1.25)
    stats = torch.empty(moe.router_stats_len(16), dtype=torch.float32, device=DEV)
    out = layer(c.x, out_dtype=torch.float32, router_stats=stats)
    assert layer.device_status()[0] == moe.MOE_OK
    C = oracle.capacity(512, 2, 16, 1.25)
    ref = oracle.forward(c.x64, c.wr64, c.w1_host(), c.w2_host(), 2, c.br64, cap=C)
    assert not ref["keep"].all()
    assert rel_rms_err(to_f64(out), ref["out"]) < output_tolerance(c, ref, cap=C)[0]
    check_stats(stats, ref["logits"], ref["idx"], 512, 16, 2)


def test_forward_zero_tokens():
    c = make_case(T=0, d=64, F=64, E=4, k=2, dt=BF16)
    out = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(moe.workspace_bytes(0, 64, 64, 4, 2, BF16), dtype=torch.uint8, device=DEV)
    moe.workspace_init(ws)
    moe.forward(c.x, c.w_r, None, c.w1, c.w2, 0, 64, 64, 4, 2, BF16, out, ws)
    assert moe.get_device_status(ws)[0] == moe.MOE_OK


@pytest.mark.parametrize("path", [moe.PATH_TENSOR, moe.PATH_STREAM, moe.PATH_TENSOR_PAIR, moe.PATH_TENSOR_T])
def test_forward_is_bit_reproducible(path):
    c = make_case(T=256, d=512, F=512, E=16, k=2, dt=BF16)
    a = run_forward(c, path)[0]
    b = run_forward(c, path)[0]
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_layer_object_matches_oracle():
    c = make_case(T=200, d=256, F=512, E=8, k=2, dt=BF16)
    layer = moe.MoELayer(c.w_r, c.w1, c.w2, k=2)
    out = layer(c.x, out_dtype=torch.float32)
    assert layer.device_status()[0] == moe.MOE_OK
    ref = oracle.forward(c.x64, c.wr64, c.w1_host(), c.w2_host(), 2)
    assert rel_rms_err(to_f64(out), ref["out"]) < TOL[BF16]


def test_bounded_wait_times_out_without_fault():
    ws = torch.empty(4096, dtype=torch.uint8, device=DEV)
    moe.workspace_init(ws)
    moe.selftest_wait_timeout(ws, 2000)
    st, detail = moe.get_device_status(ws)
    assert st == moe.MOE_ERR_DEVICE_TIMEOUT and detail == 99
    # the context stays usable
    c = make_case(T=16, d=64, F=64, E=4, k=2, dt=F32)
    out, idx, _, _ = run_forward(c)
    assert np.array_equal(idx, oracle_routing(c)[0])


def test_device_generator_matches_host():
    t = torch.empty(1 << 20, dtype=torch.bfloat16, device=DEV)
    key = ig.stream_key(0, ig.STREAM_W1)
    ig.fill_device(t, 5000, key, ig.sigma_for_fan_in(4096), BF16)
    host = ig.draw(5000, 1 << 20, key, ig.sigma_for_fan_in(4096), BF16)
    assert np.array_equal(t.view(torch.int16).cpu().numpy().view(np.uint16), host)
    t32 = torch.empty(4099, dtype=torch.float32, device=DEV)
    ig.fill_device(t32, 7, key, 1.0, F32)
    assert np.array_equal(t32.cpu().numpy(), ig.draw(7, 4099, key, 1.0, F32))


def test_binding_refuses_strided_views():
    """A strided view would be read as dense data: the binding refuses it before the library is called."""
    x = torch.zeros((64, 32), dtype=torch.bfloat16, device=DEV)
    w_r = torch.zeros((64, 8), dtype=torch.bfloat16, device=DEV)
    idx = torch.empty((64, 2), dtype=torch.int32, device=DEV)
    gate = torch.empty((64, 2), dtype=torch.float32, device=DEV)
    with pytest.raises(ValueError, match="contiguous"):  # x.t(): T = 32 tokens of d = 64, transposed
        moe.router_topk(x.t(), w_r, None, 32, 64, 8, 2, BF16, idx, gate)
    with pytest.raises(ValueError, match="contiguous"):  # the first 16 columns of each row
        moe.router_topk(x[:, :16], w_r[:16], None, 64, 16, 8, 2, BF16, idx, gate)


def test_layer_refuses_mismatched_inputs():
    """MoELayer takes x [T, d] in its weights' dtype and an out of x's shape; anything else is refused
    before a kernel could read or write it as if it had that shape."""
    w_r = torch.zeros((32, 8), dtype=torch.bfloat16, device=DEV)
    w1 = torch.zeros((8, 32, 64), dtype=torch.bfloat16, device=DEV)
    w2 = torch.zeros((8, 64, 32), dtype=torch.bfloat16, device=DEV)
    layer = moe.MoELayer(w_r, w1, w2, k=2)
    for bad in (torch.zeros((4, 16), dtype=torch.bfloat16, device=DEV),   # width is not d
                torch.zeros((4, 32), dtype=torch.float32, device=DEV),    # not the weights' dtype
                torch.zeros(128, dtype=torch.bfloat16, device=DEV)):      # not [T, d]
        with pytest.raises(ValueError):
            layer(bad)
    x = torch.zeros((4, 32), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError):
        layer(x, out=torch.empty((3, 32), dtype=torch.bfloat16, device=DEV))
    with pytest.raises(ValueError):
        moe.MoELayer(w_r.float(), w1, w2, k=2)
    with pytest.raises(ValueError):
        moe.MoELayer(w_r, w1, w2, k=2, b_r=torch.zeros(7, device=DEV))
    assert layer(x).shape == (4, 32)  # the well-formed call still runs

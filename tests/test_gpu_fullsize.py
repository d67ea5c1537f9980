"""The layer at its full workload sizes, in the launch configuration bench.py times
(moe_forward, automatic kernel choice), against the fp64 oracle.

Routing indices and per-expert counts are compared for every token, and so are the outputs:
the oracle evaluates the routed rows one expert at a time (each routed expert's matrices are
read once), then sums each token's k rows in slot order. fp32 layer: max relative-to-RMS error
1e-4. bf16 layers, on the fp32 output: within 1e-2 of the oracle run with h rounded once to bf16
(the path's one documented intermediate rounding), and within 2e-2 of the exact oracle, or, on
the workloads where that rounding alone already costs more (listed and pinned below), within
1.1x its error plus 2e-3; the bf16 output must be the fp32 output rounded once. The public
dispatch entry is also run at every full size on the oracle's routing and compared bit for bit.
Outputs sit inside guard bands that must stay untouched.
"""
import gc

import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
import sparse_mixture_experts_moe_gb300 as moe
from inputgen import workloads
from moe_cases import Guarded, guarded_workspace, make_case, rel_rms_err, to_f64, torch_dtype

pytestmark = pytest.mark.gpu

DEV = "cuda"

FULL = ["tiny_fp32", "e16_bf16", "prefill_e128", "skew_e128", "decode_t1", "decode_t8", "decode_t64"]


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def oracle_routing(c):
    logits = oracle.router_logits(c.x64, c.wr64, c.br64)
    idx = oracle.topk_select(logits, c.k)
    return idx, oracle.gates_of(oracle.softmax(logits), idx)


# Emulation bar: the bf16 path against the oracle with h rounded once to bf16, its one documented
# intermediate rounding. What remains is fp32 accumulation, the GeLU approximation and the rare h
# element whose fp32 value rounds to the neighbouring bf16 value; a wrong tile or row shows up at
# O(1) of the output RMS. Measured 0.0045 (prefill_e128).
EMULATION_TOL = 1e-2

# Workloads on which the stated metric's bar (max |error| / RMS <= 2e-2 on all T*d outputs) is
# raised: there the one rounding of h to bf16 alone, evaluated by the oracle, already costs more.
# Their outputs are heavy-tailed (a token with a gate near 0.5 has outputs up to 19x the RMS), and
# a rounding error proportional to the output lands far above 2e-2 of the RMS. The bar is then
# 1.1x that rounding's error plus 2e-3, the rule of every smaller case (moe_cases.output_tolerance).
FULL_SIZE_RAISED = {"e16_bf16", "prefill_e128", "skew_e128"}


def oracle_all_tokens(c, ridx, rgate):
    """out[t] for every token, exact, and the same with h rounded once to bf16 (bf16 layers): dispatch,
    the routed rows of each expert through both projections, the gate, and the fixed-order k-way sum
    (the oracle's step functions, which compose to its forward pass; each routed expert's matrices are
    read once per projection)."""
    dp = oracle.dispatch(ridx, c.E, rgate)
    h = oracle.expert_rows_up(c.x64[dp["perm_token"]], dp["offsets"], c.w1_host())
    ref = oracle.combine(oracle.expert_rows_down(h, dp["offsets"], dp["row_gate"], c.w2_host()), dp["row_of"])
    if c.dt != ig.DTYPE_BF16:
        return ref, None
    hb = ig.as_f64(ig.f32_to_bf16_bits(h.astype(np.float32)), ig.DTYPE_BF16)
    del h
    emul = oracle.combine(oracle.expert_rows_down(hb, dp["offsets"], dp["row_gate"], c.w2_host()), dp["row_of"])
    return ref, emul


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name):
    w = workloads.get(name)
    c = make_case(T=w.T, d=w.d, F=w.F, E=w.E, k=w.k, dt=w.dtype, bias_scale=workloads.bias_scale(w))
    ws = guarded_workspace(c)
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device=DEV)
    counts = torch.empty(w.E, dtype=torch.int32, device=DEV)
    out32 = Guarded((w.T, w.d), torch.float32)
    moe.forward(c.x, c.w_r, c.b_r, c.w1, c.w2, w.T, w.d, w.F, w.E, w.k, w.dtype, out32.t, ws.t, topk_idx=idx,
                counts=counts, out_dt=ig.DTYPE_F32)
    out_native = Guarded((w.T, w.d), torch_dtype(w.dtype))
    moe.forward(c.x, c.w_r, c.b_r, c.w1, c.w2, w.T, w.d, w.F, w.E, w.k, w.dtype, out_native.t, ws.t)
    st, detail = moe.get_device_status(ws.t)
    assert st == moe.MOE_OK, (moe.status_string(st), detail)
    assert out32.intact() and out_native.intact() and ws.intact()

    # routing of every token, bit-exact
    ridx, rgate = oracle_routing(c)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.array_equal(counts.cpu().numpy(), oracle.dispatch(ridx, w.E)["counts"])

    # outputs of every token
    ref, emul = oracle_all_tokens(c, ridx, rgate)
    got = to_f64(out32.t)
    err = rel_rms_err(got, ref)
    if w.dtype == ig.DTYPE_F32:
        assert err < 1e-4, err
        return
    assert rel_rms_err(got, emul) < EMULATION_TOL
    rounding = rel_rms_err(emul, ref)
    bar = max(2e-2, 1.1 * rounding + 2e-3)
    assert (bar > 2e-2) == (name in FULL_SIZE_RAISED), (name, rounding)
    assert err < bar, (err, bar, rounding)
    assert torch.equal(out_native.t.view(torch.int16), out32.t.to(torch.bfloat16).view(torch.int16))


@pytest.mark.parametrize("name", FULL)
def test_full_size_dispatch(name):
    """moe_dispatch on the oracle's routing of the full workload: counts, offsets, perm_token, row_of,
    row_gate and x_perm bit for bit, every output inside untouched guard bands."""
    w = workloads.get(name)
    c = make_case(T=w.T, d=w.d, F=8, E=w.E, k=w.k, dt=w.dtype, bias_scale=workloads.bias_scale(w))
    ridx, rgate = oracle_routing(c)
    A = c.A
    g = dict(counts=Guarded(w.E, torch.int32), offsets=Guarded(w.E + 1, torch.int32),
             perm_token=Guarded(A, torch.int32), row_of=Guarded((w.T, w.k), torch.int32),
             row_gate=Guarded(A, torch.float32), x_perm=Guarded((A, w.d), torch_dtype(w.dtype)))
    ws = guarded_workspace(c)
    ti = torch.from_numpy(ridx.astype(np.int32)).to(DEV)
    tg = torch.from_numpy(rgate.astype(np.float32)).to(DEV)
    moe.dispatch(c.x, ti, tg, w.T, w.d, w.E, w.k, w.dtype, g["counts"].t, g["offsets"].t, g["perm_token"].t,
                 g["row_of"].t, g["row_gate"].t, g["x_perm"].t, ws.t)
    st, detail = moe.get_device_status(ws.t)
    assert st == moe.MOE_OK, (moe.status_string(st), detail)
    for n, b in g.items():
        assert b.intact(), n
    assert ws.intact()
    ref = oracle.dispatch(ridx, w.E, rgate.astype(np.float32))
    for n in ("counts", "offsets", "perm_token", "row_of"):
        assert np.array_equal(g[n].t.cpu().numpy(), ref[n]), n
    assert np.array_equal(g["row_gate"].t.cpu().numpy(), ref["row_gate"].astype(np.float32))
    perm = torch.from_numpy(ref["perm_token"]).to(DEV)
    assert torch.equal(g["x_perm"].t, c.x[perm])


class OracleQuantised:
    """Expert e's matrix as the oracle quantises and restores it (its own 64 x 64 block quantiser on
    the exact stored weights), computed on access: only routed experts are read."""

    def __init__(self, view, bits):
        self.view, self.bits = view, bits

    def __getitem__(self, e):
        w = self.view[e].astype(np.float32)  # exact: bf16 values are fp32 numbers
        return oracle.dequantize_blocks(oracle.quantize_blocks(w, self.bits))


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("name", ["decode_t1", "decode_t8"])
def test_full_size_quantised_decode(name, bits):
    """moe_forward_q on the decode workloads' full sizes (d = d_ff = 8192, E = 128), weights quantised
    on the device, against the oracle run on the oracle's own quantisation of the same weights, on
    every token."""
    w = workloads.get(name)
    c = make_case(T=w.T, d=w.d, F=w.F, E=w.E, k=w.k, dt=w.dtype, bias_scale=workloads.bias_scale(w))
    q1, q2 = moe.quantize(c.w1, bits), moe.quantize(c.w2, bits)
    ws = guarded_workspace(c)
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device=DEV)
    out32 = Guarded((w.T, w.d), torch.float32)
    moe.forward_q(c.x, c.w_r, c.b_r, q1, q2, w.T, w.d, w.F, w.E, w.k, bits, out32.t, ws.t, topk_idx=idx,
                  out_dt=ig.DTYPE_F32)
    out_bf = Guarded((w.T, w.d), torch.bfloat16)
    moe.forward_q(c.x, c.w_r, c.b_r, q1, q2, w.T, w.d, w.F, w.E, w.k, bits, out_bf.t, ws.t)
    st, detail = moe.get_device_status(ws.t)
    assert st == moe.MOE_OK, (moe.status_string(st), detail)
    assert out32.intact() and out_bf.intact() and ws.intact()
    ridx, rgate = oracle_routing(c)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    dp = oracle.dispatch(ridx, c.E, rgate)
    y = oracle.expert_rows_ffn(c.x64[dp["perm_token"]], dp["offsets"], dp["row_gate"],
                               OracleQuantised(c.w1_host(), bits), OracleQuantised(c.w2_host(), bits))
    ref = oracle.combine(y, dp["row_of"])
    assert rel_rms_err(to_f64(out32.t), ref) < 2e-2
    assert torch.equal(out_bf.t.view(torch.int16), out32.t.to(torch.bfloat16).view(torch.int16))


def test_activations_past_2_31_elements():
    """T = 65536 tokens with d_ff = 32768: h [T*k, d_ff] holds 2^32 elements, so every offset past
    element 2^31 has to be computed in 64 bits. Routing is compared for every token, and the outputs
    of the tokens whose rows lie furthest into h (past element 2^31) against the oracle; the outputs and
    the workspace sit inside guard bands."""
    T, d, F, E, k = 65536, 256, 32768, 16, 2
    c = make_case(T=T, d=d, F=F, E=E, k=k, dt=ig.DTYPE_BF16)
    ws = guarded_workspace(c)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    out32 = Guarded((T, d), torch.float32)
    moe.forward(c.x, c.w_r, c.b_r, c.w1, c.w2, T, d, F, E, k, c.dt, out32.t, ws.t, topk_idx=idx,
                out_dt=ig.DTYPE_F32)
    st, detail = moe.get_device_status(ws.t)
    assert st == moe.MOE_OK, (moe.status_string(st), detail)
    assert out32.intact() and ws.intact()
    ridx, rgate = oracle_routing(c)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    dp_all = oracle.dispatch(ridx, E, rgate)
    last_row = dp_all["row_of"].max(axis=1)
    sel = np.sort(np.argsort(last_row)[-8:])  # the 8 tokens with rows furthest into h
    assert (last_row[sel] * F >= 2 ** 31).all()
    # the oracle on those tokens alone: their rows through both projections (h exact, and h rounded
    # once to bf16 as the path rounds it), then the fixed-order k-way sum
    dp = oracle.dispatch(ridx[sel], E, rgate[sel])
    xs = c.x64[sel][dp["perm_token"]]
    w1h, w2h = c.w1_host(), c.w2_host()
    h = oracle.expert_rows_up(xs, dp["offsets"], w1h)
    ref = oracle.combine(oracle.expert_rows_down(h, dp["offsets"], dp["row_gate"], w2h), dp["row_of"])
    hb = ig.as_f64(ig.f32_to_bf16_bits(h.astype(np.float32)), ig.DTYPE_BF16)
    emul = oracle.combine(oracle.expert_rows_down(hb, dp["offsets"], dp["row_gate"], w2h), dp["row_of"])
    got = to_f64(out32.t)[sel]
    assert rel_rms_err(got, emul) < EMULATION_TOL
    rounding = rel_rms_err(emul, ref)
    assert rel_rms_err(got, ref) < max(2e-2, 1.1 * rounding + 2e-3), (rel_rms_err(got, ref), rounding)

"""The layer at its full workload sizes, in the launch configuration bench.py times
(moe_forward, automatic kernel choice), against the fp64 oracle.

Routing indices and per-expert counts are compared for every token (the oracle's
logits are cheap); outputs are compared on a sample of tokens that the oracle
evaluates one expert matrix at a time (max relative-to-RMS error 2e-2 on the fp32
output; the bf16 output must be that fp32 output rounded once).
"""
import gc

import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
import sparse_mixture_experts_moe_gb300 as moe
from inputgen import workloads
from moe_cases import make_case, rel_rms_err, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"

# workload -> number of sampled tokens for the output check (None: all tokens)
SAMPLES = {
    "tiny_fp32": None,
    "e16_bf16": None,
    "prefill_e128": 12,
    "skew_e128": 12,
    "decode_t1": None,
    "decode_t8": None,
    "decode_t64": 6,
}


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", list(SAMPLES))
def test_full_size_workload(name):
    w = workloads.get(name)
    c = make_case(T=w.T, d=w.d, F=w.F, E=w.E, k=w.k, dt=w.dtype, bias_scale=workloads.bias_scale(w))
    ws = torch.empty(moe.workspace_bytes(w.T, w.d, w.F, w.E, w.k, w.dtype), dtype=torch.uint8, device=DEV)
    moe.workspace_init(ws)
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device=DEV)
    counts = torch.empty(w.E, dtype=torch.int32, device=DEV)
    out32 = torch.empty((w.T, w.d), dtype=torch.float32, device=DEV)
    moe.forward(c.x, c.w_r, c.b_r, c.w1, c.w2, w.T, w.d, w.F, w.E, w.k, w.dtype, out32, ws, topk_idx=idx,
                counts=counts, out_dt=ig.DTYPE_F32)
    out_native = torch.empty((w.T, w.d), dtype=torch.bfloat16 if w.dtype == ig.DTYPE_BF16 else torch.float32,
                             device=DEV)
    moe.forward(c.x, c.w_r, c.b_r, c.w1, c.w2, w.T, w.d, w.F, w.E, w.k, w.dtype, out_native, ws)
    st, detail = moe.get_device_status(ws)
    assert st == moe.MOE_OK, (moe.status_string(st), detail)

    # routing of every token, bit-exact
    logits = oracle.router_logits(c.x64, c.wr64, c.br64)
    ridx = oracle.topk_select(logits, w.k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.array_equal(counts.cpu().numpy(), oracle.dispatch(ridx, w.E)["counts"])

    # outputs on sampled tokens
    n = SAMPLES[name]
    rng = np.random.default_rng(1234)
    toks = np.arange(w.T) if n is None or n >= w.T else np.sort(rng.choice(w.T, size=n, replace=False))
    ref = oracle.forward(c.x64[toks], c.wr64, c.w1_host(), c.w2_host(), w.k, c.br64)
    assert np.array_equal(ref["idx"], ridx[toks])
    tol = 1e-4 if w.dtype == ig.DTYPE_F32 else 2e-2
    got32 = to_f64(out32)[toks]
    assert rel_rms_err(got32, ref["out"]) < tol
    if w.dtype == ig.DTYPE_BF16:
        assert torch.equal(out_native.view(torch.int16), out32.to(torch.bfloat16).view(torch.int16))


class OracleQuantised:
    """Expert e's matrix as the oracle quantises and restores it (its own 64 x 64 block quantiser on
    the exact stored weights), computed on access: only routed experts are read."""

    def __init__(self, view, bits):
        self.view, self.bits = view, bits

    def __getitem__(self, e):
        w = self.view[e].astype(np.float32)  # exact: bf16 values are fp32 numbers
        return oracle.dequantize_blocks(oracle.quantize_blocks(w, self.bits))


# quantised decode at full size: workload -> sampled tokens for the output check (None: all)
SAMPLES_Q = {"decode_t1": None, "decode_t8": 4}


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("name", list(SAMPLES_Q))
def test_full_size_quantised_decode(name, bits):
    """moe_forward_q on the decode workloads' full sizes (d = d_ff = 8192, E = 128), weights quantised
    on the device, against the oracle run on the oracle's own quantisation of the same weights."""
    w = workloads.get(name)
    c = make_case(T=w.T, d=w.d, F=w.F, E=w.E, k=w.k, dt=w.dtype, bias_scale=workloads.bias_scale(w))
    q1, q2 = moe.quantize(c.w1, bits), moe.quantize(c.w2, bits)
    ws = torch.empty(moe.workspace_bytes(w.T, w.d, w.F, w.E, w.k, w.dtype), dtype=torch.uint8, device=DEV)
    moe.workspace_init(ws)
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device=DEV)
    out32 = torch.empty((w.T, w.d), dtype=torch.float32, device=DEV)
    moe.forward_q(c.x, c.w_r, c.b_r, q1, q2, w.T, w.d, w.F, w.E, w.k, bits, out32, ws, topk_idx=idx,
                  out_dt=ig.DTYPE_F32)
    out_bf = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=DEV)
    moe.forward_q(c.x, c.w_r, c.b_r, q1, q2, w.T, w.d, w.F, w.E, w.k, bits, out_bf, ws)
    st, detail = moe.get_device_status(ws)
    assert st == moe.MOE_OK, (moe.status_string(st), detail)
    ridx = oracle.topk_select(oracle.router_logits(c.x64, c.wr64, c.br64), w.k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    n = SAMPLES_Q[name]
    rng = np.random.default_rng(4321)
    toks = np.arange(w.T) if n is None or n >= w.T else np.sort(rng.choice(w.T, size=n, replace=False))
    ref = oracle.forward(c.x64[toks], c.wr64, OracleQuantised(c.w1_host(), bits),
                         OracleQuantised(c.w2_host(), bits), w.k, c.br64)
    assert rel_rms_err(to_f64(out32)[toks], ref["out"]) < 2e-2
    assert torch.equal(out_bf.view(torch.int16), out32.to(torch.bfloat16).view(torch.int16))

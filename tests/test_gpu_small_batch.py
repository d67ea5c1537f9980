"""Decode-sized batches (T <= 8, bf16, weight-streaming GEMMs): the one-launch router + dispatch,
whose FFN reads x rows through the permutation (and, for one token, splits the weight slabs between
CTAs, stream-K), against the fp64 oracle.

Bars as for every forward: routing indices and counts bit-exact, gates within 1e-5, the output
within 2e-2 of its RMS (or the bf16-h rounding bound when that alone is larger).
"""
import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
import sparse_mixture_experts_moe_gb300 as moe
from moe_cases import make_case, output_tolerance, rel_rms_err, to_f64, workspace_for

pytestmark = pytest.mark.gpu

BF16 = ig.DTYPE_BF16
DEV = "cuda"


CASES = [
    dict(T=1, d=4096, F=64, E=64, k=2),               # decode shape: 64 CTAs, 8 clusters
    dict(T=8, d=1024, F=128, E=128, k=2),             # a decode batch: 16 CTAs
    dict(T=3, d=64, F=64, E=8, k=8),                  # k = E: every expert, 8 CTAs with 8 rows each
    dict(T=5, d=256, F=64, E=1024, k=4),              # E = 1024: two passes over expert pairs
    dict(T=2, d=136, F=64, E=8, k=1),                 # d = 17 x 8: CTAs with empty row ranges
    dict(T=2, d=136, F=64, E=6, k=1),                 # E % 8 != 0: the separate router and dispatch
    dict(T=8, d=512, F=64, E=16, k=2, cf=0.5),        # capacity: assignments dropped
    dict(T=2, d=512, F=64, E=8, k=4, cf=0.5),         # capacity on the plain-CTA (T <= 2) variant
    dict(T=4, d=512, F=64, E=32, k=3, bias=True),     # router bias
    dict(T=1, d=136, F=200, E=8, k=3),                # one token, ragged slabs: stream-K pieces of 8
    dict(T=1, d=2048, F=1024, E=16, k=8),             # one token, k = 8: slabs split between two CTAs
]


@pytest.mark.parametrize("renormalise", [False, True], ids=["raw", "renorm"])
@pytest.mark.parametrize("cfg", CASES, ids=["t1", "t8", "k_eq_e", "e1024", "d136", "e6", "cap", "cap_t2", "bias",
                                         "t1_ragged", "t1_k8"])
def test_forward_small_batch(cfg, renormalise):
    cfg = dict(cfg)
    cf = cfg.pop("cf", 0.0)
    bias = cfg.pop("bias", False)
    T, E, k = cfg["T"], cfg["E"], cfg["k"]
    c = make_case(dt=BF16, bias=np.linspace(-1.0, 1.0, E, dtype=np.float32) if bias else None, **cfg)
    cap = oracle.capacity(T, k, E, cf) if cf > 0 else 0
    out = torch.empty((T, c.d), dtype=torch.float32, device=DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    gate = torch.empty((T, k), dtype=torch.float32, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    ws = workspace_for(c)
    for _ in range(2):  # the second call also checks that the ticket was reset
        moe.forward(c.x, c.w_r, c.b_r, c.w1, c.w2, T, c.d, c.F, E, k, BF16, out, ws, topk_idx=idx,
                    topk_gate=gate, counts=counts, out_dt=ig.DTYPE_F32, renormalise=renormalise, capacity=cap)
        assert moe.get_device_status(ws)[0] == moe.MOE_OK
        ref = oracle.forward(c.x64, c.wr64, c.w1_host(), c.w2_host(), k, c.br64, renormalise=renormalise,
                             cap=cap if cap else None)
        assert np.array_equal(idx.cpu().numpy(), ref["idx"])
        assert np.max(np.abs(gate.cpu().numpy() - ref["gate"])) < 1e-5
        assert np.array_equal(counts.cpu().numpy(),
                              oracle.dispatch(ref["idx"], E, cap=cap if cap else None)["counts"])
        assert rel_rms_err(to_f64(out), ref["out"]) < output_tolerance(c, ref, cap if cap else None)[0]


def test_small_batch_matches_separate_calls():
    """The fused router + dispatch and the separate entry points give the same routing and the same
    output bits (the same kernels compute the expert halves and the combine)."""
    c = make_case(T=6, d=1024, F=256, E=32, k=2, dt=BF16)
    T, d, F, E, k = c.T, c.d, c.F, c.E, c.k
    out = torch.empty((T, d), dtype=torch.bfloat16, device=DEV)
    ws = workspace_for(c)
    moe.forward(c.x, c.w_r, c.b_r, c.w1, c.w2, T, d, F, E, k, BF16, out, ws)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    gate = torch.empty((T, k), dtype=torch.float32, device=DEV)
    moe.router_topk(c.x, c.w_r, c.b_r, T, d, E, k, BF16, idx, gate)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    row_of = torch.empty((T, k), dtype=torch.int32, device=DEV)
    row_gate = torch.empty(T * k, dtype=torch.float32, device=DEV)
    x_perm = torch.empty((T * k, d), dtype=torch.bfloat16, device=DEV)
    moe.dispatch(c.x, idx, gate, T, d, E, k, BF16, counts, offsets, perm, row_of, row_gate, x_perm, ws)
    y_perm = torch.empty((T * k, d), dtype=torch.float32, device=DEV)
    moe.grouped_ffn(x_perm, c.w1, c.w2, offsets, row_gate, T, d, F, E, k, BF16, y_perm, ws)
    out2 = torch.empty_like(out)
    moe.combine(y_perm, row_of, T, d, k, BF16, out2)
    logits = oracle.router_logits(c.x64, c.wr64, c.br64)
    assert np.array_equal(idx.cpu().numpy(), oracle.topk_select(logits, k))
    # routing equal; gates may differ in the last bit (a different softmax-sum order), so the
    # outputs agree to the gate's rounding, not bit for bit
    assert rel_rms_err(to_f64(out), to_f64(out2)) < 1e-3

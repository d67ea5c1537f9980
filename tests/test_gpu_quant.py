"""Block-quantised expert weights on the GPU: the device quantiser's codes and (scale, min) pairs
equal the oracle's bit for bit (both decide the codes in fp32), and the layer streaming INT4 / INT8
codes matches the fp64 oracle run on the dequantised weights."""
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


def unpack_codes(raw, E, K, N, bits):
    """Device code format -> codes [E, K, N].

    INT4: per expert [N/64 slabs][K/16 k-blocks][32 lanes][4 words]; k-block 4b + j is step j of the
    64-deep block b; lane 4g + t, word m covers columns c0 = 16m + g and c1 = c0 + 8 at k-rows
    kp .. kp+3 with kp = 64b + 16t + 4j, nibble i (bits 4i..4i+3) holding (k, column) = (kp, c0),
    (kp, c1), (kp+2, c0), (kp+2, c1), (kp+1, c0), (kp+1, c1), (kp+3, c0), (kp+3, c1) for i = 0..7.
    INT8: per expert [N/64 slabs][K/16 steps][2 halves][32 lanes][16 bytes]; step 2p + s is step s of
    the 32-deep range p; half h of lane 4g + t holds column tiles m = 2h, 2h + 1, 8 bytes each: byte q of
    tile m holds (k, column) = (kp, c0), (kp+1, c0), (kp, c1), (kp+1, c1), (kp+2, c0), (kp+3, c0),
    (kp+2, c1), (kp+3, c1) for q = 0..7, with kp = 32p + 8t + 4s, c0 = 16m + g and c1 = c0 + 8."""
    codes = np.zeros((E, K, N), np.uint8)
    if bits == 4:
        words = np.ascontiguousarray(raw).view("<u4").reshape(E, N // 64, K // 16, 32, 4)
        lane = np.arange(32)
        g, t = lane // 4, lane % 4
        slab = np.arange(N // 64)[:, None, None]
        k16 = np.arange(K // 16)[None, :, None]
        for m in range(4):
            for i, (dk, dc) in enumerate([(0, 0), (0, 8), (2, 0), (2, 8), (1, 0), (1, 8), (3, 0), (3, 8)]):
                k = (k16 // 4) * 64 + 4 * (k16 % 4) + (16 * t + dk)[None, None, :]
                c = slab * 64 + (16 * m + g + dc)[None, None, :]
                codes[:, k, c] = (words[..., m] >> (4 * i)) & 0xF
    else:
        b = np.ascontiguousarray(raw).reshape(E, N // 64, K // 16, 2, 32, 16)
        lane = np.arange(32)
        g, t = lane // 4, lane % 4
        slab = np.arange(N // 64)[:, None, None]
        k16 = np.arange(K // 16)[None, :, None]
        for h in range(2):
            for mi in range(2):
                m = 2 * h + mi
                for q, (dk, dc) in enumerate([(0, 0), (1, 0), (0, 8), (1, 8), (2, 0), (3, 0), (2, 8), (3, 8)]):
                    k = (k16 // 2) * 32 + 4 * (k16 % 2) + (8 * t + dk)[None, None, :]
                    c = slab * 64 + (16 * m + g + dc)[None, None, :]
                    codes[:, k, c] = b[:, :, :, h, :, 8 * mi + q]
    return codes


def oracle_quant(w_dev, bits):
    w = to_f64(w_dev).astype(np.float32)  # exact: bf16 and fp32 values are fp32 numbers
    return [oracle.quantize_blocks(w[e], bits) for e in range(w.shape[0])]


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("dt", [BF16, F32], ids=["bf16", "f32"])
def test_quantizer_matches_oracle(bits, dt):
    c = make_case(T=4, d=128, F=192, E=3, k=2, dt=dt)
    w = c.w1.clone()
    w[1, 64:128, 0:64] = 0.25  # a flat block: scale 0, codes 0
    codes, sm = moe.quantize(w, bits)
    torch.cuda.synchronize()
    assert codes.numel() == oracle.packed_code_bytes(128, 192, bits) * 3
    got = unpack_codes(codes.cpu().numpy(), 3, 128, 192, bits)
    smh = sm.cpu().numpy()
    for e, q in enumerate(oracle_quant(w, bits)):
        assert np.array_equal(got[e], q["codes"])
        assert np.array_equal(smh[e, :, :, 0], q["scale"])
        assert np.array_equal(smh[e, :, :, 1], q["min"])
    assert np.all(smh[1, 1, 0] == [0.0, 0.25])


def q_case(T, d, F, E, k, bits, seed=0, bias=None):
    c = make_case(T=T, d=d, F=F, E=E, k=k, dt=BF16, seed=seed, bias=bias)
    q1, q2 = moe.quantize(c.w1, bits), moe.quantize(c.w2, bits)
    w1h = {e: oracle.dequantize_blocks(q) for e, q in enumerate(oracle_quant(c.w1, bits))}
    w2h = {e: oracle.dequantize_blocks(q) for e, q in enumerate(oracle_quant(c.w2, bits))}
    return c, q1, q2, w1h, w2h


def q_tolerance(c, ref, w1h, w2h):
    """2e-2, unless rounding h to bf16 (the path's one intermediate rounding) alone costs more on this
    shape: then 1.1x that, computed with the oracle, plus 2e-3."""
    dp = oracle.dispatch(ref["idx"], c.E, ref["gate"])
    h = oracle.expert_rows_up(c.x64[dp["perm_token"]], dp["offsets"], w1h)
    hb = ig.as_f64(ig.f32_to_bf16_bits(h.astype(np.float32)), BF16)
    y = oracle.expert_rows_down(hb, dp["offsets"], dp["row_gate"], w2h)
    return max(2e-2, 1.1 * rel_rms_err(oracle.combine(y, dp["row_of"]), ref["out"]) + 2e-3)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("cfg", [dict(T=1, d=1024, F=1024, E=16, k=2),     # one token
                                 dict(T=8, d=512, F=768, E=32, k=2),       # decode batch, 2 rows a pass
                                 dict(T=64, d=256, F=512, E=8, k=2),       # 4 rows a pass, several passes
                                 dict(T=300, d=128, F=192, E=4, k=2),      # many passes over each expert
                                 dict(T=40, d=256, F=256, E=64, k=2),      # 2 rows a pass, some experts twice
                                 dict(T=1, d=64, F=64, E=8, k=2)],         # smallest matrices: one block
                         ids=["t1", "t8", "t64", "t300", "t40_e64", "t1_tiny"])
def test_forward_q_matches_oracle(cfg, bits):
    c, q1, q2, w1h, w2h = q_case(bits=bits, **cfg)
    out = torch.empty((c.T, c.d), dtype=torch.float32, device=DEV)
    idx = torch.empty((c.T, c.k), dtype=torch.int32, device=DEV)
    ws = workspace_for(c)
    moe.forward_q(c.x, c.w_r, c.b_r, q1, q2, c.T, c.d, c.F, c.E, c.k, bits, out, ws, topk_idx=idx, out_dt=F32)
    assert moe.get_device_status(ws)[0] == moe.MOE_OK
    ref = oracle.forward(c.x64, c.wr64, w1h, w2h, c.k, c.br64)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert rel_rms_err(to_f64(out), ref["out"]) < q_tolerance(c, ref, w1h, w2h)
    # bf16 output: the fp32 output rounded once
    out_bf = torch.empty((c.T, c.d), dtype=torch.bfloat16, device=DEV)
    moe.forward_q(c.x, c.w_r, c.b_r, q1, q2, c.T, c.d, c.F, c.E, c.k, bits, out_bf, ws)
    assert torch.equal(out_bf.view(torch.int16), out.to(torch.bfloat16).view(torch.int16))


def test_expert_halves_q_match_oracle():
    c, q1, q2, w1h, w2h = q_case(T=16, d=256, F=320, E=8, k=2, bits=4)
    ridx = oracle.topk_select(oracle.router_logits(c.x64, c.wr64, c.br64), c.k)
    gate = oracle.gates_of(oracle.softmax(oracle.router_logits(c.x64, c.wr64, c.br64)), ridx)
    dp = oracle.dispatch(ridx, c.E, gate.astype(np.float32))
    A = c.T * c.k
    x_perm = c.x[torch.from_numpy(dp["perm_token"]).to(DEV)].contiguous()
    offs = torch.from_numpy(dp["offsets"].astype(np.int32)).to(DEV)
    rg = torch.from_numpy(dp["row_gate"].astype(np.float32)).to(DEV)
    h = torch.empty((A, c.F), dtype=torch.bfloat16, device=DEV)
    moe.expert_up_q(x_perm, q1[0], q1[1], offs, c.T, c.d, c.F, c.E, c.k, 4, h)
    h_ref = oracle.expert_rows_up(c.x64[dp["perm_token"]], dp["offsets"], w1h)
    hg = to_f64(h)
    # one rounding to bf16 on top of fp32 accumulation: within 2^-8 relative plus a small absolute slack
    assert np.all(np.abs(hg - h_ref) <= 2.0 ** -8 * np.abs(h_ref) + 1e-3 * np.sqrt(np.mean(h_ref ** 2)))
    y = torch.empty((A, c.d), dtype=torch.float32, device=DEV)
    moe.expert_down_q(h, q2[0], q2[1], offs, rg, c.T, c.d, c.F, c.E, c.k, 4, y)
    y_ref = oracle.expert_rows_down(hg, dp["offsets"], dp["row_gate"], w2h)
    assert rel_rms_err(to_f64(y), y_ref) < 1e-5


def test_layer_quantised_with_graph():
    c, q1, q2, w1h, w2h = q_case(T=8, d=512, F=512, E=16, k=2, bits=4)
    layer = moe.MoELayer(c.w_r, c.w1, c.w2, k=2, b_r=c.b_r, weight_bits=4)
    out = torch.empty((c.T, c.d), dtype=torch.float32, device=DEV)
    g = layer.graph(c.x, out)
    g.launch()
    direct = layer(c.x, out_dtype=torch.float32)
    assert layer.device_status()[0] == moe.MOE_OK
    assert torch.equal(out.view(torch.int32), direct.view(torch.int32))
    ref = oracle.forward(c.x64, c.wr64, w1h, w2h, 2, c.br64)
    assert rel_rms_err(to_f64(out), ref["out"]) < q_tolerance(c, ref, w1h, w2h)


def test_quantised_rejects_bad_sizes():
    c = make_case(T=4, d=96, F=64, E=2, k=2, dt=BF16)  # d not a multiple of 64
    with pytest.raises(moe.MoeError):
        moe.quantize(c.w1, 4)
    with pytest.raises(moe.MoeError):
        moe.quantize(make_case(T=4, d=64, F=64, E=2, k=2, dt=BF16).w1, 5)

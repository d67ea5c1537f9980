"""Distinct workspaces from distinct host threads, each on its own stream.

The header promises that the library holds no global mutable state, so layers with their own
workspaces can be enqueued from several host threads at once. Here four layers of different kernel
families run at the same time, each from its own thread and on its own stream:
- the CTA-pair GEMM under skewed routing, whose work items come from a counter in the workspace;
- bf16 weight streaming;
- INT4 weights;
- the fp32 CUDA-core path.

Every output of every step must equal, bit for bit, the output of the same call made alone. The
layer is deterministic, so any difference means shared state or a race.
"""
import threading

import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
import sparse_mixture_experts_moe_gb300 as moe
from moe_cases import make_case, workspace_for, torch_dtype

DEV = "cuda"
STEPS = 8


class Layer:
    """One layer instance with its own workspace: run(out, stream) enqueues one forward pass."""

    def __init__(self, name, T, d, F, E, k, dt, bias_scale=None, path=moe.PATH_AUTO, bits=0):
        self.name, self.path, self.bits = name, path, bits
        self.c = make_case(T=T, d=d, F=F, E=E, k=k, dt=dt, bias_scale=bias_scale)
        self.ws = workspace_for(self.c)
        self.q1 = self.q2 = None
        if bits:
            self.q1, self.q2 = moe.quantize(self.c.w1, bits), moe.quantize(self.c.w2, bits)
        self.out_dtype = torch.bfloat16 if bits else torch_dtype(dt)

    def empty_out(self):
        return torch.empty((self.c.T, self.c.d), dtype=self.out_dtype, device=DEV)

    def run(self, out, stream=None):
        c = self.c
        if self.bits:
            moe.forward_q(c.x, c.w_r, c.b_r, self.q1, self.q2, c.T, c.d, c.F, c.E, c.k, self.bits, out, self.ws,
                          stream=stream)
        else:
            moe.forward(c.x, c.w_r, c.b_r, c.w1, c.w2, c.T, c.d, c.F, c.E, c.k, c.dt, out, self.ws, path=self.path,
                        stream=stream)


def layers():
    bf16, f32 = ig.DTYPE_BF16, ig.DTYPE_F32
    return [
        # 6 experts above one 256-row tile and 10 below it: the pair GEMM's counter and item ring
        Layer("skew_pair", T=2048, d=256, F=512, E=16, k=2, dt=bf16, bias_scale=0.6, path=moe.PATH_TENSOR_T),
        Layer("decode_stream", T=4, d=1024, F=1024, E=32, k=2, dt=bf16),
        Layer("decode_int4", T=8, d=512, F=512, E=16, k=2, dt=bf16, bits=4),
        Layer("fp32", T=64, d=128, F=256, E=8, k=2, dt=f32),
    ]


def test_skew_case_mixes_heavy_and_light_experts():  # host only
    """The first layer really takes the pair GEMM's mixed path: experts both above and below 256 rows."""
    c = make_case(T=2048, d=256, F=512, E=16, k=2, dt=ig.DTYPE_BF16, bias_scale=0.6, host_only=True)
    counts = oracle.dispatch(oracle.topk_select(oracle.router_logits(c.x64, c.wr64, c.br64), 2), 16)["counts"]
    assert (counts > 256).sum() >= 2 and ((counts > 0) & (counts <= 256)).sum() >= 2, counts


@pytest.mark.gpu
def test_concurrent_layers_on_distinct_workspaces():
    ls = layers()
    # each layer alone, on the default stream
    ref = []
    for lay in ls:
        o = lay.empty_out()
        lay.run(o)
        ref.append(o)
    torch.cuda.synchronize()
    for lay in ls:
        st, detail = moe.get_device_status(lay.ws)
        assert st == moe.MOE_OK, (lay.name, moe.status_string(st), detail)

    # every layer from its own thread, STEPS forward passes each on its own stream, all at once
    outs = [[lay.empty_out() for _ in range(STEPS)] for lay in ls]
    streams = [torch.cuda.Stream(device=DEV) for _ in ls]
    torch.cuda.synchronize()
    start = threading.Barrier(len(ls))
    errors = []

    def worker(i):
        try:
            start.wait(timeout=60)
            for o in outs[i]:
                ls[i].run(o, stream=streams[i])
            streams[i].synchronize()
        except Exception as e:  # reported by the main thread
            errors.append((ls[i].name, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(ls))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads), "a worker thread did not finish"
    assert not errors, errors
    torch.cuda.synchronize()
    for i, lay in enumerate(ls):
        st, detail = moe.get_device_status(lay.ws)
        assert st == moe.MOE_OK, (lay.name, moe.status_string(st), detail)
        want = ref[i].view(torch.int16 if ref[i].dtype == torch.bfloat16 else torch.int32)
        for s, o in enumerate(outs[i]):
            got = o.view(want.dtype)
            assert torch.equal(got, want), (lay.name, s, int((got != want).sum()))
    # the outputs are real results, not untouched buffers
    for r in ref:
        assert float(r.float().abs().sum()) > 0 and np.isfinite(float(r.float().sum()))


def first_call_in_fresh_thread(fn):
    """Runs fn() as the first CUDA work of a new host thread (no context is current on it yet)."""
    errors = []

    def w():
        try:
            fn()
        except Exception as e:  # reported by the caller
            errors.append(repr(e))

    t = threading.Thread(target=w)
    t.start()
    t.join(timeout=120)
    assert not t.is_alive(), "the thread did not finish"
    return errors


@pytest.mark.gpu
@pytest.mark.parametrize("entry", ["router", "up_pair", "up_tc", "up_stream", "up_int4", "forward"])
def test_first_cuda_work_of_a_fresh_thread(entry):
    """Each entry point that builds tensor maps, called as a new host thread's first CUDA work (the
    stream passed explicitly and the outputs allocated beforehand, so that nothing else binds a
    context first), gives the same result as on the main thread."""
    bf16 = ig.DTYPE_BF16
    decode = entry in ("up_stream", "up_int4")
    c = (make_case(T=4, d=512, F=512, E=16, k=2, dt=bf16) if decode
         else make_case(T=2048, d=256, F=512, E=16, k=2, dt=bf16, bias_scale=0.6))
    T, d, F, E, k, A = c.T, c.d, c.F, c.E, c.k, c.A
    ws = workspace_for(c)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    gate = torch.empty((T, k), dtype=torch.float32, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(A, dtype=torch.int32, device=DEV)
    row_of = torch.empty((T, k), dtype=torch.int32, device=DEV)
    row_gate = torch.empty(A, dtype=torch.float32, device=DEV)
    x_perm = torch.empty((A, d), dtype=torch.bfloat16, device=DEV)
    moe.router_topk(c.x, c.w_r, c.b_r, T, d, E, k, bf16, idx, gate)
    moe.dispatch(c.x, idx, gate, T, d, E, k, bf16, counts, offsets, perm, row_of, row_gate, x_perm, ws)
    q1 = moe.quantize(c.w1, 4) if entry == "up_int4" else None
    path = {"up_pair": moe.PATH_TENSOR_T, "up_tc": moe.PATH_TENSOR, "up_stream": moe.PATH_STREAM}.get(entry)

    def call(outs, stream):
        if entry == "router":
            moe.router_topk(c.x, c.w_r, c.b_r, T, d, E, k, bf16, outs[0], outs[1], stream=stream)
        elif entry == "up_int4":
            moe.expert_up_q(x_perm, q1[0], q1[1], offsets, T, d, F, E, k, 4, outs[0], stream=stream)
        elif entry == "forward":
            moe.forward(c.x, c.w_r, c.b_r, c.w1, c.w2, T, d, F, E, k, bf16, outs[0], ws, stream=stream)
        else:
            moe.expert_up(x_perm, c.w1, offsets, T, d, F, E, k, bf16, outs[0], ws, path=path, stream=stream)

    def new_outs():
        if entry == "router":
            return [torch.empty((T, k), dtype=torch.int32, device=DEV),
                    torch.empty((T, k), dtype=torch.float32, device=DEV)]
        if entry == "forward":
            return [torch.empty((T, d), dtype=torch.bfloat16, device=DEV)]
        return [torch.empty((A, F), dtype=torch.bfloat16, device=DEV)]

    ref = new_outs()
    call(ref, None)
    torch.cuda.synchronize()
    got = new_outs()
    stream = torch.cuda.Stream(device=DEV)
    torch.cuda.synchronize()
    errors = first_call_in_fresh_thread(lambda: call(got, stream))
    assert not errors, errors
    torch.cuda.synchronize()
    assert moe.get_device_status(ws)[0] == moe.MOE_OK
    for r, g in zip(ref, got):
        assert torch.equal(r.view(torch.int16) if r.dtype == torch.bfloat16 else r,
                           g.view(torch.int16) if g.dtype == torch.bfloat16 else g), entry

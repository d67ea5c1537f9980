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

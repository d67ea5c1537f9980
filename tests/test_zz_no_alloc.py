"""moe_dispatch_noalloc: dispatch for callers that cannot give the library device scratch memory.

Such callers (a plugin that its host framework hands only input and output buffers,
or a loop that must not call cudaMalloc because it can block and synchronise the
device) use this entry point; its count tables live in a fixed per-GPU array inside
the library. These tests call it through the C ABI and check that it returns
exactly what moe_dispatch returns with a workspace and what the oracle's dispatch
returns (indices and copies are compared bit for bit, as for every dispatch test), on
two calls in a row of different sizes (the array keeps the first call's contents), at
exactly its size limit, and that sizes beyond its fixed array are refused before
anything runs.

This file sorts last so that a run stopping at the first failure has run every
other test first.
"""
import numpy as np
import pytest

import sparse_mixture_experts_moe_gb300 as moe
from sparse_mixture_experts_moe_gb300 import _lib

FAKE = 1 << 20  # a non-null, 16-byte aligned address that is never dereferenced


def test_noalloc_refuses_sizes_beyond_its_array_without_gpu():
    lib = _lib.lib()
    args = (FAKE, FAKE, FAKE)
    outs = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)
    # ceil(T*k/256) * E must stay within 131072
    assert lib.moe_dispatch_noalloc(*args, 131073, 128, 128, 2, 1, *outs, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_noalloc(*args, 16385, 128, 1024, 2, 1, *outs, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_noalloc(*args, 64, 12, 8, 2, 1, *outs, None) == moe.MOE_ERR_INVALID_ARG  # d % 8


def _dispatch_both(c, idx, gate, torch):
    from moe_cases import torch_dtype, workspace_for
    dev = c.x.device
    A, E = c.A, c.E

    def bufs():
        return dict(counts=torch.full((E,), -7, dtype=torch.int32, device=dev),
                    offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
                    perm_token=torch.full((A,), -7, dtype=torch.int32, device=dev),
                    row_of=torch.full((c.T, c.k), -7, dtype=torch.int32, device=dev),
                    row_gate=torch.full((A,), -7.0, dtype=torch.float32, device=dev),
                    x_perm=torch.zeros((A, c.d), dtype=torch_dtype(c.dt), device=dev))
    ti = torch.from_numpy(idx.astype(np.int32)).to(dev)
    tg = torch.from_numpy(gate.astype(np.float32)).to(dev)
    ref = bufs()
    ws = workspace_for(c)
    moe.dispatch(c.x, ti, tg, c.T, c.d, E, c.k, c.dt, ref["counts"], ref["offsets"], ref["perm_token"],
                 ref["row_of"], ref["row_gate"], ref["x_perm"], ws)
    got = bufs()
    moe.dispatch_noalloc(c.x, ti, tg, c.T, c.d, E, c.k, c.dt, got["counts"], got["offsets"], got["perm_token"],
                         got["row_of"], got["row_gate"], got["x_perm"])
    torch.cuda.synchronize()
    return ref, got


def _check_case(cfg, torch):
    import oracle
    from moe_cases import make_case
    c = make_case(redraw=False, **cfg)
    logits = oracle.router_logits(c.x64, c.wr64, c.br64)
    idx = oracle.topk_select(logits, c.k)
    gate = oracle.gates_of(oracle.softmax(logits), idx)
    ref, got = _dispatch_both(c, idx, gate, torch)
    for name in ["counts", "offsets", "perm_token", "row_of", "row_gate"]:
        assert torch.equal(ref[name], got[name]), name
    bits = torch.int16 if c.dt == moe.MOE_DTYPE_BF16 else torch.int32
    assert torch.equal(ref["x_perm"].view(bits), got["x_perm"].view(bits))
    assert int(got["offsets"][-1]) == c.A
    # and directly against the oracle's dispatch
    want = oracle.dispatch(idx, c.E, gate.astype(np.float32))
    for name in ["counts", "offsets", "perm_token", "row_of"]:
        assert np.array_equal(got[name].cpu().numpy(), want[name]), name
    assert np.array_equal(got["row_gate"].cpu().numpy(), want["row_gate"].astype(np.float32))
    perm = torch.from_numpy(want["perm_token"]).to(c.x.device)
    assert torch.equal(got["x_perm"].view(bits), c.x[perm].view(bits))


@pytest.mark.gpu
def test_noalloc_matches_dispatch_on_two_calls_in_a_row():
    import torch
    # a larger call that fills more of the shared array, then a smaller one that reuses it
    for cfg in [dict(T=3000, d=64, F=64, E=128, k=2, dt=moe.MOE_DTYPE_BF16),
                dict(T=257, d=40, F=64, E=16, k=3, dt=moe.MOE_DTYPE_F32)]:
        _check_case(cfg, torch)


@pytest.mark.gpu
def test_noalloc_at_its_size_limit():
    """ceil(T*k/256) * E == 131072 exactly (T*k = 262144, E = 128): the tables fill the whole array."""
    import torch
    _check_case(dict(T=131072, d=8, F=8, E=128, k=2, dt=moe.MOE_DTYPE_BF16), torch)

"""GB300 (sm_103a) sparse top-k Mixture-of-Experts FFN layer, forward pass.

The layer runs in hand-written CUDA kernels behind the C ABI of include/moe.h
(libmoe.so, built in-tree). PyTorch only provides device memory and streams.

    layer = MoELayer(w_r, w1, w2, k=2)          # weights: CUDA tensors, bf16 or fp32
    out = layer(x)                              # x: [T, d] CUDA tensor

Weights layout: w_r [d, E], w1 [E, d, d_ff], w2 [E, d_ff, d], optional fp32 router bias b_r [E].
"""
from __future__ import annotations

from typing import Optional

from . import _lib
from ._lib import (  # noqa: F401
    MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_DEVICE_CHECK, MOE_ERR_DEVICE_TIMEOUT,
    GATES_RENORMALISE, CAPACITY_REROUTE, MOE_DTYPE_F32, MOE_DTYPE_BF16, PATH_AUTO, PATH_TENSOR, PATH_STREAM, PATH_SIMT, PATH_TENSOR_PAIR, PATH_TENSOR_T,
    MoeError,
    ForwardGraph, GraphCapture, ffn_path, forward_launches, CapturedGraph, qweight_bytes, qscale_bytes,
    quantize_weights, quantize,
    expert_up_q, expert_down_q, forward_q, router_topk, router_topk_stats, router_stats_len, dispatch, dispatch_noalloc, dispatch_reroute, capacity, expert_up, expert_down, grouped_ffn, combine, forward, workspace_bytes, workspace_init,
    get_device_status, status_string, selftest_wait_timeout, lib,
)


class MoELayer:
    """Holds the layer's weights and a reusable workspace; calling it runs moe_forward on the current stream."""

    def __init__(self, w_r, w1, w2, k: int = 2, b_r=None, path: int = PATH_AUTO, renormalise: bool = False,
                 capacity_factor: Optional[float] = None, weight_bits: Optional[int] = None):
        """capacity_factor: None for no expert capacity, else each call keeps at most
        ceil(T * k / E * capacity_factor) assignments per expert (the later ones are dropped).
        weight_bits: None keeps w1 / w2 as given; 4 or 8 quantises them once, here, to 64 x 64-block
        INT4 / INT8 codes (moe_quantize_weights) that every call streams instead (bf16 layers)."""
        import torch
        if not (w_r.is_cuda and w1.is_cuda and w2.is_cuda):
            raise ValueError("MoELayer: weights must be CUDA tensors")
        self.d, self.E = int(w_r.shape[0]), int(w_r.shape[1])
        self.F = int(w1.shape[2])
        if tuple(w1.shape) != (self.E, self.d, self.F) or tuple(w2.shape) != (self.E, self.F, self.d):
            raise ValueError("MoELayer: expected w1 [E, d, F] and w2 [E, F, d]")
        if not (w_r.dtype == w1.dtype == w2.dtype):
            raise ValueError("MoELayer: w_r, w1 and w2 must have one dtype")
        if b_r is not None and tuple(b_r.shape) != (self.E,):
            raise ValueError("MoELayer: expected b_r [E]")
        self.k = int(k)
        self.dt = _lib.dtype_code(w1)
        self.w_r, self.w1, self.w2 = w_r.contiguous(), w1.contiguous(), w2.contiguous()
        self.b_r = None if b_r is None else b_r.to(torch.float32).contiguous()
        self.path = path
        self.renormalise = renormalise
        self.capacity_factor = capacity_factor
        self.weight_bits = weight_bits
        self.q1 = self.q2 = None
        if weight_bits is not None:
            if self.dt != MOE_DTYPE_BF16:
                raise ValueError("MoELayer: quantised expert weights need a bf16 layer")
            self.q1 = quantize(self.w1, weight_bits)
            self.q2 = quantize(self.w2, weight_bits)
        self._ws = None
        self._ws_T = -1

    def _check_io(self, x, out):
        """x [T, d] in the weights' dtype, and out (if given) [T, d]: any other shape would be read or
        written as if it were one."""
        if x.dim() != 2 or int(x.shape[1]) != self.d or x.dtype != self.w1.dtype:
            raise ValueError(f"MoELayer: expected x [T, {self.d}] in {self.w1.dtype}, got {tuple(x.shape)} "
                             f"in {x.dtype}")
        if out is not None and tuple(out.shape) != tuple(x.shape):
            raise ValueError(f"MoELayer: expected out {tuple(x.shape)}, got {tuple(out.shape)}")

    def workspace(self, T: int):
        import torch
        if self._ws is None or T > self._ws_T:
            n = workspace_bytes(T, self.d, self.F, self.E, self.k, self.dt)
            if n == 0:
                raise MoeError(MOE_ERR_INVALID_ARG, "moe_workspace_bytes")
            self._ws = torch.empty(n, dtype=torch.uint8, device=self.w1.device)
            workspace_init(self._ws)
            self._ws_T = T
        return self._ws

    def __call__(self, x, out: Optional["object"] = None, topk_idx=None, topk_gate=None, counts=None,
                 out_dtype=None, router_stats=None):
        """Forward pass of x [T, d]; the output is in x's dtype unless out / out_dtype say otherwise.
        router_stats: optional float32 device tensor of router_stats_len(E) for the routing statistics."""
        import torch
        self._check_io(x, out)
        T = int(x.shape[0])
        if out is None:
            out = torch.empty(x.shape, dtype=out_dtype or x.dtype, device=x.device)
        cap = 0 if self.capacity_factor is None else capacity(T, self.k, self.E, self.capacity_factor)
        if cap < 0:
            raise MoeError(MOE_ERR_INVALID_ARG, "capacity_factor")
        self._run(x, out, T, cap, topk_idx, topk_gate, counts, router_stats, None)
        return out

    def _run(self, x, out, T, cap, topk_idx, topk_gate, counts, router_stats, stream):
        if self.weight_bits is not None:
            forward_q(x, self.w_r, self.b_r, self.q1, self.q2, T, self.d, self.F, self.E, self.k, self.weight_bits,
                      out, self.workspace(T), topk_idx=topk_idx, topk_gate=topk_gate, counts=counts,
                      out_dt=_lib.dtype_code(out), renormalise=self.renormalise, capacity=cap,
                      router_stats=router_stats, stream=stream)
        else:
            forward(x, self.w_r, self.b_r, self.w1, self.w2, T, self.d, self.F, self.E, self.k, self.dt, out,
                    self.workspace(T), topk_idx=topk_idx, topk_gate=topk_gate, counts=counts, path=self.path,
                    out_dt=_lib.dtype_code(out), renormalise=self.renormalise, capacity=cap,
                    router_stats=router_stats, stream=stream)

    def graph(self, x, out, topk_idx=None, topk_gate=None, counts=None, router_stats=None) -> CapturedGraph:
        """A CUDA graph of this layer on these buffers: graph.launch() reruns the layer on the current
        contents of x and writes out (one host call per step)."""
        self._check_io(x, out)
        T = int(x.shape[0])
        cap = 0 if self.capacity_factor is None else capacity(T, self.k, self.E, self.capacity_factor)
        if cap < 0:
            raise MoeError(MOE_ERR_INVALID_ARG, "capacity_factor")
        ws = self.workspace(T)
        keep = (x, out, ws, topk_idx, topk_gate, counts, router_stats, self.w_r, self.b_r, self.w1, self.w2,
                self.q1, self.q2)
        with GraphCapture(keep=keep) as cap_:
            self._run(x, out, T, cap, topk_idx, topk_gate, counts, router_stats, cap_.stream)
        return cap_.graph

    def device_status(self):
        """(status, detail) of the first device-side error since the last call; synchronises."""
        return get_device_status(self._ws) if self._ws is not None else (MOE_OK, 0)

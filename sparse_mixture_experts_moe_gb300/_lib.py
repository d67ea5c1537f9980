"""ctypes binding of libmoe.so: the C ABI in include/moe.h, one Python function per entry point.

Argument marshalling only: tensors are passed as device pointers, streams as
cudaStream_t handles. Every step of the layer runs in the library's CUDA kernels;
there is no other implementation to fall back on, and a missing library raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_DEVICE_CHECK = 4
MOE_ERR_DEVICE_TIMEOUT = 5

MOE_DTYPE_F32 = 0
MOE_DTYPE_BF16 = 1

PATH_AUTO, PATH_TENSOR, PATH_STREAM, PATH_SIMT, PATH_TENSOR_PAIR, PATH_TENSOR_T = 0, 1, 2, 3, 4, 5
GATES_RENORMALISE = 1
CAPACITY_REROUTE = 2

_p = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t

# name -> argument types (all return int moe_status unless listed in _RESTYPES)
SIGNATURES = {
    "moe_router_topk": [_p, _p, _p, _i, _i, _i, _i, _i, _p, _p, _p],
    "moe_router_topk_ex": [_p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p, _p],
    "moe_dispatch": [_p, _p, _p, _i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _sz, _p],
    "moe_dispatch_ex": [_p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _sz, _p],
    "moe_capacity": [_i, _i, _i, ctypes.c_double],
    "moe_ffn_path": [_i, _i, _i, _i, _i],
    "moe_forward_launches": [_i, _i, _i, _i, _i, _i, _i, _i],
    "moe_dispatch_noalloc": [_p, _p, _p, _i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p],
    "moe_dispatch_reroute": [_p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _p, _p, _sz, _p],
    "moe_expert_up": [_p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p, _sz, _p],
    "moe_expert_up_ex": [_p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _p, _p, _sz, _p],
    "moe_expert_down": [_p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p, _sz, _p],
    "moe_expert_down_ex": [_p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _p, _p, _sz, _p],
    "moe_grouped_ffn": [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p, _sz, _p],
    "moe_grouped_ffn_ex": [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _p, _p, _sz, _p],
    "moe_combine": [_p, _p, _i, _i, _i, _i, _p, _p],
    "moe_forward": [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _sz, _p],
    "moe_forward_ex": [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _sz, _p],
    "moe_forward_graph_create": [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p,
                                 _sz, _p],
    "moe_graph_launch": [_p, _p],
    "moe_graph_capture_begin": [_p],
    "moe_graph_capture_end": [_p, _p],
    "moe_qweight_bytes": [_i, _i, _i, _i],
    "moe_qscale_bytes": [_i, _i, _i],
    "moe_quantize_weights": [_p, _i, _i, _i, _i, _i, _p, _p, _p],
    "moe_expert_up_q": [_p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p],
    "moe_expert_down_q": [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p],
    "moe_forward_q": [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p,
                      _sz, _p],
    "moe_graph_destroy": [_p],
    "moe_router_topk_stats": [_p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p, _sz, _p],
    "moe_workspace_bytes": [_i, _i, _i, _i, _i, _i],
    "moe_workspace_init": [_p, _sz, _p],
    "moe_get_device_status": [_p, _p, _p],
    "moe_status_string": [_i],
    "moe_selftest_wait_timeout": [_p, _sz, _i, _p],
}
_RESTYPES = {"moe_workspace_bytes": ctypes.c_size_t, "moe_status_string": ctypes.c_char_p,
             "moe_qweight_bytes": ctypes.c_size_t, "moe_qscale_bytes": ctypes.c_size_t}

_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(there is no fallback implementation)")
        l = ctypes.CDLL(LIB_PATH)
        for name, args in SIGNATURES.items():
            fn = getattr(l, name)
            fn.argtypes = args
            fn.restype = _RESTYPES.get(name, ctypes.c_int)
        _LIB = l
    return _LIB


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def _ptr(t) -> Optional[int]:
    """A tensor argument's device address. The kernels dereference it on the GPU and read it as dense
    row-major data, so a host tensor (its address would fault on the device) or a strided view (it
    would be read as if dense) is refused here. Integers pass through as raw addresses."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError(f"moe: tensor arguments must be CUDA tensors (got one on {t.device})")
    if not t.is_contiguous():
        raise ValueError("moe: tensor arguments must be contiguous")
    return t.data_ptr()


def _esize(dt) -> int:
    """Bytes per element of the call's data type (an invalid code is left to the library to reject)."""
    return 2 if dt == MOE_DTYPE_BF16 else 4


def _fits(t, n, esize, name, typed=False):
    """Refuses a tensor with fewer bytes than n elements of esize bytes, which the kernels would read or
    write past, and, for the layer's data in the call's dtype (typed), a tensor whose elements have
    another size. None and raw integer addresses pass (the library checks those it needs)."""
    if t is None or isinstance(t, int):
        return
    if typed and t.element_size() != esize:
        raise ValueError(f"moe: {name} has {t.element_size()}-byte elements; the call's dtype has {esize}")
    if n > 0 and t.numel() * t.element_size() < n * esize:
        raise ValueError(f"moe: {name} holds {t.numel() * t.element_size()} bytes; the call needs {n * esize}")


def _routing_fits(T, E, k, topk_idx, topk_gate, counts=None, router_stats=None):
    _fits(topk_idx, T * k, 4, "topk_idx")
    _fits(topk_gate, T * k, 4, "topk_gate")
    _fits(counts, E, 4, "counts")
    _fits(router_stats, 2 * E + 2, 4, "router_stats")


def _dispatch_fits(T, d, E, k, dt, counts, offsets, perm_token, row_of, row_gate, x_perm):
    A = T * k
    _fits(counts, E, 4, "counts")
    _fits(offsets, E + 1, 4, "offsets")
    _fits(perm_token, A, 4, "perm_token")
    _fits(row_of, A, 4, "row_of")
    _fits(row_gate, A, 4, "row_gate")
    _fits(x_perm, A * d, _esize(dt), "x_perm", typed=True)


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str) -> int:
    if rc != MOE_OK:
        raise MoeError(rc, where)
    return rc


def dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return MOE_DTYPE_BF16
    if t.dtype == torch.float32:
        return MOE_DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


# ----------------------------------------------------------------------------- entry points

def workspace_bytes(T, d, F, E, k, dt) -> int:
    return int(lib().moe_workspace_bytes(T, d, F, E, k, dt))


def workspace_init(ws, stream=None, check=True) -> int:
    rc = lib().moe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    return _check(rc, "moe_workspace_init") if check else rc


def get_device_status(ws, stream=None):
    """(status, detail) of the first device-side error recorded in ws; clears it."""
    detail = ctypes.c_int32(0)
    rc = lib().moe_get_device_status(_ptr(ws), ctypes.addressof(detail), _stream(stream))
    return rc, detail.value


def router_topk(x, w_r, b_r, T, d, E, k, dt, topk_idx, topk_gate, renormalise=False, stream=None, check=True):
    """renormalise: gates are the softmax over the k chosen logits (GATES_RENORMALISE)."""
    _fits(x, T * d, _esize(dt), "x", typed=True)
    _fits(w_r, d * E, _esize(dt), "w_r", typed=True)
    _fits(b_r, E, 4, "b_r")
    _routing_fits(T, E, k, topk_idx, topk_gate)
    rc = lib().moe_router_topk_ex(_ptr(x), _ptr(w_r), _ptr(b_r), T, d, E, k, dt,
                                  GATES_RENORMALISE if renormalise else 0, _ptr(topk_idx), _ptr(topk_gate),
                                  _stream(stream))
    return _check(rc, "moe_router_topk") if check else rc


def router_stats_len(E) -> int:
    """Floats of the routing-statistics output: soft load [E], assignment share [E], balance, entropy."""
    return 2 * E + 2


def router_topk_stats(x, w_r, b_r, T, d, E, k, dt, topk_idx, topk_gate, stats, ws, renormalise=False, stream=None,
                      check=True):
    """moe_router_topk_stats: the router plus the batch's routing statistics in `stats`."""
    _fits(x, T * d, _esize(dt), "x", typed=True)
    _fits(w_r, d * E, _esize(dt), "w_r", typed=True)
    _fits(b_r, E, 4, "b_r")
    _routing_fits(T, E, k, topk_idx, topk_gate, router_stats=stats)
    rc = lib().moe_router_topk_stats(_ptr(x), _ptr(w_r), _ptr(b_r), T, d, E, k, dt,
                                     GATES_RENORMALISE if renormalise else 0, _ptr(topk_idx), _ptr(topk_gate),
                                     _ptr(stats), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    return _check(rc, "moe_router_topk_stats") if check else rc


def ffn_path(T, k, E, N, dt) -> int:
    """The kernel family (PATH_*) AUTO runs for an expert GEMM with N output columns."""
    return int(lib().moe_ffn_path(T, k, E, N, dt))


def forward_launches(T, d, F, E, k, dt, path=PATH_AUTO, router_stats=False) -> int:
    """Kernel launches of one forward call with these arguments (moe_forward_launches); host only."""
    return int(lib().moe_forward_launches(T, d, F, E, k, dt, path, 1 if router_stats else 0))


def capacity(T, k, E, cf) -> int:
    """ceil(T*k/E*cf), the expert capacity moe_dispatch_ex / moe_forward_ex take."""
    return int(lib().moe_capacity(T, k, E, float(cf)))


def dispatch(x, topk_idx, topk_gate, T, d, E, k, dt, counts, offsets, perm_token, row_of, row_gate, x_perm, ws,
             capacity=0, stream=None, check=True):
    """capacity > 0: each expert keeps its first `capacity` assignments (moe_dispatch_ex)."""
    _fits(x, T * d, _esize(dt), "x", typed=True)
    _routing_fits(T, E, k, topk_idx, topk_gate)
    _dispatch_fits(T, d, E, k, dt, counts, offsets, perm_token, row_of, row_gate, x_perm)
    rc = lib().moe_dispatch_ex(_ptr(x), _ptr(topk_idx), _ptr(topk_gate), T, d, E, k, dt, int(capacity),
                               _ptr(counts), _ptr(offsets), _ptr(perm_token), _ptr(row_of), _ptr(row_gate),
                               _ptr(x_perm), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    return _check(rc, "moe_dispatch") if check else rc


def dispatch_reroute(x, rank_idx, rank_gate, T, d, E, k, R, dt, capacity, final_idx, final_gate, counts, offsets,
                     perm_token, row_of, row_gate, x_perm, ws, stream=None, check=True):
    """moe_dispatch_reroute: an assignment that meets a full expert takes the next entry of its token's
    ranking rank_idx[t, k:] with room, or is dropped (final_idx -1)."""
    _fits(x, T * d, _esize(dt), "x", typed=True)
    _fits(rank_idx, T * R, 4, "rank_idx")
    _fits(rank_gate, T * R, 4, "rank_gate")
    _routing_fits(T, E, k, final_idx, final_gate)
    _dispatch_fits(T, d, E, k, dt, counts, offsets, perm_token, row_of, row_gate, x_perm)
    rc = lib().moe_dispatch_reroute(_ptr(x), _ptr(rank_idx), _ptr(rank_gate), T, d, E, k, R, dt, int(capacity),
                                    _ptr(final_idx), _ptr(final_gate), _ptr(counts), _ptr(offsets), _ptr(perm_token),
                                    _ptr(row_of), _ptr(row_gate), _ptr(x_perm), _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream))
    return _check(rc, "moe_dispatch_reroute") if check else rc


def _flags(renormalise, reroute):
    return (GATES_RENORMALISE if renormalise else 0) | (CAPACITY_REROUTE if reroute else 0)


def dispatch_noalloc(x, topk_idx, topk_gate, T, d, E, k, dt, counts, offsets, perm_token, row_of, row_gate,
                     x_perm, stream=None, check=True):
    """moe_dispatch without a workspace: the count tables live in the library's fixed per-GPU array."""
    _fits(x, T * d, _esize(dt), "x", typed=True)
    _routing_fits(T, E, k, topk_idx, topk_gate)
    _dispatch_fits(T, d, E, k, dt, counts, offsets, perm_token, row_of, row_gate, x_perm)
    rc = lib().moe_dispatch_noalloc(_ptr(x), _ptr(topk_idx), _ptr(topk_gate), T, d, E, k, dt, _ptr(counts),
                                    _ptr(offsets), _ptr(perm_token), _ptr(row_of), _ptr(row_gate), _ptr(x_perm),
                                    _stream(stream))
    return _check(rc, "moe_dispatch_noalloc") if check else rc


def expert_up(x_perm, w1, offsets, T, d, F, E, k, dt, h, ws, path=PATH_AUTO, stream=None, check=True):
    _fits(x_perm, T * k * d, _esize(dt), "x_perm", typed=True)
    _fits(w1, E * d * F, _esize(dt), "w1", typed=True)
    _fits(offsets, E + 1, 4, "offsets")
    _fits(h, T * k * F, _esize(dt), "h", typed=True)
    rc = lib().moe_expert_up_ex(_ptr(x_perm), _ptr(w1), _ptr(offsets), T, d, F, E, k, dt, path, _ptr(h), _ptr(ws),
                                ws.numel() * ws.element_size(), _stream(stream))
    return _check(rc, "moe_expert_up") if check else rc


def expert_down(h, w2, offsets, row_gate, T, d, F, E, k, dt, y_perm, ws, path=PATH_AUTO, stream=None, check=True):
    _fits(h, T * k * F, _esize(dt), "h", typed=True)
    _fits(w2, E * F * d, _esize(dt), "w2", typed=True)
    _fits(offsets, E + 1, 4, "offsets")
    _fits(row_gate, T * k, 4, "row_gate")
    _fits(y_perm, T * k * d, 4, "y_perm", typed=True)
    rc = lib().moe_expert_down_ex(_ptr(h), _ptr(w2), _ptr(offsets), _ptr(row_gate), T, d, F, E, k, dt, path,
                                  _ptr(y_perm), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    return _check(rc, "moe_expert_down") if check else rc


def grouped_ffn(x_perm, w1, w2, offsets, row_gate, T, d, F, E, k, dt, y_perm, ws, path=PATH_AUTO, stream=None,
                check=True):
    _fits(x_perm, T * k * d, _esize(dt), "x_perm", typed=True)
    _fits(w1, E * d * F, _esize(dt), "w1", typed=True)
    _fits(w2, E * F * d, _esize(dt), "w2", typed=True)
    _fits(offsets, E + 1, 4, "offsets")
    _fits(row_gate, T * k, 4, "row_gate")
    _fits(y_perm, T * k * d, 4, "y_perm", typed=True)
    rc = lib().moe_grouped_ffn_ex(_ptr(x_perm), _ptr(w1), _ptr(w2), _ptr(offsets), _ptr(row_gate), T, d, F, E, k,
                                  dt, path, _ptr(y_perm), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    return _check(rc, "moe_grouped_ffn") if check else rc


def combine(y_perm, row_of, T, d, k, dt, out, stream=None, check=True):
    _fits(y_perm, T * k * d, 4, "y_perm", typed=True)
    _fits(row_of, T * k, 4, "row_of")
    _fits(out, T * d, _esize(dt), "out", typed=True)
    rc = lib().moe_combine(_ptr(y_perm), _ptr(row_of), T, d, k, dt, _ptr(out), _stream(stream))
    return _check(rc, "moe_combine") if check else rc


def _layer_fits(x, w_r, b_r, w1, w2, T, d, F, E, k, dt, out, out_dt, topk_idx, topk_gate, counts, router_stats):
    _fits(x, T * d, _esize(dt), "x", typed=True)
    _fits(w_r, d * E, _esize(dt), "w_r", typed=True)
    _fits(b_r, E, 4, "b_r")
    _fits(w1, E * d * F, _esize(dt), "w1", typed=True)
    _fits(w2, E * F * d, _esize(dt), "w2", typed=True)
    _fits(out, T * d, _esize(out_dt), "out", typed=True)
    _routing_fits(T, E, k, topk_idx, topk_gate, counts, router_stats)


def forward(x, w_r, b_r, w1, w2, T, d, F, E, k, dt, out, ws, topk_idx=None, topk_gate=None, counts=None,
            path=PATH_AUTO, out_dt=None, renormalise=False, capacity=0, router_stats=None, stream=None, check=True,
            reroute=False):
    """out_dt: element type of `out` (default: dt); renormalise: GATES_RENORMALISE; capacity: as dispatch;
    reroute: CAPACITY_REROUTE (assignments past capacity go to the token's next-best expert with room);
    router_stats: None or a float32 device tensor of router_stats_len(E) (as router_topk_stats)."""
    out_dt = dt if out_dt is None else out_dt
    _layer_fits(x, w_r, b_r, w1, w2, T, d, F, E, k, dt, out, out_dt, topk_idx, topk_gate, counts, router_stats)
    rc = lib().moe_forward_ex(_ptr(x), _ptr(w_r), _ptr(b_r), _ptr(w1), _ptr(w2), T, d, F, E, k, dt, out_dt, path,
                              _flags(renormalise, reroute), int(capacity), _ptr(out),
                              _ptr(topk_idx), _ptr(topk_gate), _ptr(counts), _ptr(router_stats), _ptr(ws),
                              ws.numel() * ws.element_size(), _stream(stream))
    return _check(rc, "moe_forward") if check else rc


class ForwardGraph:
    """The layer's kernels for one fixed set of buffers, captured once as a CUDA graph
    (moe_forward_graph_create); launch() replays the whole layer with one host call. The tensors
    passed at creation are kept referenced so that their memory outlives the graph."""

    def __init__(self, x, w_r, b_r, w1, w2, T, d, F, E, k, dt, out, ws, topk_idx=None, topk_gate=None, counts=None,
                 path=PATH_AUTO, out_dt=None, renormalise=False, capacity=0, router_stats=None):
        out_dt = dt if out_dt is None else out_dt
        _layer_fits(x, w_r, b_r, w1, w2, T, d, F, E, k, dt, out, out_dt, topk_idx, topk_gate, counts, router_stats)
        self._keep = (x, w_r, b_r, w1, w2, out, ws, topk_idx, topk_gate, counts, router_stats)
        h = ctypes.c_void_p()
        self._lib = lib()
        rc = self._lib.moe_forward_graph_create(
            _ptr(x), _ptr(w_r), _ptr(b_r), _ptr(w1), _ptr(w2), T, d, F, E, k, dt, out_dt, path,
            GATES_RENORMALISE if renormalise else 0, int(capacity), _ptr(out), _ptr(topk_idx), _ptr(topk_gate),
            _ptr(counts), _ptr(router_stats), _ptr(ws), ws.numel() * ws.element_size(), ctypes.byref(h))
        _check(rc, "moe_forward_graph_create")
        self._h = h

    def launch(self, stream=None):
        return _check(self._lib.moe_graph_launch(self._h, _stream(stream)), "moe_graph_launch")

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value is not None:
            self._lib.moe_graph_destroy(self._h)
        self._h = None

    def __del__(self):
        self.close()


class GraphCapture:
    """Records the moe_* calls made with `cap.stream` inside the with-block into a CUDA graph
    (moe_graph_capture_begin / _end); `cap.graph` then replays them with launch(). Keep the
    tensors those calls used alive while the graph is in use (pass them as keep=...)."""

    def __init__(self, keep=()):
        self._keep = tuple(keep)
        self.stream = None
        self.graph = None

    def __enter__(self):
        cs = ctypes.c_void_p()
        _check(lib().moe_graph_capture_begin(ctypes.byref(cs)), "moe_graph_capture_begin")
        self.stream = cs.value
        return self

    def __exit__(self, exc_type, exc, tb):
        h = ctypes.c_void_p()
        rc = lib().moe_graph_capture_end(self.stream, ctypes.byref(h))
        if exc_type is None:
            _check(rc, "moe_graph_capture_end")
            self.graph = CapturedGraph(h, self._keep)
        elif rc == MOE_OK:
            lib().moe_graph_destroy(h)
        return False


class CapturedGraph:
    def __init__(self, handle, keep):
        self._h = handle
        self._keep = keep
        self._lib = lib()

    def launch(self, stream=None):
        return _check(self._lib.moe_graph_launch(self._h, _stream(stream)), "moe_graph_launch")

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value is not None:
            self._lib.moe_graph_destroy(self._h)
        self._h = None

    def __del__(self):
        self.close()


# ------------------------------------------------------------------ block-quantised weights

def qweight_bytes(K, N, E, bits) -> int:
    return int(lib().moe_qweight_bytes(K, N, E, bits))


def qscale_bytes(K, N, E) -> int:
    return int(lib().moe_qscale_bytes(K, N, E))


def quantize_weights(w, K, N, E, dt, bits, codes, scale_min, stream=None, check=True):
    """w [E, K, N] -> codes (moe_qweight_bytes bytes) and scale_min ([E, K/64, N/64, 2] fp32)."""
    _fits(w, E * K * N, _esize(dt), "w", typed=True)
    _qweights_fits(codes, scale_min, K, N, E, bits, "")
    rc = lib().moe_quantize_weights(_ptr(w), K, N, E, dt, bits, _ptr(codes), _ptr(scale_min), _stream(stream))
    return _check(rc, "moe_quantize_weights") if check else rc


def quantize(w, bits, stream=None):
    """Quantise a device tensor w [E, K, N] (bf16 or fp32); returns (codes uint8, scale_min fp32)."""
    import torch
    E, K, N = (int(v) for v in w.shape)
    nb = qweight_bytes(K, N, E, bits)
    if nb == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_qweight_bytes")
    codes = torch.empty(nb, dtype=torch.uint8, device=w.device)
    sm = torch.empty((E, K // 64, N // 64, 2), dtype=torch.float32, device=w.device)
    quantize_weights(w.contiguous(), K, N, E, dtype_code(w), bits, codes, sm, stream)
    return codes, sm


def _qweights_fits(codes, scale_min, K, N, E, bits, which):
    _fits(codes, qweight_bytes(K, N, E, bits), 1, which + "codes")
    _fits(scale_min, qscale_bytes(K, N, E) // 4, 4, which + "scale_min")


def expert_up_q(x_perm, codes, scale_min, offsets, T, d, F, E, k, bits, h, stream=None, check=True):
    _fits(x_perm, T * k * d, 2, "x_perm", typed=True)
    _qweights_fits(codes, scale_min, d, F, E, bits, "w1 ")
    _fits(offsets, E + 1, 4, "offsets")
    _fits(h, T * k * F, 2, "h", typed=True)
    rc = lib().moe_expert_up_q(_ptr(x_perm), _ptr(codes), _ptr(scale_min), _ptr(offsets), T, d, F, E, k, bits,
                               _ptr(h), _stream(stream))
    return _check(rc, "moe_expert_up_q") if check else rc


def expert_down_q(h, codes, scale_min, offsets, row_gate, T, d, F, E, k, bits, y_perm, stream=None, check=True):
    _fits(h, T * k * F, 2, "h", typed=True)
    _qweights_fits(codes, scale_min, F, d, E, bits, "w2 ")
    _fits(offsets, E + 1, 4, "offsets")
    _fits(row_gate, T * k, 4, "row_gate")
    _fits(y_perm, T * k * d, 4, "y_perm", typed=True)
    rc = lib().moe_expert_down_q(_ptr(h), _ptr(codes), _ptr(scale_min), _ptr(offsets), _ptr(row_gate), T, d, F, E,
                                 k, bits, _ptr(y_perm), _stream(stream))
    return _check(rc, "moe_expert_down_q") if check else rc


def forward_q(x, w_r, b_r, w1q, w2q, T, d, F, E, k, bits, out, ws, topk_idx=None, topk_gate=None, counts=None,
              out_dt=None, renormalise=False, capacity=0, router_stats=None, stream=None, check=True, reroute=False):
    """The layer with block-quantised expert weights; w1q / w2q are (codes, scale_min) pairs."""
    out_dt = MOE_DTYPE_BF16 if out_dt is None else out_dt
    _layer_fits(x, w_r, b_r, None, None, T, d, F, E, k, MOE_DTYPE_BF16, out, out_dt, topk_idx, topk_gate, counts,
                router_stats)
    _qweights_fits(w1q[0], w1q[1], d, F, E, bits, "w1 ")
    _qweights_fits(w2q[0], w2q[1], F, d, E, bits, "w2 ")
    rc = lib().moe_forward_q(_ptr(x), _ptr(w_r), _ptr(b_r), _ptr(w1q[0]), _ptr(w1q[1]), _ptr(w2q[0]),
                             _ptr(w2q[1]), T, d, F, E, k, bits, out_dt, _flags(renormalise, reroute),
                             int(capacity), _ptr(out), _ptr(topk_idx), _ptr(topk_gate), _ptr(counts),
                             _ptr(router_stats), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    return _check(rc, "moe_forward_q") if check else rc


def selftest_wait_timeout(ws, timeout_us, stream=None, check=True):
    rc = lib().moe_selftest_wait_timeout(_ptr(ws), ws.numel() * ws.element_size(), int(timeout_us), _stream(stream))
    return _check(rc, "moe_selftest_wait_timeout") if check else rc

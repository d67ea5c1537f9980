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

PATH_AUTO, PATH_TENSOR, PATH_STREAM, PATH_SIMT, PATH_TENSOR_PAIR = 0, 1, 2, 3, 4
GATES_RENORMALISE = 1

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
    "moe_dispatch_noalloc": [_p, _p, _p, _i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p],
    "moe_expert_up": [_p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p, _sz, _p],
    "moe_expert_up_ex": [_p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _p, _p, _sz, _p],
    "moe_expert_down": [_p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p, _sz, _p],
    "moe_expert_down_ex": [_p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _p, _p, _sz, _p],
    "moe_grouped_ffn": [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p, _sz, _p],
    "moe_grouped_ffn_ex": [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _p, _p, _sz, _p],
    "moe_combine": [_p, _p, _i, _i, _i, _i, _p, _p],
    "moe_forward": [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _sz, _p],
    "moe_forward_ex": [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _sz, _p],
    "moe_router_topk_stats": [_p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p, _sz, _p],
    "moe_workspace_bytes": [_i, _i, _i, _i, _i, _i],
    "moe_workspace_init": [_p, _sz, _p],
    "moe_get_device_status": [_p, _p, _p],
    "moe_status_string": [_i],
    "moe_selftest_wait_timeout": [_p, _sz, _i, _p],
}
_RESTYPES = {"moe_workspace_bytes": ctypes.c_size_t, "moe_status_string": ctypes.c_char_p}

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
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


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
    rc = lib().moe_router_topk_stats(_ptr(x), _ptr(w_r), _ptr(b_r), T, d, E, k, dt,
                                     GATES_RENORMALISE if renormalise else 0, _ptr(topk_idx), _ptr(topk_gate),
                                     _ptr(stats), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    return _check(rc, "moe_router_topk_stats") if check else rc


def capacity(T, k, E, cf) -> int:
    """ceil(T*k/E*cf), the expert capacity moe_dispatch_ex / moe_forward_ex take."""
    return int(lib().moe_capacity(T, k, E, float(cf)))


def dispatch(x, topk_idx, topk_gate, T, d, E, k, dt, counts, offsets, perm_token, row_of, row_gate, x_perm, ws,
             capacity=0, stream=None, check=True):
    """capacity > 0: each expert keeps its first `capacity` assignments (moe_dispatch_ex)."""
    rc = lib().moe_dispatch_ex(_ptr(x), _ptr(topk_idx), _ptr(topk_gate), T, d, E, k, dt, int(capacity),
                               _ptr(counts), _ptr(offsets), _ptr(perm_token), _ptr(row_of), _ptr(row_gate),
                               _ptr(x_perm), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    return _check(rc, "moe_dispatch") if check else rc


def dispatch_noalloc(x, topk_idx, topk_gate, T, d, E, k, dt, counts, offsets, perm_token, row_of, row_gate,
                     x_perm, stream=None, check=True):
    """moe_dispatch without a workspace: the count tables live in the library's fixed per-GPU array."""
    rc = lib().moe_dispatch_noalloc(_ptr(x), _ptr(topk_idx), _ptr(topk_gate), T, d, E, k, dt, _ptr(counts),
                                    _ptr(offsets), _ptr(perm_token), _ptr(row_of), _ptr(row_gate), _ptr(x_perm),
                                    _stream(stream))
    return _check(rc, "moe_dispatch_noalloc") if check else rc


def expert_up(x_perm, w1, offsets, T, d, F, E, k, dt, h, ws, path=PATH_AUTO, stream=None, check=True):
    rc = lib().moe_expert_up_ex(_ptr(x_perm), _ptr(w1), _ptr(offsets), T, d, F, E, k, dt, path, _ptr(h), _ptr(ws),
                                ws.numel() * ws.element_size(), _stream(stream))
    return _check(rc, "moe_expert_up") if check else rc


def expert_down(h, w2, offsets, row_gate, T, d, F, E, k, dt, y_perm, ws, path=PATH_AUTO, stream=None, check=True):
    rc = lib().moe_expert_down_ex(_ptr(h), _ptr(w2), _ptr(offsets), _ptr(row_gate), T, d, F, E, k, dt, path,
                                  _ptr(y_perm), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    return _check(rc, "moe_expert_down") if check else rc


def grouped_ffn(x_perm, w1, w2, offsets, row_gate, T, d, F, E, k, dt, y_perm, ws, path=PATH_AUTO, stream=None,
                check=True):
    rc = lib().moe_grouped_ffn_ex(_ptr(x_perm), _ptr(w1), _ptr(w2), _ptr(offsets), _ptr(row_gate), T, d, F, E, k,
                                  dt, path, _ptr(y_perm), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    return _check(rc, "moe_grouped_ffn") if check else rc


def combine(y_perm, row_of, T, d, k, dt, out, stream=None, check=True):
    rc = lib().moe_combine(_ptr(y_perm), _ptr(row_of), T, d, k, dt, _ptr(out), _stream(stream))
    return _check(rc, "moe_combine") if check else rc


def forward(x, w_r, b_r, w1, w2, T, d, F, E, k, dt, out, ws, topk_idx=None, topk_gate=None, counts=None,
            path=PATH_AUTO, out_dt=None, renormalise=False, capacity=0, router_stats=None, stream=None, check=True):
    """out_dt: element type of `out` (default: dt); renormalise: GATES_RENORMALISE; capacity: as dispatch;
    router_stats: None or a float32 device tensor of router_stats_len(E) (as router_topk_stats)."""
    out_dt = dt if out_dt is None else out_dt
    rc = lib().moe_forward_ex(_ptr(x), _ptr(w_r), _ptr(b_r), _ptr(w1), _ptr(w2), T, d, F, E, k, dt, out_dt, path,
                              GATES_RENORMALISE if renormalise else 0, int(capacity), _ptr(out),
                              _ptr(topk_idx), _ptr(topk_gate), _ptr(counts), _ptr(router_stats), _ptr(ws),
                              ws.numel() * ws.element_size(), _stream(stream))
    return _check(rc, "moe_forward") if check else rc


def selftest_wait_timeout(ws, timeout_us, stream=None, check=True):
    rc = lib().moe_selftest_wait_timeout(_ptr(ws), ws.numel() * ws.element_size(), int(timeout_us), _stream(stream))
    return _check(rc, "moe_selftest_wait_timeout") if check else rc

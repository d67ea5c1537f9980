"""C ABI checks that need no GPU: the library loads, exports every entry point the
header declares, and rejects invalid arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

import sparse_mixture_experts_moe_gb300 as moe
from sparse_mixture_experts_moe_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_layer_calls():
    names = header_functions()
    for required in ["moe_router_topk", "moe_dispatch", "moe_grouped_ffn", "moe_combine", "moe_forward",
                     "moe_expert_up", "moe_expert_down", "moe_workspace_bytes", "moe_get_device_status"]:
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = _lib.lib()
    missing = [n for n in header_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(header_functions()) == set(_lib.SIGNATURES), "binding and header disagree"


def test_status_strings():
    for s in range(6):
        assert moe.status_string(s).startswith("MOE_")


def test_workspace_bytes():
    n = moe.workspace_bytes(4096, 1024, 4096, 16, 2, moe.MOE_DTYPE_BF16)
    A = 8192
    # at least x_perm + h + y_perm
    assert n >= A * 1024 * 2 * 2 + A * 4096 * 2
    assert n % 256 == 0
    assert moe.workspace_bytes(64, 128, 256, 8, 9, moe.MOE_DTYPE_F32) == 0     # k > E
    assert moe.workspace_bytes(64, 130, 256, 8, 2, moe.MOE_DTYPE_F32) == 0     # d % 8
    assert moe.workspace_bytes(64, 128, 256, 1025, 2, moe.MOE_DTYPE_F32) == 0  # E > 1024
    assert moe.workspace_bytes(0, 128, 256, 8, 2, moe.MOE_DTYPE_F32) > 0       # T = 0 is valid


FAKE = 1 << 20  # a non-null, 16-byte aligned address that is never dereferenced


@pytest.mark.parametrize("T,d,E,k,dt", [
    (-1, 128, 8, 2, 0), (64, 0, 8, 2, 0), (64, 12, 8, 2, 0), (64, 128, 8, 0, 0), (64, 128, 8, 9, 0),
    (64, 128, 2, 3, 0), (64, 128, 1025, 2, 0), (64, 128, 8, 2, 7)])
def test_router_rejects_bad_sizes_without_gpu(T, d, E, k, dt):
    rc = _lib.lib().moe_router_topk(FAKE, FAKE, None, T, d, E, k, dt, FAKE, FAKE, None)
    assert rc == moe.MOE_ERR_INVALID_ARG


def test_null_and_misaligned_pointers_rejected_without_gpu():
    lib = _lib.lib()
    assert lib.moe_router_topk(None, FAKE, None, 4, 128, 8, 2, 1, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_router_topk(FAKE + 2, FAKE, None, 4, 128, 8, 2, 1, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(None, FAKE, 4, 128, 2, 1, FAKE, None) == moe.MOE_ERR_INVALID_ARG
    ws_small = 100
    assert lib.moe_forward(FAKE, FAKE, None, FAKE, FAKE, 4, 128, 256, 8, 2, 1, FAKE, None, None, None, FAKE,
                           ws_small, None) == moe.MOE_ERR_INVALID_ARG
    n = moe.workspace_bytes(4, 128, 256, 8, 2, 1)
    assert lib.moe_dispatch(FAKE, FAKE, FAKE, 4, 128, 8, 2, 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 256,
                            None) == moe.MOE_ERR_INVALID_ARG  # workspace too small for the count tables
    assert lib.moe_expert_up_ex(FAKE, FAKE, FAKE, 4, 128, 256, 8, 2, 1, 9, FAKE, FAKE, n,
                                None) == moe.MOE_ERR_INVALID_ARG  # unknown path
    assert lib.moe_selftest_wait_timeout(FAKE, n, 0, None) == moe.MOE_ERR_INVALID_ARG


def test_zero_tokens_is_a_no_op_without_gpu():
    lib = _lib.lib()
    n = moe.workspace_bytes(0, 128, 256, 8, 2, 1)
    assert lib.moe_router_topk(FAKE, FAKE, None, 0, 128, 8, 2, 1, FAKE, FAKE, None) == moe.MOE_OK
    assert lib.moe_combine(FAKE, FAKE, 0, 128, 2, 1, FAKE, None) == moe.MOE_OK
    assert lib.moe_forward(FAKE, FAKE, None, FAKE, FAKE, 0, 128, 256, 8, 2, 1, FAKE, None, None, None, FAKE, n,
                           None) == moe.MOE_OK


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "libmoe.so"))
    monkeypatch.setattr(_lib, "_LIB", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        _lib.lib()


def test_capacity_helper_matches_oracle():
    import oracle
    for T, k, E, cf in [(2048, 2, 128, 2.0), (1000, 2, 16, 1.0), (1000, 2, 16, 1.25), (37, 2, 4, 0.05),
                        (1, 8, 1024, 1.0), (0, 2, 16, 1.0), (65536, 8, 7, 3.3)]:
        assert moe.capacity(T, k, E, cf) == oracle.capacity(T, k, E, cf)
    assert moe.capacity(16, 2, 4, 0.0) == -1
    assert moe.capacity(16, 0, 4, 1.0) == -1


def test_graph_handles_rejected_without_gpu():
    lib = _lib.lib()
    assert lib.moe_graph_launch(None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_graph_destroy(None) == moe.MOE_OK
    assert lib.moe_forward_graph_create(*([None] * 5), 4, 64, 64, 8, 2, 1, 1, 0, 0, 0, *([None] * 6), 0,
                                        None) == moe.MOE_ERR_INVALID_ARG


def test_quantised_sizes_without_gpu():
    lib = _lib.lib()
    assert moe.qweight_bytes(8192, 8192, 128, 4) == 128 * 8192 * 8192 // 2
    assert moe.qweight_bytes(8192, 8192, 128, 8) == 128 * 8192 * 8192
    assert moe.qscale_bytes(1024, 4096, 16) == 16 * 16 * 64 * 8
    assert moe.qweight_bytes(100, 64, 2, 4) == 0 and moe.qweight_bytes(64, 64, 2, 3) == 0
    FAKE = 4096
    assert lib.moe_quantize_weights(FAKE, 64, 64, 1, 1, 5, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_graph_capture_begin(None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_graph_capture_end(None, None) == moe.MOE_ERR_INVALID_ARG


def test_forward_launch_plan_without_gpu():
    """How many kernels one forward call launches, from the library's own decisions."""
    BF16, F32 = moe.MOE_DTYPE_BF16, moe.MOE_DTYPE_F32
    # decode: router + dispatch in one launch, two weight-streaming GEMMs, combine
    assert moe.forward_launches(1, 8192, 8192, 128, 2, BF16) == 4
    assert moe.forward_launches(8, 8192, 8192, 128, 2, BF16) == 4
    # statistics, E % 8 != 0, or a GEMM family other than streaming: the separate router and dispatch
    assert moe.forward_launches(1, 8192, 8192, 128, 2, BF16, router_stats=True) == 5
    assert moe.forward_launches(2, 136, 64, 6, 1, BF16) == 6
    assert moe.forward_launches(1, 1024, 1024, 16, 2, BF16, path=moe.PATH_TENSOR) == 5
    # top-2 with the tensor-core router: the router writes the dispatch histograms
    assert moe.forward_launches(4096, 1024, 4096, 16, 2, BF16) == 5
    assert moe.forward_launches(8192, 4096, 8192, 128, 2, BF16) == 5
    # otherwise six: k != 2, E > 256, fp32
    assert moe.forward_launches(4096, 1024, 4096, 16, 4, BF16) == 6
    assert moe.forward_launches(4096, 1024, 4096, 512, 2, BF16) == 6
    assert moe.forward_launches(64, 128, 256, 8, 2, F32) == 6
    assert moe.forward_launches(0, 128, 256, 8, 2, BF16) == 0
    assert moe.forward_launches(4, 100, 256, 8, 2, BF16) == -1  # d % 8 != 0


def test_reroute_arguments_rejected_without_gpu():
    """moe_dispatch_reroute wants k <= R <= E and a capacity of at least 1; MOE_CAPACITY_REROUTE on the
    layer wants a capacity, the raw gates and no routing statistics; unknown flag bits are refused."""
    lib = _lib.lib()
    n = moe.workspace_bytes(4, 128, 256, 8, 2, 1)
    outs = (FAKE,) * 8
    assert lib.moe_dispatch_reroute(FAKE, FAKE, FAKE, 4, 128, 8, 2, 1, 1, 3, *outs, FAKE, n, None) == \
        moe.MOE_ERR_INVALID_ARG  # R < k
    assert lib.moe_dispatch_reroute(FAKE, FAKE, FAKE, 4, 128, 8, 2, 9, 1, 3, *outs, FAKE, n, None) == \
        moe.MOE_ERR_INVALID_ARG  # R > E
    assert lib.moe_dispatch_reroute(FAKE, FAKE, FAKE, 4, 128, 8, 2, 4, 1, 0, *outs, FAKE, n, None) == \
        moe.MOE_ERR_INVALID_ARG  # no capacity
    assert lib.moe_dispatch_reroute(FAKE, None, FAKE, 4, 128, 8, 2, 4, 1, 3, *outs, FAKE, n, None) == \
        moe.MOE_ERR_INVALID_ARG  # no ranking

    def fwd(flags, capacity, stats=None):
        return lib.moe_forward_ex(FAKE, FAKE, None, FAKE, FAKE, 4, 128, 256, 8, 2, 1, 1, 0, flags, capacity, FAKE,
                                  None, None, None, stats, FAKE, n, None)
    assert fwd(moe.CAPACITY_REROUTE, 0) == moe.MOE_ERR_INVALID_ARG
    assert fwd(moe.CAPACITY_REROUTE | moe.GATES_RENORMALISE, 3) == moe.MOE_ERR_INVALID_ARG
    assert fwd(moe.CAPACITY_REROUTE, 3, stats=FAKE) == moe.MOE_ERR_INVALID_ARG
    assert fwd(4, 3) == moe.MOE_ERR_INVALID_ARG
    assert moe.CAPACITY_REROUTE == 2 and moe.GATES_RENORMALISE == 1


def test_binding_refuses_host_tensors_without_gpu():
    """The binding hands the library device addresses only: a host tensor is refused before any call
    (its address would be dereferenced on the GPU); raw integer addresses and None pass through."""
    import torch
    x, w_r = torch.zeros(4, 8, dtype=torch.bfloat16), torch.zeros(8, 8, dtype=torch.bfloat16)
    idx, gate = torch.zeros(4, 2, dtype=torch.int32), torch.zeros(4, 2, dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensors"):
        moe.router_topk(x, w_r, None, 4, 8, 8, 2, moe.MOE_DTYPE_BF16, idx, gate)
    assert _lib._ptr(None) is None and _lib._ptr(4096) == 4096


def test_binding_refuses_short_or_mistyped_tensors_without_gpu():
    """A tensor with fewer bytes than the sizes passed would be read or written past its end, and the
    layer's data in another element type would be misread: both are refused before any call."""
    import torch
    x, w_r = torch.zeros(4, 8, dtype=torch.bfloat16), torch.zeros(8, 8, dtype=torch.bfloat16)
    idx, gate = torch.zeros(4, 2, dtype=torch.int32), torch.zeros(4, 2, dtype=torch.float32)
    BF16 = moe.MOE_DTYPE_BF16
    with pytest.raises(ValueError, match="the call needs"):      # T = 5 tokens, x holds 4
        moe.router_topk(x, w_r, None, 5, 8, 8, 2, BF16, idx, gate)
    with pytest.raises(ValueError, match="the call needs"):      # k = 3, the outputs hold k = 2
        moe.router_topk(x, w_r, None, 4, 8, 8, 3, BF16, idx, gate)
    with pytest.raises(ValueError, match="2-byte elements"):     # bf16 data for an fp32 call
        moe.router_topk(x, w_r, None, 4, 8, 8, 2, moe.MOE_DTYPE_F32, idx, gate)
    with pytest.raises(ValueError, match="the call needs"):      # out smaller than [T, d]
        moe.combine(torch.zeros(4 * 2 * 8), idx, 4, 8, 2, BF16, torch.zeros(3, 8, dtype=torch.bfloat16))

"""fp64 CPU oracle of the sparse top-k MoE FFN layer's forward pass.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it. The CUDA library never calls it
and shares no code with it: the only module both sides use is ``inputgen``,
which holds no arithmetic of the layer.

Every function is pinned by ``tests/test_oracle_pins.py`` against facts fixed
outside the oracle (the pages' worked router example, closed forms, library
routines for the special cases, brute force on tiny inputs). There is no
"parity unpinned" function.
"""
from .moe import (  # noqa: F401
    router_logits, softmax, topk_select, gates_of, gates_renormalised, gelu, expert_ffn, forward, dense_forward,
    dispatch, capacity, kept_assignments, reroute_assignments, expert_rows_ffn, expert_rows_up, expert_rows_down, combine, routing_stats, quantize_blocks, dequantize_blocks,
    packed_code_bytes, ambiguous_tokens,
    top_share,
)

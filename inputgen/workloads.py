"""The layer's workloads: sizes, dtypes and input recipe of each configuration.

Holds no arithmetic of the layer. Sizes follow the five workloads the pages'
problem statement is measured on (a tiny fp32 layer, a 16-expert bf16 layer, a
128-expert prefill layer, a decode-shaped layer and a skew-routed layer).

``SKEW_BIAS_SCALE`` is the constant ``c`` of the skew-routed workload's router
bias ``c*log((e+1)**-1.2)``; it was written by ``tests/golden/calibrate_skew.py``
(which calls only the oracle) so that the five most-loaded experts take 38% of
the assignments on the seed-0 draw. ``tests/golden/skew_bias_scale.json``
holds the script's output and a test checks that the two agree.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional

from . import DTYPE_BF16, DTYPE_F32

SKEW_BIAS_SCALE = 0.399227


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    F: int
    E: int
    k: int
    dtype: int
    seed: int = 0
    skew: bool = False

    @property
    def A(self) -> int:
        return self.T * self.k

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # Tiny fp32 layer: T=64, d=128, E=8, top-2, d_ff=256, no biases.
    "tiny_fp32": Workload("tiny_fp32", T=64, d=128, F=256, E=8, k=2, dtype=DTYPE_F32),
    # 16-expert bf16 layer: T=4096, d=1024, d_ff=4096, plain random router.
    "e16_bf16": Workload("e16_bf16", T=4096, d=1024, F=4096, E=16, k=2, dtype=DTYPE_BF16),
    # 128-expert prefill layer: T=8192, d=4096, d_ff=8192 (17.2 GB of expert weights).
    "prefill_e128": Workload("prefill_e128", T=8192, d=4096, F=8192, E=128, k=2, dtype=DTYPE_BF16),
    # Decode-shaped layer: d=d_ff=8192, E=128 (34.4 GB of expert weights), T = 1, 8, 64.
    "decode_t1": Workload("decode_t1", T=1, d=8192, F=8192, E=128, k=2, dtype=DTYPE_BF16),
    "decode_t8": Workload("decode_t8", T=8, d=8192, F=8192, E=128, k=2, dtype=DTYPE_BF16),
    "decode_t64": Workload("decode_t64", T=64, d=8192, F=8192, E=128, k=2, dtype=DTYPE_BF16),
    # Profiling-size decode layer: the decode layer's per-expert shape with 16 experts (4.3 GB), small
    # enough for a full ncu capture of the streaming kernel.
    "decode_t1_e16": Workload("decode_t1_e16", T=1, d=8192, F=8192, E=16, k=2, dtype=DTYPE_BF16),
    # Profiling-size prefill layer: the prefill layer's per-expert shape (about 128 rows per expert,
    # d=4096, d_ff=8192) with 16 experts (2.1 GB), small enough for a full ncu capture.
    "prefill_e16": Workload("prefill_e16", T=1024, d=4096, F=8192, E=16, k=2, dtype=DTYPE_BF16),
    # Profiling-size skew-routed layer: the skew layer's per-expert shape and router bias with 16
    # experts and T=2048 (2.1 GB of weights), small enough for a full ncu capture.
    "skew_e16": Workload("skew_e16", T=2048, d=4096, F=8192, E=16, k=2, dtype=DTYPE_BF16, skew=True),
    # Skew-routed layer: T=16384, power-law router bias, else as the prefill layer.
    "skew_e128": Workload("skew_e128", T=16384, d=4096, F=8192, E=128, k=2, dtype=DTYPE_BF16,
                          skew=True),
}


def get(name: str) -> Workload:
    return WORKLOADS[name]


def bias_scale(w: Workload) -> Optional[float]:
    """Router-bias scale c for a workload, None when it has no router bias."""
    if not w.skew:
        return None
    if SKEW_BIAS_SCALE is None:
        raise RuntimeError("skew bias scale not calibrated yet")
    return SKEW_BIAS_SCALE

"""Calibrate the skew-routed workload's router-bias scale c; writes skew_bias_scale.json.

The workload adds a per-expert router bias c*log((e+1)**-1.2) (expert e has
popularity rank e+1) so that the five most-loaded experts take about 38% of the
top-2 assignments, the share csdn/6a919c0d §2.2 reports for real traffic. The
pages give the power law and the share but not the scale of the logits it acts
on, so c is found here by bisection on the seed-0 draw of the workload
(T=16384, d=4096, E=128, bf16 x and W_r), routed by the oracle. Calls only
``oracle`` and ``inputgen``.

Run:  python tests/golden/calibrate_skew.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import inputgen as ig  # noqa: E402
import oracle  # noqa: E402

TARGET_SHARE = 0.38
TOP_N = 5


def main():
    T, d, E, k, seed = 16384, 4096, 128, 2, 0
    x = ig.as_f64(ig.draw(0, T * d, ig.stream_key(seed, ig.STREAM_X), 1.0, ig.DTYPE_BF16), ig.DTYPE_BF16)
    w_r = ig.as_f64(ig.draw(0, d * E, ig.stream_key(seed, ig.STREAM_WR), ig.sigma_for_fan_in(d), ig.DTYPE_BF16),
                    ig.DTYPE_BF16)
    logits0 = oracle.router_logits(x.reshape(T, d), w_r.reshape(d, E))

    def share(c):
        b = ig.skew_bias(E, c).astype(np.float64)
        idx = oracle.topk_select(logits0 + b[None, :], k)
        return oracle.top_share(oracle.dispatch(idx, E)["counts"], TOP_N)

    lo, hi = 0.0, 1.0
    s_lo, s_hi = share(lo), share(hi)
    assert s_lo < TARGET_SHARE < s_hi, (s_lo, s_hi)
    for _ in range(30):
        mid = 0.5 * (lo + hi)
        if share(mid) < TARGET_SHARE:
            lo = mid
        else:
            hi = mid
    c = round(0.5 * (lo + hi), 6)
    out = {
        "what": "router-bias scale c of the skew-routed workload: bias[e] = c*log((e+1)**-1.2)",
        "target": f"top-{TOP_N} experts take {TARGET_SHARE} of the top-{k} assignments (csdn/6a919c0d section 2.2)",
        "workload": {"T": T, "d": d, "E": E, "k": k, "seed": seed, "dtype": "bf16"},
        "c": c,
        "share_at_c": share(c),
        "share_at_c_equal_1": s_hi,
    }
    with open(os.path.join(HERE, "skew_bias_scale.json"), "w") as f:
        json.dump(out, f, indent=2)
    print(json.dumps(out, indent=2))


if __name__ == "__main__":
    main()

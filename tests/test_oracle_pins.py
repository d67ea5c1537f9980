"""Pins of the fp64 oracle against facts fixed outside it.

Each pin ties one oracle function to something other than itself: a worked
example printed on the pages, a closed form, a library routine for a special
case that reduces to it, or brute force on tiny inputs. ``test_planted_mistakes``
shows that a plausible mistake planted anywhere in the oracle fails at least one
pin.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import moe as om

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand_layer(rng, T, d, F, E, scale_r=1.0):
    x = rng.standard_normal((T, d))
    w_r = rng.standard_normal((d, E)) * scale_r / math.sqrt(d)
    w1 = rng.standard_normal((E, d, F)) / math.sqrt(d)
    w2 = rng.standard_normal((E, F, d)) / math.sqrt(F)
    return x, w_r, w1, w2


# ----------------------------------------------------------------------------- pin checks
# Each check raises AssertionError on failure. They look oracle functions up on the
# module at call time, so test_planted_mistakes can swap one out.

def check_worked_example():
    """aicoding/6a320eef §3.1: probabilities 0.42/0.38/0.12/0.05/(<0.01) -> experts 3 and 17, gates sum 0.80."""
    g = _load("router_worked_example.json")
    E = g["E"]
    named = {int(e): p for e, p in g["named_probs"].items()}
    rest = (1.0 - sum(named.values())) / (E - len(named))
    assert rest < g["others_below"]
    p_true = np.full(E, rest)
    for e, p in named.items():
        p_true[e] = p
    # One token whose hidden state is the first unit vector: its logits are row 0 of W_r.
    d = 4
    x = np.zeros((1, d)); x[0, 0] = 1.0
    w_r = np.zeros((d, E)); w_r[0] = np.log(p_true) + 3.0   # any common shift
    logits = om.router_logits(x, w_r)
    p = om.softmax(logits)
    idx = om.topk_select(logits, 2)
    gate = om.gates_of(p, idx)
    assert list(idx[0]) == g["expected_top2"]
    assert np.allclose(gate[0], g["expected_gates"], rtol=0, atol=1e-12)
    assert abs(gate[0].sum() - g["expected_gate_sum"]) < 1e-12
    assert np.allclose(p[0], p_true, rtol=1e-12, atol=0)


def check_router_closed_form():
    """Zero hidden state gives logits = bias; a unit vector e_i gives row i of W_r plus bias."""
    rng = np.random.default_rng(1)
    d, E = 6, 5
    w_r = rng.standard_normal((d, E))
    b_r = rng.standard_normal(E)
    x = np.zeros((d + 1, d))
    for i in range(d):
        x[i + 1, i] = 1.0
    logits = om.router_logits(x, w_r, b_r)
    assert np.array_equal(logits[0], b_r)
    for i in range(d):
        assert np.allclose(logits[i + 1], w_r[i] + b_r, rtol=0, atol=1e-15)


def check_softmax_library():
    """Softmax equals scipy's, sums to one, and is shift invariant."""
    rng = np.random.default_rng(2)
    l = rng.standard_normal((7, 13)) * 5
    p = om.softmax(l)
    assert np.allclose(p, scipy.special.softmax(l, axis=1), rtol=1e-13, atol=0)
    assert np.allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.allclose(om.softmax(l + 1000.0), p, rtol=1e-12, atol=0)


def check_topk_ties_and_order():
    """Largest first; equal logits go to the lower index; matches torch.topk where there are no ties."""
    l = np.array([[1.0, 3.0, 3.0, 2.0],
                  [5.0, 5.0, 5.0, 5.0],
                  [0.0, -1.0, 2.0, 2.0]])
    assert om.topk_select(l, 2).tolist() == [[1, 2], [0, 1], [2, 3]]
    assert om.topk_select(l, 3).tolist() == [[1, 2, 3], [0, 1, 2], [2, 3, 0]]
    rng = np.random.default_rng(3)
    l = rng.standard_normal((50, 9))
    ref = torch.topk(torch.from_numpy(l), 3, dim=1).indices.numpy()
    assert np.array_equal(om.topk_select(l, 3), ref)


def check_gelu_closed_form():
    """GeLU(z) = z*Phi(z): GeLU(0) = 0, GeLU(1) = Phi(1), GeLU(-1) = -(1 - Phi(1)), -> z and 0 in the tails; matches torch's erf GeLU."""
    facts = _load("page_facts.json")["gelu_closed_form"]
    phi1 = facts["phi_1"]
    g = om.gelu(np.array([0.0, 1.0, -1.0, 12.0, -12.0]))
    assert g[0] == 0.0
    assert abs(g[1] - phi1) < 1e-15
    assert abs(g[2] + (1.0 - phi1)) < 1e-15
    assert abs(g[3] - 12.0) < 1e-15 and abs(g[4]) < 1e-30
    z = np.linspace(-6, 6, 1001)
    ref = torch.nn.functional.gelu(torch.from_numpy(z), approximate="none").numpy()
    # 1 + erf(z/sqrt 2) cancels for z < 0, so compare absolutely (the tanh form differs by ~1e-3)
    assert np.max(np.abs(om.gelu(z) - ref)) < 1e-14


def check_single_expert_is_mlp():
    """k = E = 1: the layer is the plain two-layer GeLU MLP (gate = 1), computed here with torch."""
    rng = np.random.default_rng(4)
    x, w_r, w1, w2 = _rand_layer(rng, T=5, d=6, F=6, E=1)
    w1[0] = rng.standard_normal((6, 6))   # asymmetric square matrices: a transposed operand shows
    res = om.forward(x, w_r, w1, w2, k=1)
    tx = torch.from_numpy(x)
    ref = torch.nn.functional.gelu(tx @ torch.from_numpy(w1[0]), approximate="none") @ torch.from_numpy(w2[0])
    assert np.allclose(res["gate"], 1.0, rtol=0, atol=0)
    assert np.allclose(res["out"], ref.numpy(), rtol=1e-12, atol=1e-13)


def check_k_equals_E_is_softmax_mixture():
    """k = E: every expert is used and the layer is the dense softmax mixture sum_e p_e FFN_e(x) (torch einsum)."""
    rng = np.random.default_rng(5)
    x, w_r, w1, w2 = _rand_layer(rng, T=9, d=5, F=7, E=3)
    res = om.forward(x, w_r, w1, w2, k=3)
    tx = torch.from_numpy(x)
    p = torch.softmax(tx @ torch.from_numpy(w_r), dim=1)
    h = torch.nn.functional.gelu(torch.einsum("td,edf->etf", tx, torch.from_numpy(w1)), approximate="none")
    y = torch.einsum("etf,efd->etd", h, torch.from_numpy(w2))
    ref = torch.einsum("te,etd->td", p, y)
    assert np.allclose(res["out"], ref.numpy(), rtol=1e-12, atol=1e-13)


def check_routed_equals_dense_bruteforce():
    """The routed forward equals the brute-force all-experts evaluation masked to the top-k (to 1e-12 relative)."""
    rng = np.random.default_rng(6)
    for (T, d, F, E, k) in [(16, 8, 12, 8, 2), (11, 16, 16, 3, 2), (7, 4, 5, 2, 1), (13, 6, 9, 8, 8), (3, 8, 8, 5, 3)]:
        x, w_r, w1, w2 = _rand_layer(rng, T, d, F, E)
        b_r = rng.standard_normal(E) * 0.3
        routed = om.forward(x, w_r, w1, w2, k, b_r)["out"]
        dense = om.dense_forward(x, w_r, w1, w2, k, b_r)
        rms = math.sqrt(float(np.mean(dense ** 2)))
        assert np.max(np.abs(routed - dense)) / rms < 1e-12


def check_routing_invariants():
    """Exactly k distinct experts per token; gates are the softmax probabilities, non-increasing by slot, summing to <= 1 (< 1 when E > k)."""
    rng = np.random.default_rng(7)
    for (E, k) in [(8, 2), (128, 2), (4, 4), (16, 3)]:
        l = rng.standard_normal((200, E))
        p = om.softmax(l)
        idx = om.topk_select(l, k)
        gate = om.gates_of(p, idx)
        assert all(len(set(r)) == k for r in idx.tolist())
        assert np.array_equal(gate, p[np.arange(200)[:, None], idx])
        assert np.all(np.diff(gate, axis=1) <= 0)
        s = gate.sum(axis=1)
        assert np.all(s <= 1.0 + 1e-15)
        if E > k:
            assert np.all(s < 1.0)


def check_activation_fraction():
    """csdn/6a919c0d §2.2: top-2 of 128 experts activates 2/128 = 1.5625% of them for every token."""
    f = _load("page_facts.json")["activation_fraction"]
    rng = np.random.default_rng(8)
    l = rng.standard_normal((300, f["E"]))
    idx = om.topk_select(l, f["k"])
    counts = om.dispatch(idx, f["E"])["counts"]
    assert counts.sum() == 300 * f["k"]
    assert counts.sum() / (300 * f["E"]) == f["fraction"]


def check_dispatch_stable_sort():
    """The permutation equals numpy's stable argsort of the assignments by expert; counts and offsets match bincount/cumsum."""
    rng = np.random.default_rng(9)
    for (T, k, E) in [(40, 2, 7), (1, 2, 3), (100, 3, 16), (64, 2, 2)]:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
        gate = rng.random((T, k))
        dp = om.dispatch(idx, E, gate)
        flat = idx.reshape(-1)
        order = np.argsort(flat, kind="stable")
        assert np.array_equal(dp["perm_token"], order // k)
        inv = np.empty_like(order); inv[order] = np.arange(T * k)
        assert np.array_equal(dp["row_of"].reshape(-1), inv)
        assert np.array_equal(dp["counts"], np.bincount(flat, minlength=E))
        assert np.array_equal(dp["offsets"], np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
        assert np.array_equal(dp["row_gate"], gate.reshape(-1)[order])


def check_steps_compose_to_forward():
    """Dispatch -> per-row expert FFN with gate -> combine reproduces the forward pass."""
    rng = np.random.default_rng(10)
    x, w_r, w1, w2 = _rand_layer(rng, T=21, d=8, F=10, E=5)
    res = om.forward(x, w_r, w1, w2, k=2)
    dp = om.dispatch(res["idx"], 5, res["gate"])
    y_perm = om.expert_rows_ffn(x[dp["perm_token"]], dp["offsets"], dp["row_gate"], w1, w2)
    out = om.combine(y_perm, dp["row_of"])
    assert np.allclose(out, res["out"], rtol=1e-13, atol=1e-14)
    rows = np.array([0, 5, 17, 41])
    part = om.expert_rows_ffn(x[dp["perm_token"]], dp["offsets"], dp["row_gate"], w1, w2, rows=rows)
    assert np.allclose(part, y_perm[rows], rtol=1e-13, atol=1e-15)
    h = om.expert_rows_up(x[dp["perm_token"]], dp["offsets"], w1)
    y2 = om.expert_rows_down(h, dp["offsets"], dp["row_gate"], w2)
    assert np.allclose(y2, y_perm, rtol=1e-13, atol=1e-15)
    h_part = om.expert_rows_up(x[dp["perm_token"]], dp["offsets"], w1, rows=rows)
    assert np.allclose(h_part, h[rows], rtol=1e-13, atol=1e-15)


def check_ambiguous_tokens():
    """Tokens with a top-(k+1) adjacent gap below the threshold are flagged, others are not."""
    l = np.array([[3.0, 2.0, 1.0, 0.0],
                  [3.0, 3.0 - 5e-4, 1.0, 0.0],
                  [3.0, 2.0, 2.0 - 5e-4, 0.0],
                  [3.0, 2.0, 1.0, 1.0 - 5e-4],
                  [3.0, 2.0, 2.0 - 2e-3, 0.0]])
    assert om.ambiguous_tokens(l, 2, 1e-3).tolist() == [1, 2]


def check_renormalised_gates():
    """hotelren §4.3 gates: softmax of the k selected logits equals p_j / sum of the selected p (closed form),
    matches scipy, sums to one; k = E gives the plain gates; k = 1 gives gate 1; routed equals brute force."""
    rng = np.random.default_rng(11)
    l = rng.standard_normal((40, 16)) * 2
    idx = om.topk_select(l, 3)
    w = om.gates_renormalised(l, idx)
    p = om.softmax(l)
    sel = np.take_along_axis(p, idx, 1)
    assert np.allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-13, atol=0)
    assert np.allclose(w, scipy.special.softmax(np.take_along_axis(l, idx, 1), axis=1), rtol=1e-13, atol=0)
    assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    full = om.topk_select(l, 16)
    assert np.allclose(om.gates_renormalised(l, full), om.gates_of(p, full), rtol=1e-12, atol=0)
    assert np.array_equal(om.gates_renormalised(l, om.topk_select(l, 1)), np.ones((40, 1)))
    for (T, d, F, E, k) in [(12, 8, 10, 6, 2), (9, 6, 6, 4, 3)]:
        x, w_r, w1, w2 = _rand_layer(rng, T, d, F, E)
        routed = om.forward(x, w_r, w1, w2, k, renormalise=True)["out"]
        dense = om.dense_forward(x, w_r, w1, w2, k, renormalise=True)
        assert np.max(np.abs(routed - dense)) / math.sqrt(float(np.mean(dense ** 2))) < 1e-12


def check_capacity():
    """aicoding §3.2: capacity ceil(T*k/E*cf) (worked example 64); the first C assignments of each expert in
    (t, j) order are kept (independently ranked with numpy's stable argsort); a capacity nobody reaches changes
    nothing; the forward pass with drops equals a per-assignment brute force."""
    f = _load("page_facts.json")["capacity_worked_example"]
    assert om.capacity(f["T"], f["k"], f["E"], f["cf"]) == f["capacity"]
    rng = np.random.default_rng(12)
    T, k, E = 120, 2, 6
    l = rng.standard_normal((T, E)) + np.array([1.5, 1.0, 0.0, 0.0, -0.5, -1.0])
    idx = om.topk_select(l, k)
    gate = om.gates_of(om.softmax(l), idx)
    flat = idx.reshape(-1)
    order = np.argsort(flat, kind="stable")
    rank = np.empty_like(order)
    for e in range(E):
        pos = order[flat[order] == e]
        rank[pos] = np.arange(len(pos))
    for C in [1, 3, 17, 1000]:
        keep = om.kept_assignments(idx, E, C)
        assert np.array_equal(keep.reshape(-1), rank < C)
        dp = om.dispatch(idx, E, gate, C)
        assert np.array_equal(dp["counts"], np.minimum(np.bincount(flat, minlength=E), C))
        assert np.array_equal(dp["row_of"].reshape(-1) >= 0, keep.reshape(-1))
        kept_rows = dp["row_of"].reshape(-1)[keep.reshape(-1)]
        assert np.array_equal(np.sort(kept_rows), np.arange(dp["offsets"][-1]))
    x, w_r, w1, w2 = _rand_layer(rng, T=40, d=6, F=8, E=5)
    res = om.forward(x, w_r, w1, w2, 2)
    assert np.array_equal(om.forward(x, w_r, w1, w2, 2, cap=80)["out"], res["out"])
    C = 7
    capped = om.forward(x, w_r, w1, w2, 2, cap=C)["out"]
    brute = np.zeros_like(capped)
    seen = {}
    for t in range(40):
        for j in range(2):
            e = int(res["idx"][t, j])
            if seen.get(e, 0) < C:
                brute[t] += res["gate"][t, j] * om.expert_ffn(x[t:t + 1], w1[e], w2[e])[0]
            seen[e] = seen.get(e, 0) + 1
    assert np.max(np.abs(capped - brute)) < 1e-12


def check_capacity_reroute():
    """Rerouting at capacity (aicoding §3.2, csdn/6a919c0d §3.2): a hand-worked case; the special cases that
    reduce to plain top-k (capacity nobody reaches) and to the drop rule (no candidates beyond the k chosen);
    for one slot per token and the whole ranking, the serial rule "each token in turn takes its best expert
    with room" computed from masked logits; for k slots, a brute force that searches the ranking afresh for
    every rerouted slot; the forward pass equals a per-assignment sum over the final experts."""
    # hand-worked: 4 tokens, 3 experts, capacity 1, every token ranks 0 > 1 > 2
    ri = np.array([[0, 1, 2]] * 4)
    rp = np.array([[0.5, 0.3, 0.2]] * 4)
    fi, fg = om.reroute_assignments(ri, rp, 1, 3, 1)
    assert fi.reshape(-1).tolist() == [0, 1, 2, -1]
    assert np.allclose(fg.reshape(-1), [0.5, 0.3, 0.2, 0.0], rtol=0, atol=0)
    # k = 2, capacity 1: token 1 wants 1 (held) -> its rank-2 expert 3; wants 0 (held) -> rank-3 expert 2;
    # token 2 finds every expert held and is dropped
    ri = np.array([[0, 1, 2, 3], [1, 0, 3, 2], [0, 1, 2, 3]])
    rp = np.array([[0.4, 0.3, 0.2, 0.1], [0.4, 0.3, 0.2, 0.1], [0.4, 0.3, 0.2, 0.1]])
    fi, fg = om.reroute_assignments(ri, rp, 2, 4, 1)
    assert fi.tolist() == [[0, 1], [3, 2], [-1, -1]]
    assert fg.tolist() == [[0.4, 0.3], [0.2, 0.1], [0.0, 0.0]]
    rng = np.random.default_rng(21)
    for trial in range(12):
        T, E = int(rng.integers(5, 60)), int(rng.integers(2, 9))
        k = int(rng.integers(1, min(E, 3) + 1))
        R = int(rng.integers(k, E + 1))
        cap = int(rng.integers(1, max(2, T * k // E + 2)))
        l = rng.standard_normal((T, E)) + np.linspace(1.5, -1.5, E)
        p = om.softmax(l)
        ri = om.topk_select(l, R)
        rp = om.gates_of(p, ri)
        fi, fg = om.reroute_assignments(ri, rp, k, E, cap)
        counts = np.bincount(fi[fi >= 0], minlength=E)
        assert np.all(counts <= cap)
        for t in range(T):
            got = fi[t][fi[t] >= 0]
            assert len(set(got.tolist())) == len(got)                 # distinct experts per token
            assert set(got.tolist()) <= set(ri[t].tolist())           # within its R best
        # brute force: every slot in (t, j) order takes its own choice if it has room, else the best-ranked
        # expert among ranks k..R-1 that has room and does not hold this token already
        held = np.zeros(E, np.int64)
        bi = np.full((T, k), -1)
        bg = np.zeros((T, k))
        for t in range(T):
            for j in range(k):
                cands = [j] if held[ri[t, j]] < cap else [r for r in range(k, R)
                                                           if held[ri[t, r]] < cap and ri[t, r] not in bi[t]]
                if cands:
                    r = cands[0]
                    bi[t, j], bg[t, j] = ri[t, r], rp[t, r]
                    held[ri[t, r]] += 1
        assert np.array_equal(fi, bi) and np.array_equal(fg, bg), trial
        # a capacity nobody reaches: plain top-k with the raw gates
        fi2, fg2 = om.reroute_assignments(ri, rp, k, E, T * k)
        assert np.array_equal(fi2, ri[:, :k]) and np.array_equal(fg2, rp[:, :k])
        # no candidates beyond the k chosen: the drop rule
        fi3, _ = om.reroute_assignments(ri[:, :k], rp[:, :k], k, E, cap)
        assert np.array_equal(fi3 >= 0, om.kept_assignments(ri[:, :k], E, cap))
        # one slot per token and the whole ranking: each token in turn takes its best expert with room
        if k == 1 and R == E:
            held = np.zeros(E, np.int64)
            for t in range(T):
                masked = np.where(held < cap, l[t], -np.inf)
                want = int(np.argmax(masked)) if np.isfinite(masked).any() else -1
                assert fi[t, 0] == want
                if want >= 0:
                    held[want] += 1
    # the forward pass with rerouting: the final experts' outputs weighted by their probabilities
    x, w_r, w1, w2 = _rand_layer(rng, T=30, d=6, F=8, E=5)
    b = np.array([1.5, 1.0, 0.0, -0.5, -1.0])
    res = om.forward(x, w_r, w1, w2, 2, b_r=b, cap=8, reroute=5)
    lg = om.router_logits(x, w_r, b)
    ranked = np.argsort(-lg, axis=1, kind="stable")
    brute = np.zeros_like(res["out"])
    held = {}
    for t in range(30):
        mine = []
        for j in range(2):
            e = int(ranked[t, j])
            if held.get(e, 0) >= 8:
                e = next((int(c) for c in ranked[t, 2:] if held.get(int(c), 0) < 8 and int(c) not in mine), -1)
            if e >= 0:
                held[e] = held.get(e, 0) + 1
                mine.append(e)
                brute[t] += om.softmax(lg)[t, e] * om.expert_ffn(x[t:t + 1], w1[e], w2[e])[0]
    assert np.max(np.abs(res["out"] - brute)) < 1e-12
    assert (res["idx"] != om.topk_select(lg, 2)).any()  # something was rerouted
    dp = om.dispatch(res["idx"], 5, res["gate"])
    assert np.array_equal(dp["row_of"] >= 0, res["idx"] >= 0)
    assert dp["offsets"][-1] == (res["idx"] >= 0).sum()


def check_routing_stats():
    """Routing statistics: soft load = column means of scipy's softmax; equal logits give entropy ln E
    (closed form) and equal soft loads; entropy matches scipy.stats.entropy per token; a batch whose
    counts are equal by construction has balance exactly 0 while its soft loads differ; every token on
    one expert (k = 1) gives balance 1 - 1/E (closed form); loops over a tiny case agree."""
    import scipy.stats
    rng = np.random.default_rng(13)
    T, E, k = 50, 8, 2
    l = rng.standard_normal((T, E)) * 1.5
    idx = om.topk_select(l, k)
    st = om.routing_stats(l, idx)
    sp = scipy.special.softmax(l, axis=1)
    assert np.allclose(st["soft_load"], sp.mean(axis=0), rtol=1e-13, atol=0)
    assert abs(st["soft_load"].sum() - 1.0) < 1e-14 and abs(st["hard_load"].sum() - 1.0) < 1e-14
    assert np.array_equal(st["hard_load"] * T * k, np.bincount(idx.reshape(-1), minlength=E))
    assert abs(st["entropy"] - float(np.mean(scipy.stats.entropy(sp, axis=1)))) < 1e-13
    flat = om.routing_stats(np.full((7, 16), 0.3), om.topk_select(np.full((7, 16), 0.3), 2))
    assert abs(flat["entropy"] - math.log(16)) < 1e-14
    assert np.allclose(flat["soft_load"], 1.0 / 16, rtol=0, atol=1e-16)
    # token t prefers expert t % E, by a margin that grows with t: equal counts, unequal soft loads
    lb = np.zeros((4 * E, E))
    for t in range(4 * E):
        lb[t, t % E] = 1.0 + 0.5 * (t % E)
    bal = om.routing_stats(lb, om.topk_select(lb, 1))
    assert bal["balance"] == 0.0 and np.std(bal["soft_load"]) > 1e-3
    one = np.zeros((30, E))
    one[:, 5] = 3.0
    r1 = om.routing_stats(one, om.topk_select(one, 1))
    assert abs(r1["balance"] - (1.0 - 1.0 / E)) < 1e-15
    ls = rng.standard_normal((5, 4))
    ids = om.topk_select(ls, 2)
    soft, ent = [0.0] * 4, 0.0
    for t in range(5):
        ex = [math.exp(v) for v in ls[t]]
        z = sum(ex)
        for e in range(4):
            soft[e] += ex[e] / z / 5
            ent -= ex[e] / z * math.log(ex[e] / z) / 5
    cnt = [0] * 4
    for t in range(5):
        for j in range(2):
            cnt[ids[t, j]] += 1
    small = om.routing_stats(ls, ids)
    assert np.allclose(small["soft_load"], soft, rtol=1e-13, atol=0)
    assert abs(small["entropy"] - ent) < 1e-13
    assert abs(small["balance"] - sum((c / 10 - 0.25) ** 2 for c in cnt)) < 1e-15


def check_block_quantizer():
    """csdn/6a462500 §4.3 block quantizer: the page's size example (fp16 bytes -> INT4 code bytes); per
    64 x 64 block the minimum gets code 0 and the maximum the top code; codes are monotone in w; every
    weight is restored within half a step (the rounding bound); an equally spaced block with a
    power-of-two step is restored exactly; a flat block has scale 0 and is restored exactly."""
    f = _load("page_facts.json")["int4_size_example"]
    n_weights = f["fp16_bytes"] // 2
    assert om.packed_code_bytes(8192, n_weights // 8192, 4) == f["int4_code_bytes"]
    assert om.packed_code_bytes(8192, n_weights // 8192, 8) == 2 * f["int4_code_bytes"]
    rng = np.random.default_rng(14)
    w = (rng.standard_normal((128, 192)) * 0.05).astype(np.float32)
    for bits in (4, 8):
        q = om.quantize_blocks(w, bits)
        top = 2 ** bits - 1
        assert q["scale"].shape == (2, 3) and q["min"].shape == (2, 3)
        assert q["codes"].min() >= 0 and q["codes"].max() <= top
        wh = om.dequantize_blocks(q)
        for bi in range(2):
            for bj in range(3):
                sl = (slice(64 * bi, 64 * bi + 64), slice(64 * bj, 64 * bj + 64))
                blk, c = w[sl].astype(np.float64), q["codes"][sl]
                assert c.reshape(-1)[np.argmin(blk)] == 0 and c.reshape(-1)[np.argmax(blk)] == top
                assert q["min"][bi, bj] == blk.min()
                order = np.argsort(blk.reshape(-1), kind="stable")
                assert np.all(np.diff(c.reshape(-1)[order].astype(np.int64)) >= 0)
                step = (blk.max() - blk.min()) / top
                assert np.max(np.abs(wh[sl] - blk)) <= 0.5 * step * (1 + 1e-5)
    grid = np.zeros((64, 64), np.float32)
    for i in range(64):
        for j in range(64):
            grid[i, j] = -0.75 + 0.125 * ((3 * i + j) % 16)
    qg = om.quantize_blocks(grid, 4)
    assert qg["scale"][0, 0] == 0.125 and np.array_equal(om.dequantize_blocks(qg), grid.astype(np.float64))
    flat = np.full((64, 128), 0.3, np.float32)
    qf = om.quantize_blocks(flat, 4)
    assert np.all(qf["scale"] == 0) and np.all(qf["codes"] == 0)
    assert np.array_equal(om.dequantize_blocks(qf), flat.astype(np.float64))


PINS = [check_worked_example, check_router_closed_form, check_softmax_library, check_topk_ties_and_order,
        check_gelu_closed_form, check_single_expert_is_mlp, check_k_equals_E_is_softmax_mixture,
        check_routed_equals_dense_bruteforce, check_routing_invariants, check_activation_fraction,
        check_dispatch_stable_sort, check_steps_compose_to_forward, check_ambiguous_tokens,
        check_renormalised_gates, check_capacity, check_capacity_reroute, check_routing_stats,
        check_block_quantizer]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ----------------------------------------------------------------------------- planted mistakes

def _mut_gelu_sign(z):
    z = np.asarray(z, np.float64)
    return 0.5 * z * (1.0 - scipy.special.erf(z / math.sqrt(2.0)))


def _mut_gelu_tanh(z):
    z = np.asarray(z, np.float64)
    return 0.5 * z * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (z + 0.044715 * z ** 3)))


def _mut_softmax_unnormalised(l):
    l = np.asarray(l, np.float64)
    return np.exp(l - l.max(axis=1, keepdims=True))


def _mut_topk_smallest(l, k):
    return np.argsort(np.asarray(l), axis=1, kind="stable")[:, :k]


def _mut_topk_last_on_tie(l, k):
    l = np.asarray(l, np.float64)
    E = l.shape[1]
    rev = _ORIG_TOPK(l[:, ::-1], k)
    return E - 1 - rev


def _mut_gates_renormalised(p, idx):
    g = np.take_along_axis(np.asarray(p), np.asarray(idx), axis=1)
    return g / g.sum(axis=1, keepdims=True)


def _mut_renormalised_over_all(logits, idx):
    return np.take_along_axis(om.softmax(logits), np.asarray(idx), axis=1)


def _mut_capacity_keeps_last(idx, E, cap):
    keep = _ORIG_KEPT(np.asarray(idx)[::-1], E, cap)
    return keep[::-1]


def _mut_ffn_transposed_w1(x_rows, w1_e, w2_e):
    return om.gelu(np.asarray(x_rows) @ np.asarray(w1_e).T) @ np.asarray(w2_e)


def _mut_router_drops_bias(x, w_r, b_r=None):
    return np.asarray(x, np.float64) @ np.asarray(w_r, np.float64)


def _mut_dispatch_unstable(idx, E, gate=None, cap=None):
    res = _ORIG_DISPATCH(idx, E, gate, cap)
    # reverse the order of rows inside each expert's range
    offs = res["offsets"]
    row_of = res["row_of"].copy()
    for t in range(row_of.shape[0]):
        for j in range(row_of.shape[1]):
            r = row_of[t, j]
            if r < 0:
                continue
            e = np.searchsorted(offs, r, side="right") - 1
            row_of[t, j] = offs[e] + offs[e + 1] - 1 - r
    perm = np.full_like(res["perm_token"], -1)
    for t in range(row_of.shape[0]):
        for j in range(row_of.shape[1]):
            if row_of[t, j] >= 0:
                perm[row_of[t, j]] = t
    res = dict(res, row_of=row_of, perm_token=perm)
    return res


def _mut_combine_first_slot_twice(y_perm, row_of):
    row_of = np.asarray(row_of).copy()
    row_of[:, 1:] = row_of[:, :1]
    return _ORIG_COMBINE(y_perm, row_of)


def _mut_forward_drops_last_slot(x, w_r, w1, w2, k, b_r=None, renormalise=False, cap=None, reroute=None):
    res = _ORIG_FORWARD(x, w_r, w1, w2, k, b_r, renormalise, cap, reroute)
    res = dict(res)
    res["out"] = res["out"] - res["gate"][:, -1:] * res["y"][-1] if k > 1 else res["out"]
    return res


def _mut_stats(change):
    def f(logits, idx):
        st = dict(_ORIG_STATS(logits, idx))
        l = np.asarray(logits, np.float64)
        T, E = l.shape
        k = np.asarray(idx).shape[1]
        if change == "log2":
            st["entropy"] = st["entropy"] / math.log(2.0)
        elif change == "soft_over_assignments":
            st["soft_load"] = st["soft_load"] / k
        elif change == "balance_of_soft_load":
            st["balance"] = float(np.sum((st["soft_load"] - 1.0 / E) ** 2))
        elif change == "hard_over_tokens":
            st["hard_load"] = st["hard_load"] * k
            st["balance"] = float(np.sum((st["hard_load"] - 1.0 / E) ** 2))
        return st
    return f


def _mut_dequant_drops_min(q):
    c = np.asarray(q["codes"], np.float64)
    s = np.repeat(np.repeat(np.asarray(q["scale"], np.float64), 64, 0), 64, 1)
    return c * s  # the block minimum is lost


def _mut_quant_floor(w, bits):
    q = dict(_ORIG_QUANT(w, bits))
    w32 = np.asarray(w, np.float32)
    s = np.repeat(np.repeat(q["scale"], 64, 0), 64, 1)
    m = np.repeat(np.repeat(q["min"], 64, 0), 64, 1)
    with np.errstate(divide="ignore", invalid="ignore"):
        q["codes"] = np.where(s > 0, np.floor((w32 - m) / s), 0).astype(np.uint8)
    return q


def _mut_quant_levels(w, bits):
    q = dict(_ORIG_QUANT(w, bits))
    w32 = np.asarray(w, np.float32)
    s = np.repeat(np.repeat(q["scale"], 64, 0), 64, 1) * np.float32((2 ** bits - 1) / 2 ** bits)
    m = np.repeat(np.repeat(q["min"], 64, 0), 64, 1)
    with np.errstate(divide="ignore", invalid="ignore"):
        q["codes"] = np.where(s > 0, np.rint((w32 - m) / s), 0).astype(np.int64).clip(0, 255).astype(np.uint8)
    q["scale"] = q["scale"] * np.float32((2 ** bits - 1) / 2 ** bits)
    return q


def _mut_reroute(change):
    def fn(rank_idx, rank_p, k, E, cap):
        rank_idx = np.asarray(rank_idx)
        T, R = rank_idx.shape
        held = np.zeros(E, np.int64)
        fi, fg = np.full((T, k), -1), np.zeros((T, k))
        for t in range(T):
            nxt = k
            for j in range(k):
                e = int(rank_idx[t, j])
                if held[e] < cap:
                    fi[t, j], fg[t, j] = e, rank_p[t, j]
                    held[e] += 1
                    continue
                if change == "restart":
                    nxt = k  # the search starts over for every slot: a token may take an expert twice
                while nxt < R:
                    c = int(rank_idx[t, nxt])
                    nxt += 1
                    if change == "no_room_check" or held[c] < cap:
                        fi[t, j] = c
                        fg[t, j] = rank_p[t, j] if change == "original_gate" else rank_p[t, nxt - 1]
                        held[c] += 1
                        break
        return fi, fg
    return fn


def _mut_rows_down_drops_gate(h, offsets, row_gate, w2, rows=None):
    return _ORIG_ROWS_DOWN(h, offsets, np.ones_like(np.asarray(row_gate, np.float64)), w2, rows)


def _mut_rows_up_next_expert(x_perm, offsets, w1, rows=None):
    # each row takes the weights of the expert after its own (an off-by-one in the row -> expert map)
    E = len(w1)
    shifted = {e: w1[(e + 1) % E] for e in range(E)}
    return _ORIG_ROWS_UP(x_perm, offsets, shifted, rows)


def _mut_dispatch_inclusive_offsets(idx, E, gate=None, cap=None):
    res = dict(_ORIG_DISPATCH(idx, E, gate, cap))
    counts = np.asarray(res["counts"])
    res["offsets"] = np.concatenate([np.cumsum(counts), [int(np.sum(counts))]])
    return res


_ORIG_ROWS_DOWN = om.expert_rows_down
_ORIG_ROWS_UP = om.expert_rows_up
_ORIG_DISPATCH = om.dispatch
_ORIG_TOPK = om.topk_select
_ORIG_KEPT = om.kept_assignments
_ORIG_COMBINE = om.combine
_ORIG_FORWARD = om.forward
_ORIG_STATS = om.routing_stats
_ORIG_QUANT = om.quantize_blocks

MUTANTS = {
    "gelu_sign": ("gelu", _mut_gelu_sign),
    "gelu_tanh": ("gelu", _mut_gelu_tanh),
    "softmax_unnormalised": ("softmax", _mut_softmax_unnormalised),
    "topk_smallest": ("topk_select", _mut_topk_smallest),
    "topk_last_on_tie": ("topk_select", _mut_topk_last_on_tie),
    "gates_renormalised": ("gates_of", _mut_gates_renormalised),
    "renormalised_over_all_experts": ("gates_renormalised", _mut_renormalised_over_all),
    "capacity_keeps_last": ("kept_assignments", _mut_capacity_keeps_last),
    "ffn_transposed_w1": ("expert_ffn", _mut_ffn_transposed_w1),
    "router_drops_bias": ("router_logits", _mut_router_drops_bias),
    "dispatch_unstable": ("dispatch", _mut_dispatch_unstable),
    "combine_first_slot_twice": ("combine", _mut_combine_first_slot_twice),
    "forward_drops_last_slot": ("forward", _mut_forward_drops_last_slot),
    "stats_entropy_log2": ("routing_stats", _mut_stats("log2")),
    "stats_soft_load_over_assignments": ("routing_stats", _mut_stats("soft_over_assignments")),
    "stats_balance_of_soft_load": ("routing_stats", _mut_stats("balance_of_soft_load")),
    "stats_hard_load_over_tokens": ("routing_stats", _mut_stats("hard_over_tokens")),
    "reroute_without_room_check": ("reroute_assignments", _mut_reroute("no_room_check")),
    "reroute_keeps_original_gate": ("reroute_assignments", _mut_reroute("original_gate")),
    "reroute_search_restarts": ("reroute_assignments", _mut_reroute("restart")),
    "dequant_drops_min": ("dequantize_blocks", _mut_dequant_drops_min),
    "quant_floor": ("quantize_blocks", _mut_quant_floor),
    "quant_2^bits_levels": ("quantize_blocks", _mut_quant_levels),
    "rows_down_drops_gate": ("expert_rows_down", _mut_rows_down_drops_gate),
    "rows_up_next_expert": ("expert_rows_up", _mut_rows_up_next_expert),
    "dispatch_inclusive_offsets": ("dispatch", _mut_dispatch_inclusive_offsets),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(om, attr, fn)
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name} was caught by no pin"


def test_package_exports():
    for name in ["router_logits", "softmax", "topk_select", "gates_of", "gelu", "expert_ffn", "forward",
                 "dense_forward", "gates_renormalised", "dispatch", "capacity", "kept_assignments", "reroute_assignments", "expert_rows_ffn", "expert_rows_up", "expert_rows_down", "combine", "routing_stats", "quantize_blocks", "dequantize_blocks",
                 "packed_code_bytes", "ambiguous_tokens", "top_share"]:
        assert callable(getattr(oracle, name))

"""Plain fp64 statement of the sparse top-k MoE FFN forward pass (test infrastructure only).

Pages cited (no page has a title of its own; each is named by its address):
  csdn/6a919c0d  = devpress.csdn.net/awstech/6a919c0d2b83d06f0ec6f601.html
  csdn/6a462027  = devpress.csdn.net/awstech/6a46202710ee7a33f285c5a4.html
  csdn/6a462500  = devpress.csdn.net/awstech/6a46250010ee7a33f285d330.html
  aicoding/6a320eef = aicoding.csdn.net/6a320eef10ee7a33f27e52b3.html

Inputs are taken as their exact stored values (bf16 or fp32) upcast to fp64;
nothing is rounded in between. Library primitives used as single steps: numpy
matmul, numpy argmax, scipy's erf.

Readings where the pages are silent or disagree (each listed in the design notes):
  * inference routing is deterministic: no noise, temperature 1, no bias unless
    the workload adds one (csdn/6a462027 §3.1 says Gumbel noise is training-only);
  * top-k picks the k largest logits, the lower expert index winning a tie, and
    records them in descending order (slot 0 = largest);
  * the gate is the softmax probability itself, not renormalised over the k
    chosen experts (csdn/6a919c0d §2.2 step 4; aicoding/6a320eef §3.2);
  * the expert is d -> d_ff -> d with the erf form of GeLU and no biases
    (csdn/6a462027 §3.2);
  * within one expert, routed rows keep the row-major order of the (token, slot)
    assignments (the pages only ask for "a scatter").
"""
from __future__ import annotations

import math
from typing import Mapping, Optional, Sequence, Union

import numpy as np
from scipy.special import erf

ArrayLike = Union[np.ndarray, Sequence]


def router_logits(x: np.ndarray, w_r: np.ndarray, b_r: Optional[np.ndarray] = None) -> np.ndarray:
    """l[t, e] = sum_i x[t, i] * W_r[i, e] (+ b_r[e]).

    The router is one linear layer over the token's hidden state with one output
    per expert: csdn/6a919c0d §2.2 steps 1-2; aicoding/6a320eef §3.2 ("h x W_router",
    W_router is d x E).
    """
    logits = np.asarray(x, np.float64) @ np.asarray(w_r, np.float64)
    if b_r is not None:
        logits = logits + np.asarray(b_r, np.float64)[None, :]
    return logits


def softmax(logits: np.ndarray) -> np.ndarray:
    """p[t, e] = exp(l[t, e] - m_t) / sum_e' exp(l[t, e'] - m_t), m_t = max_e l[t, e].

    Softmax over all E router outputs (aicoding/6a320eef §3.2 "Softmax(logits)"),
    with the maximum subtracted first as csdn/6a919c0d §4.2 advises.
    """
    logits = np.asarray(logits, np.float64)
    m = logits.max(axis=1, keepdims=True)
    ex = np.exp(logits - m)
    return ex / ex.sum(axis=1, keepdims=True)


def topk_select(logits: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest logits per token, largest first, lower index first on ties.

    Deterministic top-k (csdn/6a919c0d §2.2 step 3: take the two experts with the
    highest confidence; csdn/6a462027 §3.1: deterministic at inference). Selecting
    on logits equals selecting on softmax probabilities because softmax is
    strictly increasing in each logit. Done as k rounds of "take the maximum and
    strike it out"; numpy's argmax returns the first (lowest) index among equal
    maxima, which is the tie rule.
    """
    work = np.array(logits, np.float64, copy=True)
    T, E = work.shape
    if not (1 <= k <= E):
        raise ValueError("topk_select: need 1 <= k <= E")
    idx = np.empty((T, k), np.int64)
    rows = np.arange(T)
    for j in range(k):
        e = np.argmax(work, axis=1)
        idx[:, j] = e
        work[rows, e] = -np.inf
    return idx


def gates_of(p: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """gate[t, j] = p[t, idx[t, j]]: the chosen experts' softmax probabilities, not renormalised.

    csdn/6a919c0d §2.2 step 4 (weights = each expert's confidence);
    aicoding/6a320eef §3.2 (weights = the corresponding p values) and its §3.1
    worked example (0.42 + 0.38 = 0.80).
    """
    return np.take_along_axis(np.asarray(p, np.float64), np.asarray(idx), axis=1)


def gates_renormalised(logits: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """w[t, j] = softmax over the k selected logits: exp(l[t, idx_j] - m) / sum_i exp(l[t, idx_i] - m).

    The gate variant of hotelren/2927663 §4.3 (top-k on the router logits, then a softmax over
    the k selected values only), with m the largest selected logit.
    """
    return softmax(np.take_along_axis(np.asarray(logits, np.float64), np.asarray(idx), axis=1))


def gelu(z: np.ndarray) -> np.ndarray:
    """GeLU(z) = z * Phi(z) = 0.5 * z * (1 + erf(z / sqrt(2))), the exact (erf) form.

    csdn/6a462027 §3.2 (GELU experts) and §4.2 (F.gelu, whose default is the erf form).
    """
    z = np.asarray(z, np.float64)
    return 0.5 * z * (1.0 + erf(z / math.sqrt(2.0)))


def expert_ffn(x_rows: np.ndarray, w1_e: np.ndarray, w2_e: np.ndarray) -> np.ndarray:
    """FFN_e(x) = GeLU(x W1_e) W2_e for a stack of token rows.

    Each expert is the same d -> d_ff -> d two-layer MLP with its own W1 [d, d_ff]
    and W2 [d_ff, d] (csdn/6a462027 §3.2; the stacked layout experts[E, d, d_ff]
    is its §4.2 sketch). Row r of the result depends on row r of x_rows only.
    """
    h = gelu(np.asarray(x_rows, np.float64) @ np.asarray(w1_e, np.float64))
    return h @ np.asarray(w2_e, np.float64)


def forward(x: np.ndarray, w_r: np.ndarray, w1: Union[np.ndarray, Mapping], w2: Union[np.ndarray, Mapping],
            k: int, b_r: Optional[np.ndarray] = None, renormalise: bool = False,
            cap: Optional[int] = None, reroute: Optional[int] = None) -> dict:
    """Forward pass of the layer for the tokens in x.

    out[t] = sum_{j=0..k-1} gate[t, j] * FFN_{idx[t, j]}(x[t]), summed in slot order.

    The routed tokens go only to their k experts (csdn/6a919c0d §2.2 steps 3-4;
    csdn/6a462027 §4.2 steps 4-7: route, run only the selected experts, sum the
    outputs weighted by the probabilities). ``w1[e]`` / ``w2[e]`` may be arrays
    or any mapping that yields expert e's matrices; only routed experts are read.
    With ``renormalise`` the gates are ``gates_renormalised`` instead of the raw probabilities;
    with a capacity ``cap`` the assignments ``kept_assignments`` drops contribute nothing, or, with
    ``reroute = R`` as well, the assignments go where ``reroute_assignments`` sends them within each
    token's R best experts (raw gates only).
    Returns the output and every routing intermediate.
    """
    x = np.asarray(x, np.float64)
    T, d = x.shape
    logits = router_logits(x, w_r, b_r)
    p = softmax(logits)
    idx = topk_select(logits, k)
    gate = gates_renormalised(logits, idx) if renormalise else gates_of(p, idx)
    if reroute is not None and cap is not None:
        if renormalise:
            raise ValueError("forward: rerouting uses the raw gates")
        ranked = topk_select(logits, reroute)
        idx, gate = reroute_assignments(ranked, gates_of(p, ranked), k, w_r.shape[1], cap)
        cap = None  # every remaining assignment has room
    y = np.zeros((k, T, d), np.float64)
    for j in range(k):
        for e in np.unique(idx[:, j]):
            if e < 0:
                continue
            rows = np.nonzero(idx[:, j] == e)[0]
            y[j, rows] = expert_ffn(x[rows], w1[int(e)], w2[int(e)])
    keep = (kept_assignments(idx, w_r.shape[1], cap) & (idx >= 0)).astype(np.float64)
    out = np.zeros((T, d), np.float64)
    for j in range(k):
        out = out + (keep[:, j] * gate[:, j])[:, None] * y[j]
    return {"out": out, "idx": idx, "gate": gate, "p": p, "logits": logits, "y": y, "keep": keep}


def dense_forward(x: np.ndarray, w_r: np.ndarray, w1, w2, k: int, b_r: Optional[np.ndarray] = None,
                  renormalise: bool = False) -> np.ndarray:
    """Brute force: evaluate all E experts on every token and weight them by mask_topk * p.

    The mask is the rank definition of top-k, independent of ``topk_select``:
    expert e is kept for token t when fewer than k experts beat it, where e' beats
    e if l[t, e'] > l[t, e], or l[t, e'] == l[t, e] and e' < e. Experts are summed
    in ascending index order. With ``renormalise`` each kept weight is divided by the sum of
    the kept probabilities.
    """
    x = np.asarray(x, np.float64)
    logits = router_logits(x, w_r, b_r)
    p = softmax(logits)
    T, E = logits.shape
    keep = np.zeros((T, E), np.float64)
    for e in range(E):
        le = logits[:, e:e + 1]
        beats = (logits > le) | ((logits == le) & (np.arange(E)[None, :] < e))
        keep[:, e] = (beats.sum(axis=1) < k).astype(np.float64)
    weight = keep * p
    if renormalise:
        weight = weight / weight.sum(axis=1, keepdims=True)
    out = np.zeros_like(x)
    for e in range(E):
        out = out + weight[:, e:e + 1] * expert_ffn(x, w1[e], w2[e])
    return out


def capacity(T: int, k: int, E: int, cf: float) -> int:
    """Expert capacity ceil(T*k/E * cf) (aicoding/6a320eef §3.2; its worked example: T=2048, k=2,
    E=128, cf=2.0 gives 64)."""
    return int(math.ceil(T * k / E * cf))


def kept_assignments(idx: np.ndarray, E: int, cap: Optional[int]) -> np.ndarray:
    """keep[t, j]: assignment (t, j) is among the first `cap` assignments of its expert in row-major
    (t, j) order. Reading of the capacity rule (aicoding/6a320eef §3.2: tokens beyond a full
    expert's capacity are diverted): the assignments past capacity are dropped."""
    idx = np.asarray(idx)
    T, k = idx.shape
    keep = np.ones((T, k), bool)
    if cap is None:
        return keep
    seen = np.zeros(E, np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            if e < 0:
                continue
            keep[t, j] = seen[e] < cap
            seen[e] += 1
    return keep


def reroute_assignments(rank_idx: np.ndarray, rank_p: np.ndarray, k: int, E: int, cap: int):
    """Expert capacity with rerouting: (final_idx [T, k], final_gate [T, k]).

    The capacity rule as aicoding/6a320eef §3.2 states it: when the expert the router chose already
    holds `cap` queued tokens, the token is rerouted to the next-best expert; csdn/6a919c0d §3.2
    describes the same as a retry that sends a dropped request to the next-best expert. Reading:
    the T*k assignments queue in row-major (t, j) order; slot j of token t goes to its chosen expert
    rank_idx[t, j] while that expert has room, and otherwise to the next expert in the token's
    ranking (rank_idx[t, k:], best first) that has room, each ranking entry being tried at most once
    per token; with none left the slot is dropped (final_idx -1, gate 0). The gate of a slot is the
    router probability of the expert that takes it (rank_p at that rank), so a rerouted slot is
    weighted by that expert's confidence (csdn/6a919c0d §2.2 step 4). rank_idx / rank_p: each token's
    R highest-ranked experts and their softmax probabilities, best first (R = E: the whole ranking).
    """
    rank_idx = np.asarray(rank_idx)
    rank_p = np.asarray(rank_p, np.float64)
    T, R = rank_idx.shape
    if not (1 <= k <= R):
        raise ValueError("reroute_assignments: need 1 <= k <= R")
    held = np.zeros(E, np.int64)
    final_idx = np.full((T, k), -1, np.int64)
    final_gate = np.zeros((T, k), np.float64)
    for t in range(T):
        nxt = k  # the next ranking entry this token may be rerouted to
        for j in range(k):
            e = int(rank_idx[t, j])
            if held[e] < cap:
                final_idx[t, j], final_gate[t, j] = e, rank_p[t, j]
                held[e] += 1
                continue
            while nxt < R:
                c = int(rank_idx[t, nxt])
                nxt += 1
                if held[c] < cap:
                    final_idx[t, j], final_gate[t, j] = c, rank_p[t, nxt - 1]
                    held[c] += 1
                    break
    return final_idx, final_gate


def dispatch(idx: np.ndarray, E: int, gate: Optional[np.ndarray] = None, cap: Optional[int] = None) -> dict:
    """Per-expert histogram, exclusive scan and stable permutation of the T*k assignments.

    counts[e] = #{(t, j) : idx[t, j] == e}; offsets = exclusive scan of counts
    (offsets[E] = T*k); the row of assignment (t, j) is offsets[e] plus the number
    of earlier assignments, in row-major (t, j) order, routed to the same e.
    perm_token[row] = t and row_gate[row] = gate[t, j] invert that map. This is
    the "scatter" of csdn/6a462027 §4.2 step 5 (group each expert's tokens), done
    as a counting sort. With a capacity, only the kept assignments (``kept_assignments``) get
    rows; a dropped one has row_of = -1, and so has an assignment whose index is already negative
    (dropped by ``reroute_assignments``).
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    keep = kept_assignments(idx, E, cap) & (idx >= 0)  # a negative index: an assignment already dropped
    counts = np.zeros(E, np.int64)
    for t in range(T):
        for j in range(k):
            if keep[t, j]:
                counts[idx[t, j]] += 1
    offsets = np.zeros(E + 1, np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    seen = np.zeros(E, np.int64)
    row_of = np.empty((T, k), np.int64)
    perm_token = np.full(T * k, -1, np.int64)
    row_gate = np.zeros(T * k, np.float64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            if not keep[t, j]:
                row_of[t, j] = -1
                continue
            r = offsets[e] + seen[e]
            seen[e] += 1
            row_of[t, j] = r
            perm_token[r] = t
            if gate is not None:
                row_gate[r] = gate[t, j]
    return {"counts": counts, "offsets": offsets, "row_of": row_of, "perm_token": perm_token,
            "row_gate": row_gate}


def expert_rows_ffn(x_perm: np.ndarray, offsets: np.ndarray, row_gate: np.ndarray, w1, w2,
                    rows: Optional[np.ndarray] = None) -> np.ndarray:
    """y_perm[r] = row_gate[r] * FFN_e(x_perm[r]) for the expert e whose range [offsets[e], offsets[e+1]) holds r.

    The per-expert FFN over only the routed rows (csdn/6a462027 §4.2 step 6, "in
    practice a grouped GEMM") with the gate applied to the expert's output
    (csdn/6a919c0d §2.2 step 4). ``rows`` restricts the evaluation to some rows.
    """
    x_perm = np.asarray(x_perm, np.float64)
    offsets = np.asarray(offsets)
    A = x_perm.shape[0]
    rows = np.arange(A) if rows is None else np.asarray(rows)
    expert_of_row = np.searchsorted(offsets, rows, side="right") - 1
    y = np.zeros((len(rows), x_perm.shape[1]), np.float64)
    for e in np.unique(expert_of_row):
        sel = np.nonzero(expert_of_row == e)[0]
        y[sel] = np.asarray(row_gate, np.float64)[rows[sel], None] * expert_ffn(x_perm[rows[sel]], w1[int(e)], w2[int(e)])
    return y


def _expert_of_rows(offsets: np.ndarray, rows: np.ndarray) -> np.ndarray:
    return np.searchsorted(np.asarray(offsets), rows, side="right") - 1


def expert_rows_up(x_perm: np.ndarray, offsets: np.ndarray, w1, rows: Optional[np.ndarray] = None) -> np.ndarray:
    """h[r] = GeLU(x_perm[r] W1_e) for the expert e whose range holds row r (first half of FFN_e).

    csdn/6a462027 §3.2 (the d -> d_ff GELU layer of each expert).
    """
    x_perm = np.asarray(x_perm, np.float64)
    rows = np.arange(x_perm.shape[0]) if rows is None else np.asarray(rows)
    eo = _expert_of_rows(offsets, rows)
    out = None
    for e in np.unique(eo):
        sel = np.nonzero(eo == e)[0]
        h = gelu(x_perm[rows[sel]] @ np.asarray(w1[int(e)], np.float64))
        if out is None:
            out = np.zeros((len(rows), h.shape[1]), np.float64)
        out[sel] = h
    return out if out is not None else np.zeros((0, 0))


def expert_rows_down(h: np.ndarray, offsets: np.ndarray, row_gate: np.ndarray, w2,
                     rows: Optional[np.ndarray] = None) -> np.ndarray:
    """y_perm[r] = row_gate[r] * (h[r] W2_e) (second half of FFN_e, weighted by the gate).

    csdn/6a462027 §3.2 (the d_ff -> d layer); csdn/6a919c0d §2.2 step 4 (weight = confidence).
    """
    h = np.asarray(h, np.float64)
    rows = np.arange(h.shape[0]) if rows is None else np.asarray(rows)
    eo = _expert_of_rows(offsets, rows)
    out = None
    for e in np.unique(eo):
        sel = np.nonzero(eo == e)[0]
        y = np.asarray(row_gate, np.float64)[rows[sel], None] * (h[rows[sel]] @ np.asarray(w2[int(e)], np.float64))
        if out is None:
            out = np.zeros((len(rows), y.shape[1]), np.float64)
        out[sel] = y
    return out if out is not None else np.zeros((0, 0))


def combine(y_perm: np.ndarray, row_of: np.ndarray) -> np.ndarray:
    """out[t] = sum_{j=0..k-1} y_perm[row_of[t, j]], summed in slot order.

    The weighted sum of the k expert outputs (csdn/6a462027 §4.2 step 7,
    "scatter_add"); the weights were already applied per row. A slot with row -1 (dropped at
    capacity) contributes nothing.
    """
    y_perm = np.asarray(y_perm, np.float64)
    row_of = np.asarray(row_of)
    T, k = row_of.shape
    out = np.zeros((T, y_perm.shape[1]), np.float64)
    for j in range(k):
        valid = row_of[:, j] >= 0
        out = out + np.where(valid[:, None], y_perm[np.where(valid, row_of[:, j], 0)], 0.0)
    return out


def routing_stats(logits: np.ndarray, idx: np.ndarray) -> dict:
    """Statistics of one batch's routing, reported beside the top-k selection.

    soft_load[e] = (1/T) sum_t p[t, e]: the expected share of expert e, the probabilities summed
        over the batch and divided by the number of tokens (csdn/6a462027 §4.2, its expert-load
        buffer);
    hard_load[e] = #{(t, j) : idx[t, j] = e} / (T k): the share of the T*k assignments that go
        to expert e;
    balance = sum_e (hard_load[e] - 1/E)^2: the load-balancing term without its weight lambda
        (aicoding/6a320eef §3.2; csdn/6a462027 §3.1). Reading: the formula's "tokens routed to
        expert i over all tokens" counts the T*k assignments, so the shares sum to one and the
        target 1/E is the balanced point;
    entropy = (1/T) sum_t -sum_e p[t, e] ln p[t, e], in nats: the mean entropy of the router's
        output distribution (aicoding/6a320eef §5.2, whose alert level lies between 0 and ln 128).
    The probabilities are the full softmax over the E experts, whatever the gates are.
    """
    l = np.asarray(logits, np.float64)
    idx = np.asarray(idx)
    T, E = l.shape
    k = idx.shape[1]
    p = softmax(l)
    soft = p.sum(axis=0) / T
    counts = np.zeros(E, np.int64)
    for e in idx.reshape(-1):
        counts[int(e)] += 1
    hard = counts / float(T * k)
    balance = float(np.sum((hard - 1.0 / E) ** 2))
    z = l - l.max(axis=1, keepdims=True)
    log_p = z - np.log(np.exp(z).sum(axis=1, keepdims=True))  # ln p, finite where p underflows
    entropy = float(np.mean(-(p * log_p).sum(axis=1)))
    return {"soft_load": soft, "hard_load": hard, "balance": balance, "entropy": entropy}


QBLOCK = 64


def quantize_blocks(w: np.ndarray, bits: int) -> dict:
    """Block quantisation of one weight matrix w [K, N] (csdn/6a462500 §4.3, 64 x 64 blocks with
    their own min / max; csdn/6a919c0d §2.3 and §3 for INT4 / INT8 expert weights).

    For each 64 x 64 block: scale = (max - min) / (2^bits - 1) and the code of w is
    round((w - min) / scale), so the block's min gets code 0 and its max the top code. Reading:
    the page's dequantisation adds the zero point back on top of codes that already had it
    removed, which loses the block minimum; here w is restored as min + code * scale. A block
    whose values are all equal has scale 0 and codes 0. The codes are integers decided by
    floating point, so they are decided in fp32 (the weights are bf16 or fp32, exact in fp32):
    fp32 subtraction and division, rounding half to even.
    """
    w32 = np.asarray(w, np.float32)
    K, N = w32.shape
    if K % QBLOCK or N % QBLOCK:
        raise ValueError("quantize_blocks: K and N must be multiples of 64")
    levels = np.float32(2 ** bits - 1)
    codes = np.zeros((K, N), np.uint8)
    scale = np.zeros((K // QBLOCK, N // QBLOCK), np.float32)
    wmin = np.zeros((K // QBLOCK, N // QBLOCK), np.float32)
    for bi in range(K // QBLOCK):
        for bj in range(N // QBLOCK):
            blk = w32[bi * QBLOCK:(bi + 1) * QBLOCK, bj * QBLOCK:(bj + 1) * QBLOCK]
            lo, hi = blk.min(), blk.max()
            s = np.float32(np.float32(hi - lo) / levels)
            scale[bi, bj], wmin[bi, bj] = s, lo
            if s > 0:
                q = np.rint((blk - lo) / s)  # float32 operands: fp32 subtraction and division
                codes[bi * QBLOCK:(bi + 1) * QBLOCK, bj * QBLOCK:(bj + 1) * QBLOCK] = q.astype(np.uint8)
    return {"codes": codes, "scale": scale, "min": wmin, "bits": bits}


def dequantize_blocks(q: Mapping) -> np.ndarray:
    """w_hat = min + code * scale per 64 x 64 block, in fp64 (the inverse map of quantize_blocks)."""
    codes = np.asarray(q["codes"], np.float64)
    s = np.repeat(np.repeat(np.asarray(q["scale"], np.float64), QBLOCK, 0), QBLOCK, 1)
    m = np.repeat(np.repeat(np.asarray(q["min"], np.float64), QBLOCK, 0), QBLOCK, 1)
    return m + codes * s


def packed_code_bytes(K: int, N: int, bits: int) -> int:
    """Bytes of the codes of a K x N matrix at `bits` per weight (csdn/6a462500 §4.3 counts a
    52,428,800-weight fp16 matrix as 104,857,600 bytes and its INT4 codes as 26,214,400)."""
    return K * N * bits // 8


def ambiguous_tokens(logits: np.ndarray, k: int, min_gap: float) -> np.ndarray:
    """Tokens whose top-(k+1) logits (top-k when E == k) have an adjacent gap below min_gap.

    Used by the input recipe to re-draw such tokens so that every routing index
    is decided by a margin far above fp32 rounding of the logits.
    """
    logits = np.asarray(logits, np.float64)
    T, E = logits.shape
    m = min(k + 1, E)
    top = -np.sort(-logits, axis=1)[:, :m]
    if m < 2:
        return np.zeros(0, np.int64)
    gaps = top[:, :-1] - top[:, 1:]
    return np.nonzero((gaps < min_gap).any(axis=1))[0]


def top_share(counts: np.ndarray, n: int) -> float:
    """Fraction of all assignments taken by the n most-loaded experts."""
    c = np.sort(np.asarray(counts, np.int64))[::-1]
    return float(c[:n].sum()) / float(c.sum())

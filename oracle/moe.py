"""fp64 CPU oracle of one MoE FFN layer forward pass (test infrastructure only).

The layer, step by step (the plain definition the method computes):
  1. logits  l[t,e] = sum_h x[t,h] * W_r[e,h] (+ b[e])
  2. select  the k largest logits of each token, descending, exact ties to
             the lower expert index
  3. weights softmax over the selected logits (== softmax over all E then
             renormalised over the selection), or sigmoid, normalised over
             the selection, times route_scale
  4. counts  per-expert token counts, offsets = exclusive prefix sum
  5. permute rows of expert e ordered by ascending token index
  6. experts h = silu(x W_g^T) * (x W_u^T);  y = h W_d^T, per expert
  7. combine out[t] = sum_j w[t,j] * y_{e_tj}(x[t]) + shared(x[t])

Every array is float64 except integer maps (int64).  Expert weights are
reached through a callable ``experts(e) -> (W_g, W_u, W_d)`` so that a
caller can hand over one expert at a time (the weights of a DeepSeek-V3
shaped layer do not fit in host memory as float64).
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):                      # torch tensor -> numpy
        a = a.detach().to("cpu")
        import torch
        if a.dtype in (torch.bfloat16, torch.float16):
            a = a.to(torch.float64)
        a = a.numpy()
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------- 1. logits
def router_logits(x, w_router, bias=None) -> np.ndarray:
    """Gated routing, first half: one score per (token, expert).

    AFD write-up, section 3 "Data-Flow Closed Loop" step 3 ("gated routing +
    expert computation").  The router is a linear map of the hidden state;
    an optional per-expert bias (the skewed workload's Zipf bias) is added
    to the logit and so moves both selection and weights.
    """
    lg = _f64(x) @ _f64(w_router).T
    if bias is not None:
        lg = lg + _f64(bias)[None, :]
    return lg


# ---------------------------------------------------------------- 2. select
def select_topk(logits, k: int) -> np.ndarray:
    """Indices of the k largest logits per token, in descending logit order,
    exact ties broken toward the lower expert index.

    ASAP section 5.1: 8 of 256 routed experts active per token.  Selection
    on logits equals selection on softmax or sigmoid scores, both strictly
    increasing.  A stable sort of the negated logits keeps equal logits in
    ascending index order.
    """
    lg = _f64(logits)
    order = np.argsort(-lg, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


# ---------------------------------------------------------------- 3. weights
def routing_weights(logits, ids, score: str, renormalize: bool = True,
                    route_scale: float = 1.0) -> np.ndarray:
    """Gate weight of each selected expert.

    softmax: w_j = exp(l_j - m) / sum_{j' in sel} exp(l_j' - m) when
             renormalised (otherwise the full softmax over all E experts,
             read at the selected positions);
    sigmoid: s_j = 1 / (1 + exp(-l_j)), w_j = s_j / sum_sel s (renormalised)
             or s_j;
    both then multiplied by route_scale.
    """
    lg = _f64(logits)
    ids = np.asarray(ids)
    sel = np.take_along_axis(lg, ids, axis=1)
    if score == "softmax":
        if renormalize:
            m = sel.max(axis=1, keepdims=True)
            p = np.exp(sel - m)
            w = p / p.sum(axis=1, keepdims=True)
        else:
            m = lg.max(axis=1, keepdims=True)
            p = np.exp(lg - m)
            w = np.take_along_axis(p / p.sum(axis=1, keepdims=True), ids, axis=1)
    elif score == "sigmoid":
        s = 1.0 / (1.0 + np.exp(-sel))
        w = s / s.sum(axis=1, keepdims=True) if renormalize else s
    else:
        raise ValueError(score)
    return w * route_scale


def softmax_all_then_renormalize(logits, ids) -> np.ndarray:
    """Second form of renormalised softmax routing (softmax over all E experts,
    then divide the selected probabilities by their sum).  Used only to pin
    routing_weights: both forms must agree."""
    lg = _f64(logits)
    m = lg.max(axis=1, keepdims=True)
    p = np.exp(lg - m)
    p = p / p.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(p, np.asarray(ids), axis=1)
    return sel / sel.sum(axis=1, keepdims=True)


# ---------------------------------------------------------------- 4. counts
def expert_histogram(ids, E: int):
    """Per-expert token counts (ASAP table 2: token counts per expert in the
    dispatch metadata) and their exclusive prefix sum (offsets[E] = T*k)."""
    ids = np.asarray(ids).reshape(-1)
    counts = np.zeros(E, dtype=np.int64)
    for e in ids:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    return counts, offsets


# ---------------------------------------------------------------- 5. permute
def permutation(ids, E: int):
    """Token-to-expert permutation that groups routed rows by expert.

    row(t, j) = offsets[e] + #{t' < t : e in ids[t']}   with e = ids[t, j]:
    rows of one expert in ascending token order (a reading: the pages give
    only the per-expert counts; a token selects an expert at most once, so
    the order does not depend on the slot j).
    Returns perm_token [T*k] (row -> token), perm_slot [T*k] (row -> j) and
    inv_row [T, k] ((t, j) -> row).
    """
    ids = np.asarray(ids)
    T, k = ids.shape
    _, offsets = expert_histogram(ids, E)
    fill = offsets[:-1].copy()
    perm_token = np.full(T * k, -1, dtype=np.int64)
    perm_slot = np.full(T * k, -1, dtype=np.int64)
    inv_row = np.full((T, k), -1, dtype=np.int64)
    for t in range(T):                      # ascending token index
        for j in range(k):
            e = ids[t, j]
            r = fill[e]
            fill[e] += 1
            perm_token[r] = t
            perm_slot[r] = j
            inv_row[t, j] = r
    return perm_token, perm_slot, inv_row


# ---------------------------------------------------------------- 6. experts
def silu(z) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z))."""
    z = _f64(z)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu_ffn(rows, w_gate, w_up, w_down) -> np.ndarray:
    """One expert on a block of rows: h = silu(rows W_g^T) * (rows W_u^T), y = h W_d^T.

    ASAP section 3.4.2: the expert computation is a matrix product with the
    hidden states on the left and the expert's weights on the right."""
    rows = _f64(rows)
    h = silu(rows @ _f64(w_gate).T) * (rows @ _f64(w_up).T)
    return h @ _f64(w_down).T


def grouped_ffn(x_perm, offsets, experts, row_weight=None) -> np.ndarray:
    """Grouped evaluation over the permuted rows: rows [offsets[e], offsets[e+1])
    go through expert e (ASAP section 3.4.2 grouped matrix multiplication;
    DWDP section 4.2: each expert's weights are a separate buffer, reached
    here through ``experts(e)``).  Each output row is multiplied by its
    routing weight when ``row_weight`` is given."""
    x_perm = _f64(x_perm)
    offsets = np.asarray(offsets)
    E = len(offsets) - 1
    out = np.zeros(x_perm.shape, dtype=np.float64)       # W_d maps I back to H
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b == a:
            continue
        wg, wu, wd = experts(e)
        out[a:b] = swiglu_ffn(x_perm[a:b], wg, wu, wd)
    if row_weight is not None:
        out = out * _f64(row_weight)[:, None]
    return out


# ---------------------------------------------------------------- 7. combine
def combine(y_perm, inv_row, shared_out=None) -> np.ndarray:
    """out[t] = sum_j y_perm[inv_row[t, j]] (+ shared_out[t]); rows already weighted."""
    y_perm = _f64(y_perm)
    inv_row = np.asarray(inv_row)
    T, k = inv_row.shape
    out = np.zeros((T, y_perm.shape[1]), dtype=np.float64)
    for j in range(k):
        out += y_perm[inv_row[:, j]]
    if shared_out is not None:
        out += _f64(shared_out)
    return out


# ---------------------------------------------------------------- whole layer
def route(x, w_router, bias, k, score, renormalize, route_scale):
    """Steps 1-3: (logits, ids, weights)."""
    lg = router_logits(x, w_router, bias)
    ids = select_topk(lg, k)
    w = routing_weights(lg, ids, score, renormalize, route_scale)
    return lg, ids, w


def moe_layer(x, w_router, bias, experts, shared, k, score, renormalize=True,
              route_scale=1.0):
    """The whole layer through the grouped (permuted) evaluation.

    ``shared`` is None or a tuple (W_sg, W_su, W_sd) of the always-on shared
    expert (ASAP section 5.1: 1 shared expert), weight 1.
    Returns a dict with every intermediate."""
    x = _f64(x)
    E = _f64(w_router).shape[0]
    lg, ids, w = route(x, w_router, bias, k, score, renormalize, route_scale)
    counts, offsets = expert_histogram(ids, E)
    perm_token, perm_slot, inv_row = permutation(ids, E)
    x_perm = x[perm_token]
    row_weight = w[perm_token, perm_slot]
    y_perm = grouped_ffn(x_perm, offsets, experts, row_weight)
    s = swiglu_ffn(x, *shared) if shared is not None else None
    out = combine(y_perm, inv_row, s)
    return dict(logits=lg, ids=ids, weights=w, counts=counts, offsets=offsets,
                perm_token=perm_token, perm_slot=perm_slot, inv_row=inv_row,
                x_perm=x_perm, row_weight=row_weight, y_perm=y_perm,
                shared_out=s, out=out)


def moe_tokens(x_rows, ids, w, experts, shared) -> np.ndarray:
    """Brute-force per-token evaluation, no permutation: for each token t and
    slot j, run expert ids[t, j] on x[t] alone and add w[t, j] times the
    result, then the shared expert.  Used on small inputs to pin the grouped
    path, and on sampled tokens of full-size layers."""
    x_rows = _f64(x_rows)
    ids = np.asarray(ids)
    w = _f64(w)
    T, k = ids.shape
    out = None
    cache = {}
    for t in range(T):
        acc = None
        for j in range(k):
            e = int(ids[t, j])
            if e not in cache:
                cache[e] = experts(e)
            y = swiglu_ffn(x_rows[t:t + 1], *cache[e])[0]
            acc = w[t, j] * y if acc is None else acc + w[t, j] * y
        if shared is not None:
            acc = acc + swiglu_ffn(x_rows[t:t + 1], *shared)[0]
        if out is None:
            out = np.zeros((T, acc.shape[0]), dtype=np.float64)
        out[t] = acc
    if out is None:
        out = np.zeros((0, x_rows.shape[1]), dtype=np.float64)
    return out


def moe_tokens_by_expert(x_rows, ids, w, expert_rows, shared_rows=None, map_fn=map):
    """The same per-token sum as ``moe_tokens``, evaluated expert by expert so
    that only one expert's weights need to exist at a time: for every expert e
    that some token selected, the rows of the tokens that selected it go
    through ``expert_rows(e, rows) -> [n, H]`` in one call, and each token adds
    w[t, j] times its row of the result; then ``shared_rows(x_rows)`` (the
    always-on shared expert, weight 1) when given.

    The expert functions are row-independent (each output row depends on its
    own input row only), so this equals the token-by-token sum.  ``map_fn``
    runs the per-expert calls; any function with the signature of the builtin
    ``map`` (which is the default) serves, e.g. a process pool's ``map``."""
    x_rows = _f64(x_rows)
    ids = np.asarray(ids)
    w = _f64(w)
    T = x_rows.shape[0]
    experts = sorted({int(e) for e in ids.reshape(-1)})
    where = [np.nonzero(ids == e) for e in experts]          # (tokens, slots) per expert
    ys = list(map_fn(expert_rows, experts, [x_rows[t] for t, _ in where]))
    out = None
    for (t, j), y in zip(where, ys):
        y = _f64(y)
        if out is None:
            out = np.zeros((T, y.shape[1]), dtype=np.float64)
        np.add.at(out, t, w[t, j][:, None] * y)
    if shared_rows is not None:
        s = _f64(shared_rows(x_rows))
        out = s.copy() if out is None else out + s
    if out is None:
        out = np.zeros((T, x_rows.shape[1]), dtype=np.float64)
    return out

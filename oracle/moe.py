"""Plain fp64 definition of the MoE layer forward, step by step.

TEST INFRASTRUCTURE ONLY (see the package docstring): slow, single-purpose, obviously
correct. Every array is numpy float64 / int64; library primitives (matmul, argsort,
bincount, cumsum, exp) serve as steps, with no blocking, fusion or reordering beyond the
definitions below.

Sources, cited by page title and section:
  [HF-EP]  Hugging Face Transformers docs, "Expert parallelism": sections
           "DistributedConfig", "Token dispatch", "How the sizes combine".
  [UL-EP]  Ultralytics glossary, "Expert Parallelism": sections "How tokens move between
           GPUs" (the four steps and the routing example) and "Load balancing and
           capacity".

Readings taken where the pages are silent:
  * the router score is the raw linear logit; the k largest are chosen, ties going to
    the lower expert id; the routing weights are a softmax over the k chosen logits;
  * each expert is a SwiGLU FFN  y = Wd (silu(Wg x) * (Wu x)), no biases;
  * capacity C = ceil(cf * N * k / E) per expert over the whole call; the first C pairs
    of an expert in token order are kept, the rest contribute zero, with no
    renormalisation of the surviving weights;
  * the mask-and-sum mode sums partition partial outputs in partition order.

Parity status: routing and load counts are pinned by the worked example's printed loads;
dispatch, expert math and combine are pinned by an independent dense brute force, a
library SwiGLU-MLP special case and a library softmax special case. The widened steps:
layer_backward / silu_grad by finite differences and torch autograd of a dense layer,
token_input_grads / expert_weight_grads against layer_backward, slot-major priority by a
loop and a cumulative-sum formulation, balance_stats by closed forms and torch.softmax,
tp_slices / tp_row_split_forward by their cover rule and the brute force (see tests/).
No function is left unpinned.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np


def _f64(a):
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------- step 1: routing
def router_logits(x, w_router, b_router=None):
    """[UL-EP] "How tokens move between GPUs", step 1 and its routing example: the
    router is a linear layer (weight [E, H] in nn.Linear's out x in layout, optional
    bias [E]) that scores every token against every expert.
    logits[t, e] = b[e] + sum_h x[t, h] * w_router[e, h]."""
    logits = _f64(x) @ _f64(w_router).T
    if b_router is not None:
        logits = logits + _f64(b_router)[None, :]
    return logits


def top_k_experts(logits, k):
    """[UL-EP] step 1: keep the k best-scoring experts of each token (the example takes
    top-k of the raw logits). Returned in descending score order; equal scores are
    ordered by lower expert id (the pages do not fix a tie rule; this is ours).
    A stable ascending sort of -logits realises exactly that order."""
    order = np.argsort(-_f64(logits), axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def routing_weights(logits, idx):
    """[UL-EP] step 4 weights expert outputs "by the router scores"; [HF-EP] "Token
    dispatch" combines "with the routing weights". Reading: softmax over the k chosen
    logits, w[t, j] = exp(l[t, idx[t, j]] - m_t) / sum_j' exp(l[t, idx[t, j']] - m_t),
    m_t the largest chosen logit."""
    chosen = np.take_along_axis(_f64(logits), idx, axis=1)
    m = chosen.max(axis=1, keepdims=True)
    e = np.exp(chosen - m)
    return e / e.sum(axis=1, keepdims=True)


def route(x, w_router, b_router, k):
    """Step 1 end to end: (logits, topk_idx [N,k] int64, topk_w [N,k] float64)."""
    logits = router_logits(x, w_router, b_router)
    idx = top_k_experts(logits, k)
    return logits, idx, routing_weights(logits, idx)


# ---------------------------------------------------------------- routing variants
def selection_scores(logits, selection_bias=None):
    """[UL-EP] "Load balancing and capacity", bias-based balancing: DeepSeek-V3 adds a
    per-expert bias to the router scores that only influences which experts are chosen.
    s[t, e] = logits[t, e] + beta[e]; the routing weights stay a softmax over the chosen
    experts' own logits (routing_weights(logits, idx))."""
    s = _f64(logits)
    if selection_bias is not None:
        s = s + _f64(selection_bias)[None, :]
    return s


def group_limited_top_k(scores, k, ep_size, group_limit):
    """[UL-EP] "Load balancing and capacity", last paragraph: DeepSeek-V3 sends each
    token to experts on at most 4 of its 8 nodes. Here the nodes are the ep_size
    partitions. The pages give no rule for which partitions; reading: a partition's score
    is the best score among its experts, the group_limit best partitions are kept (equal
    scores: lower partition id), and the k best experts inside them are chosen (equal
    scores: lower expert id). None or group_limit >= ep_size is plain top-k.
    Ordering key per token: (expert's partition is kept, score, -expert id), descending."""
    s = _f64(scores)
    N, E = s.shape
    if group_limit is None or group_limit >= ep_size:
        return top_k_experts(s, k)
    owner = expert_partition(np.arange(E), E, ep_size)
    part_best = np.stack([s[:, owner == p].max(axis=1) for p in range(ep_size)], axis=1)
    kept_parts = np.argsort(-part_best, axis=1, kind="stable")[:, :group_limit]
    allowed_part = np.zeros((N, ep_size), dtype=bool)
    allowed_part[np.arange(N)[:, None], kept_parts] = True
    allowed = allowed_part[:, owner]
    ids = np.broadcast_to(np.arange(E), (N, E))
    order = np.lexsort((ids, -s, ~allowed), axis=-1)
    return order[:, :k].astype(np.int64)


def route_variant(x, w_router, b_router, k, selection_bias=None, ep_size=1,
                  group_limit=None):
    """Step 1 with the routing variants: selection on logits + selection_bias, optionally
    limited to group_limit partitions; weights from the chosen experts' logits.
    Returns (logits, topk_idx, topk_w)."""
    logits = router_logits(x, w_router, b_router)
    s = selection_scores(logits, selection_bias)
    idx = group_limited_top_k(s, k, ep_size, group_limit)
    return logits, idx, routing_weights(logits, idx)


def update_selection_bias(selection_bias, routed_counts, num_tokens, k, gamma):
    """[UL-EP] bias-based balancing: after each step the bias of an overloaded expert is
    lowered and that of an idle one raised. Reading: overloaded / idle means above /
    below the equal share N*k/E of the step's routed assignments, and the step is a fixed
    gamma: beta_e - gamma, beta_e + gamma, or unchanged when the load equals the share.
    The comparison is exact in integers (count * E against N * k) and the bias is kept
    in float32, its storage type, so the update is computed in float32."""
    b = np.asarray(selection_bias, dtype=np.float32)
    c = np.asarray(routed_counts, dtype=np.int64)
    diff = c * b.shape[0] - int(num_tokens) * int(k)
    g = np.float32(gamma)
    return np.where(diff > 0, b - g, np.where(diff < 0, b + g, b)).astype(np.float32)


# ---------------------------------------------------------------- step 2: dispatch
def expert_partition(expert, num_experts, ep_size):
    """[HF-EP] "How the sizes combine": ep_size splits the expert list into ep_size
    contiguous blocks of num_experts/ep_size; [UL-EP] routing example: owner =
    expert // (num_experts // num_gpus)."""
    if num_experts % ep_size:
        raise ValueError("ep_size must divide the number of experts")
    return np.asarray(expert) // (num_experts // ep_size)


def load_counts(idx, num_experts, ep_size):
    """[UL-EP] routing example: bincount of the chosen expert ids (per-expert load) and
    of their owners (per-partition load)."""
    flat = np.asarray(idx).reshape(-1)
    per_expert = np.bincount(flat, minlength=num_experts).astype(np.int64)
    per_part = np.bincount(expert_partition(flat, num_experts, ep_size),
                           minlength=ep_size).astype(np.int64)
    return per_expert, per_part


def expert_capacity(capacity_factor, num_tokens, k, num_experts):
    """[UL-EP] "Load balancing and capacity": each expert takes at most capacity_factor
    times its equal share of the batch's assignments (e.g. 1.25). Reading:
    C = ceil(cf * N * k / E), evaluated in exact rational arithmetic on the float32
    value of cf (the library's argument type). None (no limit) when cf <= 0 or None."""
    if capacity_factor is None:
        return None
    cf = Fraction(float(np.float32(capacity_factor)))
    if cf <= 0:
        return None
    return math.ceil(cf * num_tokens * k / num_experts)


def dispatch_layout(idx, num_experts, ep_size, capacity=None, priority="token"):
    """[HF-EP] "Token dispatch": every (token, expert) pair is sent to the partition that
    owns the expert; [UL-EP] step 2. On one device the send buffer is grouped by expert,
    so each partition's rows are contiguous (experts are split contiguously).

    Pair p = t*k + j. Its rank is the number of earlier pairs (lower token index) routed
    to the same expert. With a capacity C, a pair is kept iff rank < C ([UL-EP] "Load
    balancing and capacity": overflow pairs skip that expert; reading: the first C in
    token order are kept).

    priority="slot" is the GShard-style variant: pairs are ranked slot-major -- every
    token's first choice before any token's second choice, then by token -- so p's
    priority key is j*N + t instead of t*k + j. The rank, the capacity test and the row
    order inside an expert's segment all follow that key.

    Returns dict of int64 arrays:
      routed_counts [E]    pairs routed to each expert before capacity
      counts        [E]    pairs kept
      expert_offsets[E+1]  exclusive prefix sum of counts (send-row start per expert)
      part_offsets  [P+1]  send-row start per partition = expert_offsets[p*E/P]
      slot_pos      [N*k]  send row of pair p, -1 when dropped
      perm          [A']   pair id held by send row r (inverse of slot_pos on kept pairs)
    """
    idx = np.asarray(idx)
    N, k = idx.shape
    E = num_experts
    flat = idx.reshape(-1).astype(np.int64)
    routed = np.bincount(flat, minlength=E).astype(np.int64)
    if priority == "token":
        order = np.arange(N * k)                       # pairs in priority order
    elif priority == "slot":
        order = np.arange(N * k).reshape(N, k).T.reshape(-1)
    else:
        raise ValueError(priority)
    # pairs grouped by expert; the stable sort keeps priority order inside a group
    by_expert = order[np.argsort(flat[order], kind="stable")]
    group_start = np.concatenate([[0], np.cumsum(routed)[:-1]])
    rank = np.empty(N * k, dtype=np.int64)
    rank[by_expert] = np.arange(N * k) - group_start[flat[by_expert]]
    keep = np.ones(N * k, dtype=bool) if capacity is None else rank < capacity
    counts = np.bincount(flat[keep], minlength=E).astype(np.int64)
    expert_offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    slot_pos = np.where(keep, expert_offsets[flat] + rank, -1).astype(np.int64)
    perm = np.empty(int(expert_offsets[-1]), dtype=np.int64)
    perm[slot_pos[keep]] = np.nonzero(keep)[0]
    part_offsets = expert_offsets[np.arange(ep_size + 1) * (E // ep_size)]
    return dict(routed_counts=routed, counts=counts, expert_offsets=expert_offsets,
                part_offsets=part_offsets, slot_pos=slot_pos, perm=perm)


def permute(x, perm, k):
    """[UL-EP] step 2 (the all-to-all that carries each token's hidden state to its
    experts' owner), on one device: send row r holds the hidden state of token
    perm[r] // k."""
    return _f64(x)[np.asarray(perm, dtype=np.int64) // k]


# ---------------------------------------------------------------- step 3: experts
def silu(z):
    """silu(z) = z * sigmoid(z) = z / (1 + exp(-z))."""
    z = _f64(z)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu_expert(rows, w_gate, w_up, w_down):
    """One expert's feed-forward network on its received rows ([UL-EP] step 3). The
    pages never define the expert network; reading: SwiGLU without biases,
    y = W_down (silu(W_gate x) * (W_up x)), weights in nn.Linear layout
    (w_gate, w_up [I, H]; w_down [H, I])."""
    rows = _f64(rows)
    g = rows @ _f64(w_gate).T
    u = rows @ _f64(w_up).T
    return (silu(g) * u) @ _f64(w_down).T


def expert_outputs(send, expert_offsets, w_gate, w_up, w_down,
                   expert_begin=0, expert_end=None):
    """[UL-EP] step 3 / [HF-EP] "Token dispatch": each partition runs its local experts
    on what it received. Send rows of expert e are [expert_offsets[e],
    expert_offsets[e+1]). Rows of experts outside [expert_begin, expert_end) stay 0."""
    send = _f64(send)
    E = len(expert_offsets) - 1
    expert_end = E if expert_end is None else expert_end
    y = np.zeros((send.shape[0], np.shape(w_down)[1]), dtype=np.float64)
    for e in range(expert_begin, expert_end):
        a, b = int(expert_offsets[e]), int(expert_offsets[e + 1])
        if b > a:
            y[a:b] = swiglu_expert(send[a:b], w_gate[e], w_up[e], w_down[e])
    return y


# ---------------------------------------------------------------- step 4: combine
def combine_dispatch(y_send, slot_pos, topk_w, num_tokens, k):
    """[UL-EP] step 4 / [HF-EP] "Token dispatch": expert outputs return to their token
    and are summed weighted by the routing weights. out[t] = sum over kept slots j, in
    slot order, of w[t, j] * y[slot_pos[t*k + j]]. A dropped pair adds nothing (the
    token's residual path lives outside the layer)."""
    y_send = _f64(y_send)
    out = np.zeros((num_tokens, y_send.shape[1]), dtype=np.float64)
    sp = np.asarray(slot_pos).reshape(num_tokens, k)
    w = _f64(topk_w).reshape(num_tokens, k)
    for j in range(k):
        kept = sp[:, j] >= 0
        out[kept] += w[kept, j, None] * y_send[sp[kept, j]]
    return out


def combine_mask_sum(y_send, slot_pos, topk_idx, topk_w, num_experts, ep_size):
    """[HF-EP] "DistributedConfig" / plan rules "ep_router" + "moe_tp_experts": each
    partition masks the experts it does not own, computes its local ones, and an
    all-reduce sums the partitions' outputs. Here partial[p, t] = sum over kept slots j
    of token t whose expert lives in partition p (slot order) of w[t,j] * y, and
    out = partial[0] + partial[1] + ... in partition order. Returns (partials, out)."""
    y_send = _f64(y_send)
    idx = np.asarray(topk_idx)
    N, k = idx.shape
    sp = np.asarray(slot_pos).reshape(N, k)
    w = _f64(topk_w).reshape(N, k)
    owner = expert_partition(idx, num_experts, ep_size)
    partials = np.zeros((ep_size, N, y_send.shape[1]), dtype=np.float64)
    for p in range(ep_size):
        for j in range(k):
            sel = (sp[:, j] >= 0) & (owner[:, j] == p)
            partials[p, sel] += w[sel, j, None] * y_send[sp[sel, j]]
    out = np.zeros((N, y_send.shape[1]), dtype=np.float64)
    for p in range(ep_size):
        out += partials[p]
    return partials, out


# ---------------------------------------------------------------- the whole layer
def layer_forward(x, w_router, b_router, w_gate, w_up, w_down, top_k, ep_size,
                  capacity_factor=None, mode="dispatch", selection_bias=None,
                  group_limit=None, capacity_priority="token"):
    """Route -> dispatch -> local experts -> weighted combine, all in fp64.
    Returns a dict with every intermediate (logits, topk_idx, topk_w, the dispatch
    layout, send, y_send, out and, in mask mode, partials)."""
    x = _f64(x)
    N = x.shape[0]
    E = np.shape(w_router)[0]
    logits, idx, w = route_variant(x, w_router, b_router, top_k, selection_bias, ep_size,
                                   group_limit)
    C = expert_capacity(capacity_factor, N, top_k, E)
    lay = dispatch_layout(idx, E, ep_size, C, capacity_priority)
    send = permute(x, lay["perm"], top_k)
    y_send = expert_outputs(send, lay["expert_offsets"], w_gate, w_up, w_down)
    res = dict(logits=logits, topk_idx=idx, topk_w=w, capacity=C, send=send,
               y_send=y_send, **lay)
    if mode == "dispatch":
        res["out"] = combine_dispatch(y_send, lay["slot_pos"], w, N, top_k)
    elif mode == "mask_sum":
        res["partials"], res["out"] = combine_mask_sum(y_send, lay["slot_pos"], idx, w,
                                                       E, ep_size)
    else:
        raise ValueError(mode)
    return res


def balance_stats(logits, routed_counts, num_tokens, k):
    """Router load statistics ([UL-EP] "Load balancing and capacity": an auxiliary loss
    term pushes the router towards an even spread of tokens; the pages name no formula,
    so only its two usual ingredients are computed, not a loss):
      load_frac[e] = routed_counts[e] / (N * k), the share of the step's routed pairs
                     that chose expert e (before capacity);
      prob_mean[e] = mean over tokens of softmax(logits[t])[e], the router's average
                     probability for e over all E experts.
    logits are the raw router logits (bias included, selection bias not)."""
    lg = _f64(logits)
    N = lg.shape[0]
    load = _f64(routed_counts) / float(num_tokens * k) if num_tokens * k else \
        np.zeros(np.shape(routed_counts))
    if N == 0:
        return dict(load_frac=load, prob_mean=np.zeros(lg.shape[1]))
    m = lg.max(axis=1, keepdims=True)
    ex = np.exp(lg - m)
    prob = ex / ex.sum(axis=1, keepdims=True)
    return dict(load_frac=load, prob_mean=prob.sum(axis=0) / N)


def tp_slices(num_tokens, tp_size):
    """[HF-EP] "With tensor parallelism": the ranks of a TP group hold the same batch
    and each dispatches a disjoint 1/tp_size of its tokens; slices may be uneven or
    empty. Reading: contiguous slices, the first N mod tp one token longer
    (numpy.array_split's rule). Returns [(begin, end)] per TP rank."""
    q, r = divmod(num_tokens, tp_size)
    out, b = [], 0
    for s in range(tp_size):
        n = q + (1 if s < r else 0)
        out.append((b, b + n))
        b += n
    return out


def tp_row_split_forward(x, w_router, b_router, w_gate, w_up, w_down, top_k, ep_size,
                         tp_size, capacity_factor=None, mode="dispatch"):
    """[HF-EP] "With tensor parallelism": TP rank s dispatches only its slice of the
    shared batch, its results come back to it, and an all-reduce over the TP group of
    the zero-padded slice outputs restores the full output. Each slice is a layer call
    of its own over its tokens (reading: a capacity limit is therefore taken over the
    slice's tokens). padded[s] holds slice s's rows and zeros elsewhere;
    out = padded[0] + padded[1] + ... in rank order. Returns (padded, out)."""
    x = _f64(x)
    N, H = x.shape
    padded = np.zeros((tp_size, N, H))
    for s, (b, e) in enumerate(tp_slices(N, tp_size)):
        if e > b:
            padded[s, b:e] = layer_forward(x[b:e], w_router, b_router, w_gate, w_up, w_down,
                                           top_k, ep_size, capacity_factor, mode)["out"]
    out = np.zeros((N, H))
    for s in range(tp_size):
        out += padded[s]
    return padded, out


def token_outputs(x_rows, idx_rows, w_rows, keep_rows, expert_weights):
    """Layer output of a few tokens, one at a time (for sampled checks at full size).

    x_rows [n, H]; idx_rows / w_rows / keep_rows [n, k] (keep from the full-batch
    dispatch layout, since capacity depends on every token). expert_weights(e) returns
    (w_gate[e], w_up[e], w_down[e]). out[i] = sum_j keep * w * FFN_idx(x_i), in j order.
    """
    x_rows = _f64(x_rows)
    n, k = np.shape(idx_rows)
    needed = sorted({int(idx_rows[i][j]) for i in range(n) for j in range(k)
                     if keep_rows[i][j]})
    y = {}
    for e in needed:
        wg, wu, wd = expert_weights(e)
        for i in range(n):
            for j in range(k):
                if keep_rows[i][j] and int(idx_rows[i][j]) == e:
                    y[(i, j)] = swiglu_expert(x_rows[i:i + 1], wg, wu, wd)[0]
    out = np.zeros((n, np.shape(x_rows)[1]), dtype=np.float64)
    for i in range(n):
        for j in range(k):
            if keep_rows[i][j]:
                out[i] += float(w_rows[i][j]) * y[(i, j)]
    return out


# ---------------------------------------------------------------- backward of the layer
def silu_grad(z):
    """d silu(z) / dz = sigmoid(z) * (1 + z * (1 - sigmoid(z)))."""
    z = _f64(z)
    with np.errstate(over="ignore"):
        sig = 1.0 / (1.0 + np.exp(-z))
    return sig * (1.0 + z * (1.0 - sig))


def layer_backward(x, w_router, b_router, w_gate, w_up, w_down, top_k, ep_size, dout,
                   capacity_factor=None, selection_bias=None, group_limit=None,
                   capacity_priority="token"):
    """Gradients of the layer output (dispatch rule; the mask-and-sum rule computes the
    same output) with respect to its inputs and weights, for the upstream gradient dout
    [N, H]: the chain rule through each step of layer_forward, in fp64. The expert
    selection and the capacity drops are piecewise constant and carry no gradient; a
    dropped pair's output is zero but its routing weight stays in the softmax, so the
    weights' Jacobian still couples it ([UL-EP] "Load balancing and capacity": no
    renormalisation). An expert's weight gradient sums over every token it received, as
    the pages sum an expert's gradient over the batches of its group ([HF-EP] "How the
    sizes combine").

    out[t] = sum_j keep[t,j] * w[t,j] * y_{e_tj}(x_t),
    y_e(x) = Wd_e (silu(Wg_e x) * (Wu_e x)),  w = softmax over the k chosen logits.
    Returns dict dx [N,H], dw_router [E,H], db_router [E], dw_gate / dw_up [E,I,H],
    dw_down [E,H,I]."""
    x = _f64(x)
    dout = _f64(dout)
    N, H = x.shape
    E = np.shape(w_router)[0]
    k = top_k
    fwd = layer_forward(x, w_router, b_router, w_gate, w_up, w_down, k, ep_size,
                        capacity_factor, "dispatch", selection_bias, group_limit,
                        capacity_priority)
    idx, w, sp = fwd["topk_idx"], fwd["topk_w"], np.asarray(fwd["slot_pos"]).reshape(N, k)
    dx = np.zeros_like(x)
    dwg = np.zeros(np.shape(w_gate))
    dwu = np.zeros(np.shape(w_up))
    dwd = np.zeros(np.shape(w_down))
    dweight = np.zeros((N, k))          # d out / d w[t, j] contracted with dout
    for e in range(E):
        pairs = [(t, j) for t in range(N) for j in range(k) if idx[t, j] == e and sp[t, j] >= 0]
        if not pairs:
            continue
        ts = np.array([t for t, _ in pairs])
        js = np.array([j for _, j in pairs])
        xe = x[ts]                                   # [n, H]
        g = xe @ _f64(w_gate[e]).T                   # [n, I]
        u = xe @ _f64(w_up[e]).T
        a = silu(g) * u
        y = a @ _f64(w_down[e]).T                    # [n, H]
        dy = w[ts, js][:, None] * dout[ts]           # d loss / d y
        dweight[ts, js] = np.sum(dout[ts] * y, axis=1)
        da = dy @ _f64(w_down[e])                    # [n, I]
        dwd[e] += dy.T @ a
        dg = da * u * silu_grad(g)
        du = da * silu(g)
        dwg[e] += dg.T @ xe
        dwu[e] += du.T @ xe
        np.add.at(dx, ts, dg @ _f64(w_gate[e]) + du @ _f64(w_up[e]))
    # softmax over the chosen logits: dl_c = w_c (dweight_c - sum_c' w_c' dweight_c')
    dl_chosen = w * (dweight - np.sum(w * dweight, axis=1, keepdims=True))
    dlogits = np.zeros((N, E))
    np.put_along_axis(dlogits, idx, dl_chosen, axis=1)
    dx += dlogits @ _f64(w_router)
    dwr = dlogits.T @ x
    dbr = dlogits.sum(axis=0)
    return dict(dx=dx, dw_router=dwr, db_router=dbr, dw_gate=dwg, dw_up=dwu, dw_down=dwd,
                dlogits=dlogits, forward=fwd)


def token_input_grads(x_rows, dout_rows, idx_rows, w_rows, keep_rows, w_router, expert_weights):
    """dx of a few tokens, one at a time (for sampled checks at full size), by the same
    chain rule as layer_backward with the batch's routing and keep decisions given.
    Per token: y_j = FFN_{e_j}(x) for kept pairs, dweight_j = <dout, y_j> (0 if dropped),
    dl_j = w_j (dweight_j - sum_j' w_j' dweight_j'), and
    dx = sum_j kept [W_g^T dg_j + W_u^T du_j] + sum_j dl_j W_r[e_j], with
    dg_j = w_j (W_d^T dout) * u * silu'(g), du_j = w_j (W_d^T dout) * silu(g).
    expert_weights(e) returns (w_gate[e], w_up[e], w_down[e])."""
    x_rows = _f64(x_rows)
    dout_rows = _f64(dout_rows)
    n, k = np.shape(idx_rows)
    wr = _f64(w_router)
    out = np.zeros_like(x_rows)
    for i in range(n):
        x, dy = x_rows[i], dout_rows[i]
        dweight = np.zeros(k)
        dx = np.zeros_like(x)
        for j in range(k):
            if not keep_rows[i][j]:
                continue
            wg, wu, wd = (_f64(a) for a in expert_weights(int(idx_rows[i][j])))
            g, u = wg @ x, wu @ x
            y = wd @ (silu(g) * u)
            dweight[j] = float(dy @ y)
            da = float(w_rows[i][j]) * (wd.T @ dy)
            dx += wg.T @ (da * u * silu_grad(g)) + wu.T @ (da * silu(g))
        w = _f64(w_rows[i])
        dl = w * (dweight - float(np.sum(w * dweight)))
        for j in range(k):
            dx += dl[j] * wr[int(idx_rows[i][j])]
        out[i] = dx
    return out


def expert_weight_grads(x_rows, dout_rows, w_rows, w_gate, w_up, w_down):
    """Weight gradients of one expert from all its kept rows (send order): x_rows,
    dout_rows [n, H] of the rows' tokens, w_rows [n] their routing weights.
    dW_down = sum_r (w_r dout_r) a_r^T, dW_gate = sum_r dg_r x_r^T, dW_up = sum_r du_r x_r^T
    with a = silu(g) * u, da = W_d^T (w dout), dg = da * u * silu'(g), du = da * silu(g).
    Returns (dw_gate [I, H], dw_up [I, H], dw_down [H, I])."""
    X = _f64(x_rows)
    dY = _f64(dout_rows) * _f64(w_rows)[:, None]
    wg, wu, wd = _f64(w_gate), _f64(w_up), _f64(w_down)
    G, U = X @ wg.T, X @ wu.T
    A = silu(G) * U
    dA = dY @ wd
    dG = dA * U * silu_grad(G)
    dU = dA * silu(G)
    return dG.T @ X, dU.T @ X, dY.T @ A

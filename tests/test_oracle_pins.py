"""Pins of the fp64 oracle against things other than itself.

* the worked routing example's printed loads (tests/golden/ul_ep_routing_example.txt);
* an independent dense brute force (explicit index sums, a different top-k rule
  formulation, softmax-then-renormalise weights, capacity by counting earlier tokens)
  on tiny inputs, in both layer modes;
* library special cases: one expert with k=1 is a SwiGLU MLP (torch.nn.functional);
  k=E gives the full softmax (scipy);
* invariants the pages state (loads sum to N*k, owner = expert // (E/ep_size), ...);
* planted mistakes in the oracle must make a pin fail.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import oracle.moe as om
import workloads
from conftest import read_golden


# ------------------------------------------------------------------ helpers
def tiny_inputs(seed, N, H, I, E, grid=None, bias=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((N, H))
    wr = rng.uniform(-1, 1, (E, H)) / math.sqrt(H)
    b = rng.uniform(-1, 1, E) / math.sqrt(H) if bias else None
    if grid is not None:          # coarse grid -> genuine ties between logits
        x = np.round(x / grid) * grid
        wr = np.round(wr / grid) * grid
        if b is not None:
            b = np.round(b / grid) * grid
    wg = rng.standard_normal((E, I, H)) * 0.3
    wu = rng.standard_normal((E, I, H)) * 0.3
    wd = rng.standard_normal((E, H, I)) * 0.3
    return x, wr, b, wg, wu, wd


def brute_force_layer(x, wr, b, wg, wu, wd, k, ep_size, capacity, sel_bias=None,
                      group_limit=None):
    """Dense evaluation: every expert on every token, masked to the kept top-k.
    Written independently of the oracle: explicit subscripts, 'fewer than k experts
    beat it' selection, full softmax renormalised over the selection, capacity by
    counting earlier tokens that selected the same expert. Routing variants: selection
    on S = L + sel_bias (weights still from L); with a group limit M a partition is
    eligible iff fewer than M partitions beat its best score, and an expert is selected
    iff its partition is eligible and fewer than k eligible experts beat it."""
    N, H = x.shape
    E = wr.shape[0]
    L = np.einsum("th,eh->te", x, wr)
    if b is not None:
        L = L + b[None, :]
    S = L if sel_bias is None else L + np.asarray(sel_bias, dtype=np.float64)[None, :]
    owner = np.arange(E) // (E // ep_size)
    eligible = np.ones((N, E), dtype=bool)
    if group_limit is not None:
        for t in range(N):
            best = [max(S[t, e] for e in range(E) if owner[e] == p) for p in range(ep_size)]
            for e in range(E):
                p = owner[e]
                beaten = sum(1 for q in range(ep_size)
                             if best[q] > best[p] or (best[q] == best[p] and q < p))
                eligible[t, e] = beaten < group_limit
    selected = np.zeros((N, E), dtype=bool)
    for t in range(N):
        for e in range(E):
            beaten_by = sum(1 for e2 in range(E) if eligible[t, e2] and
                            (S[t, e2] > S[t, e] or (S[t, e2] == S[t, e] and e2 < e)))
            selected[t, e] = eligible[t, e] and beaten_by < k
    full = scipy.special.softmax(L, axis=1)
    weight = np.where(selected, full, 0.0)
    weight = weight / weight.sum(axis=1, keepdims=True)
    kept = selected.copy()
    if capacity is not None:
        for e in range(E):
            for t in range(N):
                earlier = int(selected[:t, e].sum())
                kept[t, e] = selected[t, e] and earlier < capacity
    dense_y = np.zeros((E, N, H))
    for e in range(E):
        g = np.einsum("ih,th->ti", wg[e], x)
        u = np.einsum("ih,th->ti", wu[e], x)
        h = g / (1.0 + np.exp(-g)) * u
        dense_y[e] = np.einsum("hi,ti->th", wd[e], h)
    out = np.einsum("te,eth->th", np.where(kept, weight, 0.0), dense_y)
    per_part = np.zeros((ep_size, N, H))
    owner = np.arange(E) // (E // ep_size)
    for e in range(E):
        per_part[owner[e]] += np.where(kept[:, e], weight[:, e], 0.0)[:, None] * dense_y[e]
    return dict(selected=selected, kept=kept, weight=weight, out=out, partials=per_part,
                logits=L)


def rel_err(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


TINY_CASES = [
    # seed, N, H, I, E, k, P, cf, grid
    (1, 13, 8, 5, 4, 2, 2, None, None),
    (2, 16, 12, 6, 6, 3, 3, 1.0, None),
    (3, 9, 8, 4, 8, 2, 4, 0.5, 0.25),      # coarse grid: ties
    (4, 20, 6, 3, 5, 5, 5, None, None),    # k = E
    (5, 7, 10, 7, 3, 1, 1, 0.01, None),    # capacity 1 per expert
    (6, 1, 8, 4, 4, 2, 2, None, None),     # a single token
    (7, 18, 8, 8, 8, 2, 8, 1.25, 0.5),     # I == H (catches transposed weights), ties
    (8, 12, 4, 6, 2, 1, 2, 2.0, None),
]


def _oracle_with_bf(case, mode="dispatch"):
    seed, N, H, I, E, k, P, cf, grid = case
    x, wr, b, wg, wu, wd = tiny_inputs(seed, N, H, I, E, grid)
    res = oracle.layer_forward(x, wr, b, wg, wu, wd, k, P, cf, mode)
    bf = brute_force_layer(x, wr, b, wg, wu, wd, k, P, res["capacity"])
    return res, bf


# ------------------------------------------------------------------ worked example
def test_routing_example_loads_match_printed_values():
    gold = read_golden("ul_ep_routing_example.txt")
    x, w, b = workloads.snippet_inputs()
    _, idx, _ = oracle.route(x.numpy(), w.numpy(), b.numpy(), 2)
    per_expert, per_part = oracle.load_counts(idx, 8, 4)
    assert per_expert.sum() == gold["total_assignments"] == per_part.sum()
    assert per_expert.min() == gold["expert_load_min"]
    assert per_expert.max() == gold["expert_load_max"]
    assert gold["total_assignments"] // 8 == gold["equal_share"]
    assert per_part.min() == gold["partition_load_min"]
    assert per_part.max() == gold["partition_load_max"]


# ------------------------------------------------------------------ brute force
@pytest.mark.parametrize("case", TINY_CASES)
@pytest.mark.parametrize("mode", ["dispatch", "mask_sum"])
def test_oracle_equals_dense_brute_force(case, mode):
    res, bf = _oracle_with_bf(case, mode)
    N, k = res["topk_idx"].shape
    sel = np.zeros_like(bf["selected"])
    np.put_along_axis(sel, res["topk_idx"], True, axis=1)
    assert np.array_equal(sel, bf["selected"])
    kept = np.zeros_like(sel)
    sp = res["slot_pos"].reshape(N, k)
    for t in range(N):
        for j in range(k):
            if sp[t, j] >= 0:
                kept[t, res["topk_idx"][t, j]] = True
    assert np.array_equal(kept, bf["kept"])
    w_bf = np.take_along_axis(bf["weight"], res["topk_idx"], axis=1)
    assert np.allclose(res["topk_w"], w_bf, rtol=1e-13, atol=1e-15)
    assert rel_err(res["out"], bf["out"]) < 1e-12
    if mode == "mask_sum":
        assert rel_err(res["partials"], bf["partials"]) < 1e-12


@pytest.mark.parametrize("case", TINY_CASES)
def test_dispatch_mode_equals_mask_sum_mode(case):
    seed, N, H, I, E, k, P, cf, grid = case
    x, wr, b, wg, wu, wd = tiny_inputs(seed, N, H, I, E, grid)
    a = oracle.layer_forward(x, wr, b, wg, wu, wd, k, P, cf, "dispatch")
    m = oracle.layer_forward(x, wr, b, wg, wu, wd, k, P, cf, "mask_sum")
    assert rel_err(m["out"], a["out"]) < 1e-12


# ------------------------------------------------------------------ library special cases
def test_single_expert_top1_is_swiglu_mlp():
    x, wr, b, wg, wu, wd = tiny_inputs(11, 24, 16, 12, 1)
    res = oracle.layer_forward(x, wr, b, wg, wu, wd, 1, 1)
    X = torch.from_numpy(x)
    ref = (torch.nn.functional.silu(X @ torch.from_numpy(wg[0]).T)
           * (X @ torch.from_numpy(wu[0]).T)) @ torch.from_numpy(wd[0]).T
    assert np.allclose(res["topk_w"], 1.0)
    assert rel_err(res["out"], ref.numpy()) < 1e-13


def test_k_equals_e_weights_are_full_softmax():
    x, wr, b, *_ = tiny_inputs(12, 40, 16, 4, 7)
    logits, idx, w = oracle.route(x, wr, b, 7)
    full = scipy.special.softmax(logits, axis=1)
    assert np.allclose(w, np.take_along_axis(full, idx, axis=1), rtol=1e-13, atol=1e-16)
    assert np.allclose(w.sum(axis=1), 1.0)


def test_topk_matches_torch_topk_on_distinct_scores():
    rng = np.random.default_rng(3)
    L = rng.standard_normal((200, 64))
    idx = oracle.top_k_experts(L, 8)
    tv, ti = torch.topk(torch.from_numpy(L), 8, dim=1, sorted=True)
    assert np.array_equal(idx, ti.numpy())


def test_topk_ties_go_to_lower_expert_id():
    L = np.array([[1.0, 2.0, 2.0, 0.5, 2.0],
                  [0.0, 0.0, 0.0, 0.0, 0.0],
                  [3.0, -1.0, 3.0, 3.0, -1.0]])
    assert oracle.top_k_experts(L, 2).tolist() == [[1, 2], [0, 1], [0, 2]]
    assert oracle.top_k_experts(L, 4).tolist() == [[1, 2, 4, 0], [0, 1, 2, 3], [0, 2, 3, 1]]


def test_routing_weights_closed_form_two_experts():
    # softmax of two logits is the logistic function of their difference
    L = np.array([[0.3, -1.2, 2.0, 0.0]])
    idx = oracle.top_k_experts(L, 2)
    w = oracle.routing_weights(L, idx)
    d = 2.0 - 0.3
    assert idx.tolist() == [[2, 0]]
    assert abs(w[0, 0] - 1 / (1 + math.exp(-d))) < 1e-15
    assert abs(w[0, 1] - 1 / (1 + math.exp(d))) < 1e-15


def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(1.0) - 1 / (1 + math.exp(-1))) < 1e-16
    assert abs(oracle.silu(-40.0)) < 1e-15
    assert oracle.silu(-1000.0) == 0.0
    assert oracle.silu(1000.0) == 1000.0


# ------------------------------------------------------------------ capacity
def test_capacity_values():
    # the skewed workload: ceil(1.25 * 32768 * 8 / 64) = 5120
    assert oracle.expert_capacity(1.25, 32768, 8, 64) == 5120
    assert oracle.expert_capacity(None, 10, 2, 4) is None
    assert oracle.expert_capacity(0.0, 10, 2, 4) is None
    assert oracle.expert_capacity(-1.0, 10, 2, 4) is None
    assert oracle.expert_capacity(1.0, 10, 2, 4) == 5
    assert oracle.expert_capacity(1.0, 10, 3, 4) == 8       # 7.5 -> 8
    assert oracle.expert_capacity(1e-6, 10, 3, 4) == 1
    # 0.1 is not a binary fraction: float32(0.1) * 40 / 4 is just above 1
    assert oracle.expert_capacity(0.1, 40, 1, 4) == 2


def test_capacity_keeps_first_tokens_in_token_order():
    # every token picks experts (0, 1): expert 0 and 1 keep tokens 0..C-1 only
    idx = np.array([[0, 1]] * 6 + [[1, 2]] * 2)
    lay = oracle.dispatch_layout(idx, 4, 2, capacity=3)
    sp = lay["slot_pos"].reshape(8, 2)
    assert lay["routed_counts"].tolist() == [6, 8, 2, 0]
    assert lay["counts"].tolist() == [3, 3, 2, 0]
    assert lay["expert_offsets"].tolist() == [0, 3, 6, 8, 8]
    assert lay["part_offsets"].tolist() == [0, 6, 8]
    assert sp[:, 0].tolist() == [0, 1, 2, -1, -1, -1, -1, -1]
    assert sp[:, 1].tolist() == [3, 4, 5, -1, -1, -1, 6, 7]
    assert lay["perm"].tolist() == [0, 2, 4, 1, 3, 5, 13, 15]


def test_all_dropped_token_outputs_zero():
    x, wr, b, wg, wu, wd = tiny_inputs(21, 10, 8, 4, 2)
    res = oracle.layer_forward(x, wr, b, wg, wu, wd, 2, 2, capacity_factor=0.05)
    assert res["capacity"] == 1
    sp = res["slot_pos"].reshape(10, 2)
    dead = np.all(sp < 0, axis=1)
    # k = E = 2: every token picks both experts, so only token 0's two pairs survive
    assert dead.tolist() == [False] + [True] * 9
    assert np.all(res["out"][dead] == 0.0)


# ------------------------------------------------------------------ invariants
@pytest.mark.parametrize("cf", [None, 1.25, 0.3])
def test_dispatch_invariants(cf):
    shape = workloads.LayerShape("inv", N=3000, H=32, I=16, E=16, top_k=4, ep_size=4,
                                 capacity_factor=cf, zipf_s=1.1)
    inp = workloads.layer_inputs(shape, seed=5, with_experts=False)
    x = inp["x"].double().numpy()
    _, idx, w = oracle.route(x, inp["w_router"].double().numpy(),
                             inp["b_router"].double().numpy(), 4)
    N, k, E, P = 3000, 4, 16, 4
    C = oracle.expert_capacity(cf, N, k, E)
    lay = oracle.dispatch_layout(idx, E, P, C)
    assert lay["routed_counts"].sum() == N * k
    dropped = int((lay["slot_pos"] < 0).sum())
    assert lay["counts"].sum() + dropped == N * k
    if C is None:
        assert dropped == 0
    else:
        assert np.array_equal(lay["counts"], np.minimum(lay["routed_counts"], C))
    # no token picks an expert twice
    assert all(len(set(r)) == k for r in idx.tolist())
    # partitions: owner = expert // (E/P), contiguous in the send buffer
    for p in range(P):
        lo, hi = lay["part_offsets"][p], lay["part_offsets"][p + 1]
        assert hi - lo == lay["counts"][p * E // P:(p + 1) * E // P].sum()
        owners = oracle.expert_partition(idx.reshape(-1)[lay["perm"][lo:hi]], E, P)
        assert np.all(owners == p)
    # perm is a bijection onto kept pairs, inverse of slot_pos
    kept = np.nonzero(lay["slot_pos"] >= 0)[0]
    assert np.array_equal(np.sort(lay["perm"]), kept)
    assert np.array_equal(lay["slot_pos"][lay["perm"]], np.arange(len(lay["perm"])))
    # inside each expert segment: right expert, strictly increasing token ids
    for e in range(E):
        seg = lay["perm"][lay["expert_offsets"][e]:lay["expert_offsets"][e + 1]]
        assert np.all(idx.reshape(-1)[seg] == e)
        assert np.all(np.diff(seg // k) > 0)
    # dropped pairs of an expert are exactly those after its first C in token order
    if C is not None:
        for e in range(E):
            pairs = np.nonzero(idx.reshape(-1) == e)[0]
            assert np.all(lay["slot_pos"][pairs[:C]] >= 0)
            assert np.all(lay["slot_pos"][pairs[C:]] < 0)


def test_partition_of_experts_matches_page_table():
    # "How the sizes combine": with 8 experts, ep_size=4 gives E0E1 | E2E3 | E4E5 | E6E7
    # and ep_size=2 gives E0-3 | E4-7
    assert oracle.expert_partition(np.arange(8), 8, 4).tolist() == [0, 0, 1, 1, 2, 2, 3, 3]
    assert oracle.expert_partition(np.arange(8), 8, 2).tolist() == [0] * 4 + [1] * 4
    assert oracle.expert_partition(np.arange(8), 8, 8).tolist() == list(range(8))
    with pytest.raises(ValueError):
        oracle.expert_partition(np.arange(6), 6, 4)


# ------------------------------------------------------------------ exact-grid precondition
@pytest.mark.parametrize("shape", workloads.ALL_SHAPES, ids=lambda s: s.name)
def test_exact_variant_router_sums_fit_fp32(shape):
    """In the exact variant every product x*w is a multiple of 2^-16 (fp32 layers) or
    2^-18 (bf16 layers); if sum_h |x*w| + |b| stays below 2^8 resp. 2^6, every partial
    sum in any order needs at most 24 significant bits and fp32 accumulation is exact."""
    inp = workloads.layer_inputs(shape, seed=0, variant="exact", with_experts=False)
    x = inp["x"].double()
    wr = inp["w_router"].double()
    step_x = 2.0 ** -8
    step_w = workloads.router_grid_step(shape)

    def on_grid(t, step):
        return bool(torch.equal(torch.round(t / step), t / step))

    assert on_grid(x, step_x) and on_grid(wr, step_w)
    bound = x.abs() @ wr.abs().T
    if inp["b_router"] is not None:
        b = inp["b_router"].double()
        assert on_grid(b, step_w)
        bound = bound + b.abs()[None, :]
    bound = float(bound.max())
    limit = 2.0 ** 24 * step_x * step_w
    assert bound < limit


def test_token_outputs_equal_full_batch_layer():
    """The per-token path used for sampled checks at full size gives the same rows as the
    whole-batch path (with the batch's keep decisions)."""
    x, wr, b, wg, wu, wd = tiny_inputs(31, 40, 8, 6, 5)
    res = oracle.layer_forward(x, wr, b, wg, wu, wd, 2, 5, capacity_factor=0.6)
    sample = np.array([0, 3, 17, 39])
    keep = (res["slot_pos"].reshape(40, 2) >= 0)[sample]
    assert not keep.all()
    got = oracle.token_outputs(x[sample], res["topk_idx"][sample], res["topk_w"][sample], keep,
                               lambda e: (wg[e], wu[e], wd[e]))
    assert rel_err(got, res["out"][sample]) < 1e-13


# ------------------------------------------------------------------ planted mistakes
MUTANTS = {
    "tie_to_higher_id": ("top_k_experts",
                         lambda L, k: (L.shape[1] - 1 - np.argsort(
                             -np.asarray(L)[:, ::-1], axis=1, kind="stable"))[:, :k]),
    "softmax_over_all_experts": ("routing_weights",
                                 lambda L, idx: np.take_along_axis(
                                     scipy.special.softmax(L, axis=1), idx, axis=1)),
    "silu_on_up_not_gate": ("swiglu_expert",
                            lambda r, g, u, d: (om.silu(r @ u.T) * (r @ g.T)) @ d.T),
    "transposed_gate": ("swiglu_expert",
                        lambda r, g, u, d: (om.silu(r @ g) * (r @ u.T)) @ d.T),
    "missing_bias": ("router_logits", lambda x, w, b=None: np.asarray(x) @ np.asarray(w).T),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_oracle_mistake_is_caught(name, monkeypatch):
    fn, bad = MUTANTS[name]
    monkeypatch.setattr(om, fn, bad)
    caught = False
    for case in TINY_CASES:
        try:
            res, bf = _oracle_with_bf(case)
        except Exception:
            caught = True
            break
        sel = np.zeros_like(bf["selected"])
        np.put_along_axis(sel, res["topk_idx"], True, axis=1)
        if not np.array_equal(sel, bf["selected"]) or rel_err(res["out"], bf["out"]) > 1e-12:
            caught = True
            break
    assert caught, f"planted mistake {name} went unnoticed"


def test_planted_drop_order_mistake_is_caught(monkeypatch):
    real = om.dispatch_layout

    def keep_last(idx, E, P, capacity=None, priority="token"):
        lay = real(idx, E, P, capacity, priority)
        flat = np.asarray(idx).reshape(-1)
        sp = np.full(flat.size, -1, dtype=np.int64)
        for e in range(E):
            pairs = np.nonzero(flat == e)[0]
            keep = pairs[len(pairs) - lay["counts"][e]:]    # last C instead of first C
            sp[keep] = lay["expert_offsets"][e] + np.arange(len(keep))
        perm = np.empty(len(lay["perm"]), dtype=np.int64)
        perm[sp[sp >= 0]] = np.nonzero(sp >= 0)[0]
        return dict(lay, slot_pos=sp, perm=perm)

    monkeypatch.setattr(om, "dispatch_layout", keep_last)
    res, bf = _oracle_with_bf((5, 7, 10, 7, 3, 1, 1, 0.01, None))
    assert rel_err(res["out"], bf["out"]) > 1e-6


# ------------------------------------------------------------------ routing variants
# [UL-EP] "Load balancing and capacity": a per-expert bias that only influences the
# choice of experts, updated after each step; at most M partitions (nodes) per token.
VARIANT_CASES = [
    # case index into TINY_CASES, selection-bias scale, group limit
    (0, 0.5, None), (1, 0.3, 2), (2, 0.25, 1), (3, 0.0, 3), (6, 1.0, 2), (7, 0.2, 1),
]


def _variant(case_i, scale, M, mode="dispatch"):
    seed, N, H, I, E, k, P, cf, grid = TINY_CASES[case_i]
    x, wr, b, wg, wu, wd = tiny_inputs(seed, N, H, I, E, grid)
    rng = np.random.default_rng(100 + case_i)
    beta = np.round(rng.uniform(-1, 1, E) * scale * 8) / 8     # dyadic: exact sums
    if M is not None and M * (E // P) < k:
        M = -(-k // (E // P))
    res = oracle.layer_forward(x, wr, b, wg, wu, wd, k, P, cf, mode, selection_bias=beta,
                               group_limit=M)
    bf = brute_force_layer(x, wr, b, wg, wu, wd, k, P, res["capacity"], sel_bias=beta,
                           group_limit=M)
    return res, bf, dict(E=E, P=P, k=k, M=M, beta=beta, x=x, wr=wr, b=b)


@pytest.mark.parametrize("mode", ["dispatch", "mask_sum"])
@pytest.mark.parametrize("vc", VARIANT_CASES, ids=lambda v: f"case{v[0]}-s{v[1]}-M{v[2]}")
def test_variant_oracle_equals_dense_brute_force(vc, mode):
    res, bf, _ = _variant(*vc, mode=mode)
    sel = np.zeros_like(bf["selected"])
    np.put_along_axis(sel, res["topk_idx"], True, axis=1)
    assert np.array_equal(sel, bf["selected"])
    w = np.zeros(sel.shape)
    np.put_along_axis(w, res["topk_idx"], res["topk_w"], axis=1)
    assert rel_err(w, bf["weight"]) < 1e-12
    assert rel_err(res["out"], bf["out"]) < 1e-12


def test_zero_or_constant_selection_bias_is_plain_routing():
    x, wr, b, *_ = tiny_inputs(3, 9, 8, 4, 8, grid=0.25)
    _, idx0, w0 = oracle.route(x, wr, b, 3)
    for beta in (np.zeros(8), np.full(8, 0.75)):
        _, idx, w = oracle.route_variant(x, wr, b, 3, selection_bias=beta)
        assert np.array_equal(idx, idx0) and np.array_equal(w, w0)


def test_selection_bias_moves_the_choice_but_weights_use_raw_logits():
    # two experts chosen out of three; a large bias on expert 2 forces it into every
    # selection, and the pair's weights follow the logistic closed form of the RAW
    # logits: w0 = 1 / (1 + exp(l1 - l0))
    L = np.array([[2.0, 1.0, 0.0], [0.5, 3.0, -1.0], [1.0, 1.0, 1.0]])
    beta = np.array([0.0, 0.0, 10.0])
    idx = oracle.group_limited_top_k(oracle.selection_scores(L, beta), 2, 1, None)
    assert idx.tolist() == [[2, 0], [2, 1], [2, 0]]
    w = oracle.routing_weights(L, idx)
    for t in range(3):
        l0, l1 = L[t, idx[t, 0]], L[t, idx[t, 1]]
        assert abs(w[t, 0] - 1.0 / (1.0 + math.exp(l1 - l0))) < 1e-15


def test_group_limit_reduces_to_plain_top_k():
    x, wr, b, *_ = tiny_inputs(2, 16, 12, 6, 6)
    L = oracle.router_logits(x, wr, b)
    plain = oracle.top_k_experts(L, 3)
    assert np.array_equal(oracle.group_limited_top_k(L, 3, 3, 3), plain)
    assert np.array_equal(oracle.group_limited_top_k(L, 3, 3, None), plain)
    # tokens whose plain top-k already spans at most M partitions keep it
    owner = plain // 2
    spans = np.array([len(set(r)) for r in owner])
    lim = oracle.group_limited_top_k(L, 3, 3, 2)
    assert np.array_equal(lim[spans <= 2], plain[spans <= 2])
    assert np.all([len(set(r)) <= 2 for r in lim // 2])


def test_group_limit_one_keeps_the_argmax_partition():
    rng = np.random.default_rng(7)
    L = rng.standard_normal((40, 12))
    idx = oracle.group_limited_top_k(L, 3, 4, 1)        # 4 partitions of 3 experts
    for t in range(40):
        p = int(np.argmax(L[t])) // 3
        inside = list(range(3 * p, 3 * p + 3))
        assert sorted(idx[t].tolist()) == sorted(inside)
        assert idx[t].tolist() == sorted(inside, key=lambda e: (-L[t, e], e))


def test_selection_bias_update_closed_form():
    beta = np.array([0.5, -0.25, 0.0, 1.0], dtype=np.float32)
    # N = 6 tokens, k = 2: equal share 3 per expert
    new = oracle.update_selection_bias(beta, [5, 1, 3, 3], 6, 2, 0.125)
    assert new.dtype == np.float32
    assert new.tolist() == [0.375, -0.125, 0.0, 1.0]
    same = oracle.update_selection_bias(beta, [3, 3, 3, 3], 6, 2, 0.125)
    assert np.array_equal(same, beta)


VARIANT_MUTANTS = ["weights_from_biased_scores", "partition_score_is_sum",
                   "partition_ties_to_higher_id", "group_limit_ignored"]


def _mutant(name):
    real_w, real_g = om.routing_weights, om.group_limited_top_k
    if name == "weights_from_biased_scores":
        def route_variant(x, w_router, b_router, k, selection_bias=None, ep_size=1,
                          group_limit=None):
            logits = om.router_logits(x, w_router, b_router)
            s = om.selection_scores(logits, selection_bias)
            idx = real_g(s, k, ep_size, group_limit)
            return logits, idx, real_w(s, idx)
        return "route_variant", route_variant

    def glt(scores, k, ep_size, group_limit):
        s = np.asarray(scores, dtype=np.float64)
        N, E = s.shape
        if group_limit is None or group_limit >= ep_size:
            return om.top_k_experts(s, k)
        if name == "group_limit_ignored":
            return om.top_k_experts(s, k)
        owner = np.arange(E) // (E // ep_size)
        red = (lambda a: a.sum(axis=1)) if name == "partition_score_is_sum" else (
            lambda a: a.max(axis=1))
        best = np.stack([red(s[:, owner == p]) for p in range(ep_size)], axis=1)
        if name == "partition_ties_to_higher_id":
            kept = np.argsort(-best[:, ::-1], axis=1, kind="stable")[:, :group_limit]
            kept = ep_size - 1 - kept
        else:
            kept = np.argsort(-best, axis=1, kind="stable")[:, :group_limit]
        allowed_part = np.zeros((N, ep_size), dtype=bool)
        allowed_part[np.arange(N)[:, None], kept] = True
        allowed = allowed_part[:, owner]
        ids = np.broadcast_to(np.arange(E), (N, E))
        return np.lexsort((ids, -s, ~allowed), axis=-1)[:, :k].astype(np.int64)
    return "group_limited_top_k", glt


@pytest.mark.parametrize("name", VARIANT_MUTANTS)
def test_planted_variant_mistake_is_caught(name, monkeypatch):
    fn, bad = _mutant(name)
    monkeypatch.setattr(om, fn, bad)
    caught = False
    for vc in VARIANT_CASES + [(2, 0.0, 1), (6, 0.0, 1), (3, 0.0, 1)]:
        res, bf, _ = _variant(*vc)
        sel = np.zeros_like(bf["selected"])
        np.put_along_axis(sel, res["topk_idx"], True, axis=1)
        if not np.array_equal(sel, bf["selected"]) or rel_err(res["out"], bf["out"]) > 1e-12:
            caught = True
            break
    assert caught, f"planted mistake {name} went unnoticed"

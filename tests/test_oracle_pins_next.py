"""Pins of the oracle's widened steps against things other than themselves.

* backward: central finite differences of the oracle's own (separately pinned) forward,
  and torch autograd through an independent dense formulation of the layer;
* slot-major capacity priority: an explicit double loop (slot, then token) and the
  GShard-style cumulative-sum formulation (positions of slot j offset by the earlier
  slots' totals);
* balance statistics: closed forms (uniform logits, two experts), shift invariance and
  torch.softmax;
* TP row split: the slice rule's cover / size properties, equality with the unsplit
  layer when no capacity applies, per-slice capacity by brute force;
* planted mistakes in each of these must make a pin fail.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import oracle.moe as om
from test_oracle_pins import brute_force_layer, rel_err, tiny_inputs


# ------------------------------------------------------------------ backward
BWD_CASES = [
    # seed, N, H, I, E, k, P, cf, grid
    (11, 7, 6, 5, 4, 2, 2, None, None),
    (12, 9, 5, 4, 3, 3, 3, None, None),     # k = E
    (13, 10, 6, 6, 4, 2, 2, 0.5, None),     # drops
    (14, 6, 4, 3, 2, 1, 1, None, None),     # k = 1: weight 1, no router gradient
]


def _bwd_inputs(case):
    seed, N, H, I, E, k, P, cf, _ = case
    x, wr, b, wg, wu, wd = tiny_inputs(seed, N, H, I, E)
    wr = wr * 4.0                              # spread the logits: nonzero softmax Jacobian
    dout = np.random.default_rng(seed + 100).standard_normal((N, H))
    return x, wr, b, wg, wu, wd, dout


def _loss(x, wr, b, wg, wu, wd, k, P, cf, dout):
    return float(np.sum(oracle.layer_forward(x, wr, b, wg, wu, wd, k, P, cf)["out"] * dout))


@pytest.mark.parametrize("case", BWD_CASES)
def test_backward_matches_finite_differences(case):
    seed, N, H, I, E, k, P, cf, _ = case
    x, wr, b, wg, wu, wd, dout = _bwd_inputs(case)
    g = oracle.layer_backward(x, wr, b, wg, wu, wd, k, P, dout, cf)
    args = dict(x=x, wr=wr, b=b, wg=wg, wu=wu, wd=wd)
    keys = dict(x="dx", wr="dw_router", b="db_router", wg="dw_gate", wu="dw_up", wd="dw_down")
    eps = 1e-6
    for name, arr in args.items():
        num = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            hi, lo = arr.copy(), arr.copy()
            hi[i] += eps
            lo[i] -= eps
            a_hi, a_lo = dict(args, **{name: hi}), dict(args, **{name: lo})
            num[i] = (_loss(**a_hi, k=k, P=P, cf=cf, dout=dout)
                      - _loss(**a_lo, k=k, P=P, cf=cf, dout=dout)) / (2 * eps)
        scale = max(np.max(np.abs(num)), 1e-3)
        assert np.max(np.abs(num - g[keys[name]])) < 1e-6 * scale + 1e-9, name


def _autograd_dense(x, wr, b, wg, wu, wd, k, P, cf, dout):
    """The layer as one dense torch expression with the oracle-independent brute-force
    routing decisions frozen: out = sum_e kept[t,e] * w[t,e] * FFN_e(x_t), w the softmax
    of the logits restricted to the selection (computed with -inf masking)."""
    bf = brute_force_layer(x, wr, b, wg, wu, wd, k, P,
                           oracle.expert_capacity(cf, x.shape[0], k, wr.shape[0]))
    T = lambda a: torch.tensor(a, dtype=torch.float64, requires_grad=True)  # noqa: E731
    tx, twr, tb, twg, twu, twd = T(x), T(wr), T(b), T(wg), T(wu), T(wd)
    L = tx @ twr.T + tb
    sel = torch.tensor(bf["selected"])
    w = torch.softmax(L.masked_fill(~sel, -math.inf), dim=1)
    kept = torch.tensor(bf["kept"], dtype=torch.float64)
    out = torch.zeros_like(tx)
    for e in range(wr.shape[0]):
        h = torch.nn.functional.silu(tx @ twg[e].T) * (tx @ twu[e].T)
        out = out + (kept[:, e] * w[:, e])[:, None] * (h @ twd[e].T)
    (out * torch.tensor(dout)).sum().backward()
    return dict(dx=tx.grad, dw_router=twr.grad, db_router=tb.grad, dw_gate=twg.grad,
                dw_up=twu.grad, dw_down=twd.grad)


@pytest.mark.parametrize("case", BWD_CASES)
def test_backward_matches_torch_autograd_of_dense_layer(case):
    seed, N, H, I, E, k, P, cf, _ = case
    x, wr, b, wg, wu, wd, dout = _bwd_inputs(case)
    g = oracle.layer_backward(x, wr, b, wg, wu, wd, k, P, dout, cf)
    ref = _autograd_dense(x, wr, b, wg, wu, wd, k, P, cf, dout)
    for key, val in ref.items():
        assert rel_err(g[key], val.numpy()) < 1e-12, key


def test_silu_grad_closed_forms():
    assert om.silu_grad(0.0) == pytest.approx(0.5)
    z = 1.3
    s = 1 / (1 + math.exp(-z))
    assert om.silu_grad(z) == pytest.approx(s + z * s * (1 - s), rel=1e-15)
    assert om.silu_grad(-60.0) == pytest.approx(0.0, abs=1e-20)
    assert om.silu_grad(60.0) == pytest.approx(1.0, rel=1e-15)


BWD_MUTANTS = {
    # the softmax Jacobian dropped: dlogit = dweight
    "no_softmax_jacobian": "dlogits",
    # sigmoid in place of the SiLU derivative
    "silu_grad_is_sigmoid": "silu_grad",
}


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_planted_backward_mistake_is_caught(name, monkeypatch):
    if name == "silu_grad_is_sigmoid":
        monkeypatch.setattr(om, "silu_grad", lambda z: 1 / (1 + np.exp(-np.asarray(z, float))))
    else:
        real_bwd = om.layer_backward

        def bad_bwd(*a, **kw):
            # the router gradient recomputed with dlogit = dweight (no softmax Jacobian)
            g = real_bwd(*a, **kw)
            fwd, dl = g["forward"], g["dlogits"]
            x, wr = np.asarray(a[0], float), np.asarray(a[1], float)
            w = fwd["topk_w"]
            chosen = np.take_along_axis(dl, fwd["topk_idx"], axis=1)
            s = np.sum(chosen, axis=1, keepdims=True)      # = 0: sum_c w_c (dw_c - <w,dw>)
            dweight = np.where(w > 0, chosen / np.where(w > 0, w, 1.0), 0.0) + s
            wrong = np.zeros_like(dl)
            np.put_along_axis(wrong, fwd["topk_idx"], dweight, axis=1)
            g["dx"] = g["dx"] - dl @ wr + wrong @ wr
            g["dw_router"] = wrong.T @ x
            return g
        monkeypatch.setattr(om, "layer_backward", bad_bwd)
    caught = False
    for case in BWD_CASES:
        seed, N, H, I, E, k, P, cf, _ = case
        x, wr, b, wg, wu, wd, dout = _bwd_inputs(case)
        g = om.layer_backward(x, wr, b, wg, wu, wd, k, P, dout, cf)
        ref = _autograd_dense(x, wr, b, wg, wu, wd, k, P, cf, dout)
        if any(rel_err(g[key], val.numpy()) > 1e-9 for key, val in ref.items()):
            caught = True
            break
    assert caught, name


# ------------------------------------------------------------------ slot-major priority
def _slot_major_loop(idx, E, capacity):
    """Explicit loops: slot j outer, token t inner; a pair is kept iff its expert has
    taken fewer than C pairs so far."""
    N, k = idx.shape
    taken = [0] * E
    keep = np.zeros((N, k), dtype=bool)
    order = {e: [] for e in range(E)}
    for j in range(k):
        for t in range(N):
            e = int(idx[t, j])
            if capacity is None or taken[e] < capacity:
                keep[t, j] = True
                taken[e] += 1
                order[e].append(t * k + j)
    return keep, order


def _gshard_cumsum(idx, E, capacity):
    """GShard-style positions: one-hot masks per slot, position = running count within
    the slot plus the totals of the earlier slots."""
    N, k = idx.shape
    pos = np.zeros((N, k), dtype=np.int64)
    offset = np.zeros(E, dtype=np.int64)
    for j in range(k):
        mask = np.zeros((N, E), dtype=np.int64)
        mask[np.arange(N), idx[:, j]] = 1
        p = np.cumsum(mask, axis=0) - 1 + offset[None, :]
        pos[:, j] = p[np.arange(N), idx[:, j]]
        offset += mask.sum(axis=0)
    keep = np.ones((N, k), bool) if capacity is None else pos < capacity
    return pos, keep


@pytest.mark.parametrize("seed,N,E,k,C", [(1, 30, 4, 2, 5), (2, 64, 8, 3, 7), (3, 17, 3, 3, 4),
                                          (4, 40, 6, 2, None), (5, 9, 2, 1, 3), (6, 1, 4, 2, 1)])
def test_slot_priority_layout_matches_loop_and_cumsum(seed, N, E, k, C):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(N)])
    lay = oracle.dispatch_layout(idx, E, 1, C, priority="slot")
    keep, order = _slot_major_loop(idx, E, C)
    pos, keep2 = _gshard_cumsum(idx, E, C)
    sp = lay["slot_pos"].reshape(N, k)
    assert np.array_equal(sp >= 0, keep)
    assert np.array_equal(keep, keep2)
    for e in range(E):
        a, b = lay["expert_offsets"][e], lay["expert_offsets"][e + 1]
        assert list(lay["perm"][a:b]) == order[e]
    kept = sp >= 0
    assert np.array_equal(sp[kept] - lay["expert_offsets"][idx[kept]], pos[kept])


def test_slot_priority_differs_from_token_priority_and_k1_agrees():
    idx = np.array([[0, 1], [1, 0], [0, 1]])
    tok = oracle.dispatch_layout(idx, 2, 1, 2, "token")
    slot = oracle.dispatch_layout(idx, 2, 1, 2, "slot")
    # expert 0 is chosen by t0 (slot 0), t1 (slot 1), t2 (slot 0): token order keeps
    # t0, t1; slot order keeps t0, t2
    assert list(tok["slot_pos"].reshape(3, 2)[:, :][[0, 1, 2], [0, 1, 0]] >= 0) == [True, True, False]
    assert list(slot["slot_pos"].reshape(3, 2)[[0, 1, 2], [0, 1, 0]] >= 0) == [True, False, True]
    idx1 = np.array([[2], [0], [2], [1], [2]])
    a = oracle.dispatch_layout(idx1, 3, 1, 2, "token")
    b = oracle.dispatch_layout(idx1, 3, 1, 2, "slot")
    for key in a:
        assert np.array_equal(a[key], b[key]), key


def test_slot_priority_layer_equals_brute_force_without_capacity():
    x, wr, b, wg, wu, wd = tiny_inputs(41, 15, 8, 5, 4)
    res = oracle.layer_forward(x, wr, b, wg, wu, wd, 2, 2, None, capacity_priority="slot")
    bf = brute_force_layer(x, wr, b, wg, wu, wd, 2, 2, None)
    assert rel_err(res["out"], bf["out"]) < 1e-12


def test_planted_slot_priority_mistake_is_caught(monkeypatch):
    real = om.dispatch_layout
    monkeypatch.setattr(om, "dispatch_layout",
                        lambda idx, E, P, C=None, priority="token": real(idx, E, P, C, "token"))
    rng = np.random.default_rng(9)
    idx = np.stack([rng.choice(6, 2, replace=False) for _ in range(40)])
    keep, _ = _slot_major_loop(idx, 6, 5)
    lay = om.dispatch_layout(idx, 6, 1, 5, "slot")
    assert not np.array_equal(lay["slot_pos"].reshape(40, 2) >= 0, keep)


# ------------------------------------------------------------------ balance statistics
def test_balance_stats_closed_forms():
    N, E, k = 12, 4, 2
    st = oracle.balance_stats(np.zeros((N, E)), np.array([6, 6, 6, 6]), N, k)
    assert np.allclose(st["prob_mean"], 0.25, rtol=0, atol=1e-16)
    assert np.allclose(st["load_frac"], 0.25, rtol=0, atol=0)
    d = np.array([0.3, -1.2, 2.5])
    lg = np.stack([d, np.zeros(3)], axis=1)
    st = oracle.balance_stats(lg, np.array([2, 1]), 3, 1)
    assert st["prob_mean"][0] == pytest.approx(np.mean(1 / (1 + np.exp(-d))), rel=1e-15)
    assert list(st["load_frac"]) == [2 / 3, 1 / 3]


def test_balance_stats_sums_shift_invariance_and_torch_softmax():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((50, 7)) * 3
    counts = np.bincount(rng.integers(0, 7, 100), minlength=7)
    st = oracle.balance_stats(lg, counts, 50, 2)
    assert st["prob_mean"].sum() == pytest.approx(1.0, rel=1e-14)
    assert st["load_frac"].sum() == pytest.approx(1.0, rel=1e-15)
    shifted = oracle.balance_stats(lg + rng.standard_normal((50, 1)) * 100, counts, 50, 2)
    assert rel_err(shifted["prob_mean"], st["prob_mean"]) < 1e-12
    ref = torch.softmax(torch.tensor(lg), dim=1).mean(dim=0).numpy()
    assert rel_err(st["prob_mean"], ref) < 1e-14


def test_planted_balance_stats_mistake_is_caught():
    lg = np.random.default_rng(4).standard_normal((20, 5))
    st = oracle.balance_stats(lg, np.full(5, 8), 20, 2)
    wrong = np.exp(lg).mean(axis=0)                  # unnormalised probabilities
    assert rel_err(wrong, st["prob_mean"]) > 1e-3


# ------------------------------------------------------------------ TP row split
@pytest.mark.parametrize("N,tp", [(0, 2), (1, 2), (1, 4), (7, 3), (8, 2), (5, 8), (100, 3)])
def test_tp_slices_cover_disjointly_and_evenly(N, tp):
    sl = oracle.tp_slices(N, tp)
    assert len(sl) == tp
    assert sl[0][0] == 0 and sl[-1][1] == N
    for (a, b), (c, _) in zip(sl, sl[1:]):
        assert b == c
    sizes = [b - a for a, b in sl]
    assert max(sizes) - min(sizes) <= 1 and sum(sizes) == N
    assert sizes == sorted(sizes, reverse=True)


@pytest.mark.parametrize("mode", ["dispatch", "mask_sum"])
@pytest.mark.parametrize("N,tp", [(13, 2), (13, 4), (1, 2), (3, 5)])
def test_tp_split_equals_unsplit_layer_without_capacity(N, tp, mode):
    x, wr, b, wg, wu, wd = tiny_inputs(50 + N + tp, N, 8, 5, 4)
    padded, out = oracle.tp_row_split_forward(x, wr, b, wg, wu, wd, 2, 2, tp, None, mode)
    bf = brute_force_layer(x, wr, b, wg, wu, wd, 2, 2, None)
    assert rel_err(out, bf["out"]) < 1e-12
    for s, (a, e) in enumerate(oracle.tp_slices(N, tp)):
        assert not padded[s, :a].any() and not padded[s, e:].any()


def test_tp_split_capacity_is_per_slice():
    N, tp, k, E = 20, 2, 2, 4
    x, wr, b, wg, wu, wd = tiny_inputs(61, N, 8, 5, E)
    _, out = oracle.tp_row_split_forward(x, wr, b, wg, wu, wd, k, 2, tp, 0.5)
    ref = np.zeros_like(out)
    for a, e in oracle.tp_slices(N, tp):
        C = oracle.expert_capacity(0.5, e - a, k, E)
        ref[a:e] = brute_force_layer(x[a:e], wr, b, wg, wu, wd, k, 2, C)["out"]
    assert rel_err(out, ref) < 1e-12
    whole = brute_force_layer(x, wr, b, wg, wu, wd, k, 2,
                              oracle.expert_capacity(0.5, N, k, E))["out"]
    assert rel_err(out, whole) > 1e-6          # the slices' drops differ from the batch's


# ------------------------------------------------------------------ sampled backward
def test_sampled_backward_functions_equal_the_batch_backward():
    """The per-token dx and per-expert weight gradients used for full-size sampled checks
    give the whole-batch backward's rows and blocks (with the batch's keep decisions)."""
    case = (71, 24, 8, 6, 5, 2, 5, 0.6, None)
    seed, N, H, I, E, k, P, cf, _ = case
    x, wr, b, wg, wu, wd, dout = _bwd_inputs(case)
    g = oracle.layer_backward(x, wr, b, wg, wu, wd, k, P, dout, cf)
    fwd = g["forward"]
    keep = fwd["slot_pos"].reshape(N, k) >= 0
    assert not keep.all()
    sample = np.array([0, 5, 11, 23])
    got = oracle.token_input_grads(x[sample], dout[sample], fwd["topk_idx"][sample],
                                   fwd["topk_w"][sample], keep[sample], wr,
                                   lambda e: (wg[e], wu[e], wd[e]))
    assert rel_err(got, g["dx"][sample]) < 1e-12
    for e in range(E):
        a, z = fwd["expert_offsets"][e], fwd["expert_offsets"][e + 1]
        pairs = fwd["perm"][a:z]
        if len(pairs) == 0:
            continue
        t = pairs // k
        w = fwd["topk_w"].reshape(-1)[pairs]
        dg, du, dd = oracle.expert_weight_grads(x[t], dout[t], w, wg[e], wu[e], wd[e])
        assert rel_err(dg, g["dw_gate"][e]) < 1e-12
        assert rel_err(du, g["dw_up"][e]) < 1e-12
        assert rel_err(dd, g["dw_down"][e]) < 1e-12


@pytest.mark.parametrize("priority", ["token", "slot"])
def test_backward_under_routing_variants_matches_finite_differences(priority):
    """The backward paths the GPU tests compare against: a selection-only bias, a group
    limit and both capacity priorities. The selection (piecewise constant) is unchanged
    by the small perturbations, so central differences of the forward pin every
    gradient."""
    N, H, I, E, k, P, cf = 12, 5, 4, 6, 2, 3, 0.7
    x, wr, b, wg, wu, wd = tiny_inputs(81, N, H, I, E)
    wr = wr * 4.0
    beta = np.random.default_rng(82).uniform(-0.3, 0.3, E)
    dout = np.random.default_rng(83).standard_normal((N, H))
    g = oracle.layer_backward(x, wr, b, wg, wu, wd, k, P, dout, cf, selection_bias=beta,
                              group_limit=2, capacity_priority=priority)

    def loss(**kw):
        a = dict(x=x, wr=wr, b=b, wg=wg, wu=wu, wd=wd)
        a.update(kw)
        return float(np.sum(oracle.layer_forward(a["x"], a["wr"], a["b"], a["wg"], a["wu"],
                                                 a["wd"], k, P, cf, "dispatch", beta, 2,
                                                 priority)["out"] * dout))

    eps = 1e-6
    for name, arr, key in [("x", x, "dx"), ("wr", wr, "dw_router"), ("b", b, "db_router"),
                           ("wg", wg, "dw_gate"), ("wd", wd, "dw_down")]:
        num = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            hi, lo = arr.copy(), arr.copy()
            hi[i] += eps
            lo[i] -= eps
            num[i] = (loss(**{name: hi}) - loss(**{name: lo})) / (2 * eps)
        assert np.max(np.abs(num - g[key])) < 1e-6 * max(np.max(np.abs(num)), 1e-3), name
    # and the routing really is a variant: the bias or the limit changed the selection
    plain = oracle.layer_forward(x, wr, b, wg, wu, wd, k, P, cf)
    assert not np.array_equal(plain["topk_idx"], g["forward"]["topk_idx"])

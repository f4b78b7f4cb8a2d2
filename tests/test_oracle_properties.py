"""Property checks of the oracle on random small layers (hypothesis): the sparse,
sort-based oracle equals the independent dense brute force of test_oracle_pins for any
shape, capacity, mode and routing variant drawn, and its layout invariants hold."""
import numpy as np
from hypothesis import given, settings
from hypothesis import strategies as st

import oracle
from test_oracle_pins import brute_force_layer, rel_err, tiny_inputs


@st.composite
def layers(draw):
    P = draw(st.sampled_from([1, 2, 4]))
    E = P * draw(st.integers(1, 3))
    k = draw(st.integers(1, E))
    N = draw(st.integers(1, 24))
    H = draw(st.sampled_from([4, 8]))
    I = draw(st.sampled_from([3, 6]))
    cf = draw(st.sampled_from([None, 0.3, 0.8, 1.25]))
    grid = draw(st.sampled_from([None, 0.25]))
    seed = draw(st.integers(0, 10**6))
    mode = draw(st.sampled_from(["dispatch", "mask_sum"]))
    return seed, N, H, I, E, k, P, cf, grid, mode


@settings(max_examples=60, deadline=None)
@given(layers())
def test_oracle_equals_brute_force_on_random_layers(case):
    seed, N, H, I, E, k, P, cf, grid, mode = case
    x, wr, b, wg, wu, wd = tiny_inputs(seed, N, H, I, E, grid)
    res = oracle.layer_forward(x, wr, b, wg, wu, wd, k, P, cf, mode)
    bf = brute_force_layer(x, wr, b, wg, wu, wd, k, P, res["capacity"])
    sel = np.zeros((N, E), dtype=bool)
    np.put_along_axis(sel, res["topk_idx"], True, axis=1)
    assert np.array_equal(sel, bf["selected"])
    assert rel_err(res["out"], bf["out"]) < 1e-10 or np.max(np.abs(bf["out"])) == 0
    # layout invariants: perm is a bijection onto the kept pairs, token order within a
    # segment, partition offsets at the partition's first expert
    sp, perm, off = res["slot_pos"], res["perm"], res["expert_offsets"]
    kept = np.nonzero(sp >= 0)[0]
    assert np.array_equal(np.sort(perm), kept)
    assert np.array_equal(sp[perm], np.arange(len(perm)))
    for e in range(E):
        seg = perm[off[e]:off[e + 1]]
        assert np.all(np.diff(seg // k) > 0)
        assert np.all(res["topk_idx"].reshape(-1)[seg] == e)
    assert np.array_equal(res["part_offsets"], off[np.arange(P + 1) * (E // P)])


@settings(max_examples=40, deadline=None)
@given(layers(), st.sampled_from([0.0, 0.05]), st.integers(1, 4))
def test_routing_variants_equal_brute_force_on_random_layers(case, bias_scale, m):
    seed, N, H, I, E, k, P, cf, grid, mode = case
    x, wr, b, wg, wu, wd = tiny_inputs(seed, N, H, I, E, grid)
    beta = np.random.default_rng(seed + 1).uniform(-bias_scale, bias_scale, E)
    gl = m if m * (E // P) >= k else None
    res = oracle.layer_forward(x, wr, b, wg, wu, wd, k, P, cf, mode, selection_bias=beta,
                               group_limit=gl)
    bf = brute_force_layer(x, wr, b, wg, wu, wd, k, P, res["capacity"], sel_bias=beta,
                           group_limit=gl)
    sel = np.zeros((N, E), dtype=bool)
    np.put_along_axis(sel, res["topk_idx"], True, axis=1)
    assert np.array_equal(sel, bf["selected"])
    assert rel_err(res["out"], bf["out"]) < 1e-10 or np.max(np.abs(bf["out"])) == 0

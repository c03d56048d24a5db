"""Pins of the oracle's router variants -- softmax top-k without
renormalisation, group-limited noaux_tc (n_group > 1) and the adaptive expert
top-p trim -- to hand-computed examples, brute force on tiny inputs and
invariants.  Each test names the mistake it is there to catch."""
import itertools
import math

import numpy as np
import pytest
import scipy.special

import oracle
from inputs import numpy_swiglu
from test_oracle_pins import _layer, logistic, rand_expert


def lay(E, k, mode=0, rsf=1.0, n_group=0, topk_group=0, top_p=0.0, H=128, I=128, shared=0):
    return oracle.layout(num_experts=E, top_k=k, hidden=H, intermediate=I, n_shared=shared,
                         shared_intermediate=192 if shared else 0, router_mode=mode, x_dtype=0,
                         routed_scaling_factor=rsf, n_group=n_group, topk_group=topk_group,
                         top_p=top_p)


LN = np.log(np.array([[1.0, 2.0, 3.0, 4.0]]))      # softmax(LN) = [0.1, 0.2, 0.3, 0.4]


# ------------------------------------------------ unrenormalised softmax --

def test_raw_softmax_hand_example():
    """Mode 2 keeps the full-softmax probabilities (renormalising them, or
    leaving out rsf, fails)."""
    idx, w, _, _ = oracle.route_from_logits(lay(4, 2, mode=0), None, LN)
    assert list(idx[0]) == [3, 2] and np.allclose(w[0], [4 / 7, 3 / 7], rtol=1e-14)
    idx, w, _, _ = oracle.route_from_logits(lay(4, 2, mode=2, rsf=2.0), None, LN)
    assert list(idx[0]) == [3, 2] and np.allclose(w[0], [0.8, 0.6], rtol=1e-14)


def test_raw_softmax_full_k_is_library_softmax():
    rng = np.random.default_rng(21)
    z = rng.normal(0, 2, (12, 9))
    b = rng.normal(0, 0.3, 9).astype(np.float32)
    idx, w, _, _ = oracle.route_from_logits(lay(9, 9, mode=2, rsf=1.5), b, z)
    p = scipy.special.softmax(z + b.astype(np.float64), axis=1)
    for t in range(12):
        assert np.allclose(w[t], 1.5 * p[t, idx[t]], rtol=1e-13, atol=0)


def test_raw_softmax_selection_equals_renormalised_selection():
    """Only the weights differ between modes 0 and 2; their ratio is the
    selected probability mass, at most 1."""
    rng = np.random.default_rng(22)
    z = rng.normal(0, 1, (30, 16))
    i0, w0, _, g0 = oracle.route_from_logits(lay(16, 4, mode=0), None, z)
    i2, w2, _, g2 = oracle.route_from_logits(lay(16, 4, mode=2), None, z)
    assert np.array_equal(i0, i2) and np.array_equal(g0, g2)
    mass = w2.sum(1)
    assert np.all(mass < 1) and np.allclose(w2, w0 * mass[:, None], rtol=1e-13)


# ------------------------------------------------------ grouped noaux_tc --

def grouped_example():
    """8 experts in 4 groups of 2; keys = sigmoid(z) + b, built from dyadic
    values.  Group sums of the two largest keys: g0 0.875, g1 1.0, g2 0.875,
    g3 0.75; group maxima: 0.875, 0.5, 0.4375, 0.75."""
    z = np.zeros((1, 8))
    z[0, 0] = math.log(3.0)                               # s0 = 0.75
    b = np.array([0.125, -0.5, 0.0, 0.0, -0.0625, -0.0625, 0.25, -0.5], np.float32)
    return z, b   # keys 0.875, 0, 0.5, 0.5, 0.4375, 0.4375, 0.75, 0


def test_grouped_hand_example():
    """Groups by the sum of their top-2 keys, ties to the lower group: groups 1
    and 0 stay; then experts 0 and 2 (2 beats 3 on the tie).  Without groups
    it would be {0, 6}; ranking groups by their maximum would keep groups 0
    and 3 and also give {0, 6}."""
    z, b = grouped_example()
    idx, w, _, gap = oracle.route_from_logits(lay(8, 2, mode=1, rsf=2.0, n_group=4,
                                                  topk_group=2), b, z)
    assert list(idx[0]) == [0, 2]
    assert np.allclose(w[0], [2.0 * 0.75 / 1.25, 2.0 * 0.5 / 1.25], rtol=1e-12)
    assert gap[0] == 0.0                        # the group tie and the expert tie
    idx1, _, _, _ = oracle.route_from_logits(lay(8, 2, mode=1, rsf=2.0), b, z)
    assert list(idx1[0]) == [0, 6]


@pytest.mark.parametrize("E,G,TG,k", [(8, 4, 2, 2), (8, 4, 2, 3), (12, 3, 1, 2), (12, 4, 3, 5),
                                      (16, 4, 2, 4)])
def test_grouped_matches_bruteforce(E, G, TG, k):
    """Brute force over every choice of topk_group groups (largest total of
    group scores, each the best pair of its keys), then every k-subset of
    their experts (largest key sum), listed by descending key."""
    rng = np.random.default_rng(1000 + E * 10 + G + TG + k)
    z = rng.normal(0, 1.5, (25, E))
    b = rng.normal(0, 0.1, E).astype(np.float32)
    idx, w, _, gap = oracle.route_from_logits(lay(E, k, mode=1, rsf=2.5, n_group=G,
                                                  topk_group=TG), b, z)
    s = logistic(z)
    keys = s + b.astype(np.float64)
    gsz = E // G
    for t in range(z.shape[0]):
        score = [max(keys[t, g * gsz + i] + keys[t, g * gsz + j]
                     for i, j in itertools.combinations(range(gsz), 2)) for g in range(G)]
        groups = max(itertools.combinations(range(G), TG), key=lambda c: sum(score[g] for g in c))
        members = [g * gsz + i for g in groups for i in range(gsz)]
        best = max(itertools.combinations(members, k), key=lambda S: sum(keys[t, list(S)]))
        assert list(idx[t]) == sorted(best, key=lambda e: -keys[t, e])
        assert np.allclose(w[t], 2.5 * s[t, idx[t]] / s[t, idx[t]].sum(), rtol=1e-13)
        assert gap[t] > 0


def test_grouped_all_groups_or_one_group_is_ungrouped():
    rng = np.random.default_rng(23)
    z = rng.normal(0, 1.5, (40, 32))
    b = rng.normal(0, 0.1, 32).astype(np.float32)
    ref = oracle.route_from_logits(lay(32, 6, mode=1, rsf=2.5), b, z)
    for G, TG in ((8, 8), (1, 1), (0, 0)):
        got = oracle.route_from_logits(lay(32, 6, mode=1, rsf=2.5, n_group=G, topk_group=TG), b, z)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


def test_grouped_choice_stays_in_kept_groups():
    rng = np.random.default_rng(24)
    z = rng.normal(0, 1.5, (200, 256))
    b = rng.normal(0, 0.1, 256).astype(np.float32)
    idx, _, _, _ = oracle.route_from_logits(lay(256, 8, mode=1, rsf=2.5, n_group=8,
                                                topk_group=4), b, z)
    assert all(len(set(row // 32)) <= 4 for row in idx)


# ---------------------------------------------------------- top-p trim --

@pytest.mark.parametrize("p,ids,ws", [
    (0.65, [3, 2, -1, -1], [4 / 7, 3 / 7, 0, 0]),        # C = 0, .4, .7, .9
    (0.75, [3, 2, 1, -1], [4 / 9, 3 / 9, 2 / 9, 0]),
    (0.35, [3, -1, -1, -1], [1, 0, 0, 0]),
    (0.95, [3, 2, 1, 0], [0.4, 0.3, 0.2, 0.1]),
])
def test_top_p_hand_example_softmax(p, ids, ws):
    """Slots are kept while the share of the slots before them is below p, and
    the kept weights renormalise (keeping the crossing slot's predecessor
    only, or forgetting to renormalise, fails)."""
    idx, w, _, _ = oracle.route_from_logits(lay(4, 4, mode=0, top_p=p), None, LN)
    assert list(idx[0]) == ids and np.allclose(w[0], ws, rtol=1e-13, atol=0)


def test_top_p_raw_softmax_keeps_probabilities():
    idx, w, _, _ = oracle.route_from_logits(lay(4, 4, mode=2, top_p=0.65), None, LN)
    assert list(idx[0]) == [3, 2, -1, -1] and np.allclose(w[0], [0.4, 0.3, 0, 0], rtol=1e-13)


def test_top_p_sigmoid_uses_selection_order():
    """Sigmoid mode: the shares follow slot (key) order, not score order.
    s = [0.75, 0.5, 0.25], bias lifts expert 1 to the first slot: shares
    1/3, 1/2, 1/6; p = 0.6 keeps experts 1 and 0, weights 0.5 and 0.75 over
    1.25, times rsf."""
    z = np.array([[math.log(3.0), 0.0, -math.log(3.0)]])
    b = np.array([0.0, 0.5, 0.0], np.float32)
    idx, w, _, _ = oracle.route_from_logits(lay(3, 3, mode=1, rsf=2.0, top_p=0.6), b, z)
    assert list(idx[0]) == [1, 0, -1]
    assert np.allclose(w[0], [0.8, 1.2, 0.0], rtol=1e-12, atol=0)


def test_top_p_off_values_and_invariants():
    rng = np.random.default_rng(25)
    z = rng.normal(0, 1.5, (60, 16))
    b = rng.normal(0, 0.1, 16).astype(np.float32)
    for mode in (0, 1, 2):
        base = oracle.route_from_logits(lay(16, 6, mode=mode, rsf=2.5), b, z)
        for off in (0.0, 1.0, 3.0):
            got = oracle.route_from_logits(lay(16, 6, mode=mode, rsf=2.5, top_p=off), b, z)
            assert np.array_equal(got[0], base[0]) and np.array_equal(got[1], base[1])
        idx, w, _, _ = oracle.route_from_logits(lay(16, 6, mode=mode, rsf=2.5, top_p=0.5), b, z)
        kept = (idx >= 0).sum(1)
        assert np.all(kept >= 1)
        for t in range(60):
            assert np.all(idx[t, :kept[t]] == base[0][t, :kept[t]])    # a prefix of the slots
            assert np.all(idx[t, kept[t]:] == -1) and np.all(w[t, kept[t]:] == 0)
            share = base[1][t] / base[1][t].sum()      # each slot's share of the selection
            c = np.concatenate([[0.0], np.cumsum(share)])
            assert c[kept[t] - 1] < 0.5 and (kept[t] == 6 or c[kept[t]] >= 0.5)   # minimal
            if mode == 2:
                assert np.allclose(w[t, :kept[t]], base[1][t, :kept[t]], rtol=1e-14)
            else:
                assert abs(w[t].sum() - 2.5) < 1e-12
        tiny = oracle.route_from_logits(lay(16, 6, mode=mode, rsf=2.5, top_p=1e-9), b, z)
        assert np.all(tiny[0][:, 1:] == -1)


def test_top_p_margin_in_gap():
    """The decision margin counts the distance from p to each cumulative share."""
    _, _, _, gap = oracle.route_from_logits(lay(4, 4, mode=0, top_p=0.7 + 1e-7), None, LN)
    assert gap[0] == pytest.approx(1e-7, rel=1e-6)


def test_dispatch_skips_dropped_slots():
    idx = np.array([[3, 2, -1], [0, -1, -1], [2, 0, 3]], np.int32)
    counts, offsets, perm, inv = oracle.dispatch(idx, 4)
    assert counts.tolist() == [2, 0, 2, 2] and offsets.tolist() == [0, 2, 2, 4, 6]
    assert perm[:6].tolist() == [3, 7, 1, 6, 0, 8]
    assert inv.tolist() == [4, 2, -1, 0, -1, -1, 3, 1, 5]


def test_top_p_layer_is_weighted_sum_of_kept_experts():
    E, H, I = 6, 128, 128
    L = lay(E, 4, mode=1, rsf=2.5, top_p=0.55, H=H, I=I, shared=1)
    Wr, ex, sh, x = _layer(L, 31, E, H, I, shared=True, T=24)
    b = np.random.default_rng(32).normal(0, 0.1, E).astype(np.float32)
    out, idx, w = oracle.moe_forward(L, oracle.weights(L, Wr, b, ex, sh), x)
    assert (idx == -1).any() and (idx[:, 1] >= 0).any()
    xd = x.astype(np.float64)
    ref = numpy_swiglu(sh, xd)
    for t in range(x.shape[0]):
        for j in range(4):
            if idx[t, j] >= 0:
                ref[t] += w[t, j] * numpy_swiglu(ex[idx[t, j]], xd[t:t + 1])[0]
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-11 * np.abs(ref).max())


@pytest.mark.parametrize("kw", [dict(mode=3), dict(n_group=4, topk_group=2),       # softmax
                                dict(mode=1, n_group=3, topk_group=1),              # 8 % 3
                                dict(mode=1, n_group=8, topk_group=1),              # groups of 1
                                dict(mode=1, n_group=4, topk_group=5),
                                dict(mode=1, n_group=4, topk_group=0),
                                dict(mode=1, n_group=4, topk_group=1, k=3),         # k > 1 * 2
                                dict(top_p=-0.1), dict(top_p=float("nan")), dict(n_group=-1)])
def test_variant_layouts_rejected(kw):
    kw = dict(kw)
    k = kw.pop("k", 2)
    L = lay(8, k, **kw)
    b = np.zeros(8, np.float32)
    with pytest.raises(RuntimeError):
        oracle.route_from_logits(L, b, np.zeros((1, 8)))

"""Pins of the f64 oracle to things other than itself: the pages' worked
grouping example, closed forms, invariants, textbook special cases and brute
force on tiny inputs.  Each test names the mistake it is there to catch."""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
import synth
from inputs import dense_weight, numpy_swiglu, unpack_int4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small_layout(E=6, k=2, H=128, I=128, mode=0, rsf=1.0, shared=0, I_shared=128, x_dtype=0):
    return oracle.layout(num_experts=E, top_k=k, hidden=H, intermediate=I, n_shared=shared,
                         shared_intermediate=I_shared if shared else 0, router_mode=mode,
                         x_dtype=x_dtype, routed_scaling_factor=rsf)


def rand_expert(seed, e, H, I):
    """Seeded random packed expert from the generator (canonical layout)."""
    g = synth
    return (g.int4(seed, 0, 4, e, I * H // 2).reshape(I, H // 2),
            g.scales(seed, 0, 5, e, I * H // 64).reshape(I, H // 64),
            g.int4(seed, 0, 6, e, I * H // 2).reshape(I, H // 2),
            g.scales(seed, 0, 7, e, I * H // 64).reshape(I, H // 64),
            g.int4(seed, 0, 8, e, H * I // 2).reshape(H, I // 2),
            g.scales(seed, 0, 9, e, H * I // 64).reshape(H, I // 64))


def logistic(v):
    return 0.5 * (1.0 + np.tanh(0.5 * np.asarray(v, np.float64)))


# ------------------------------------------------------------- dequant --

def test_dequant_exact_hand_computed():
    """Nibble order, two's-complement sign and the 64-wide scale group.
    Bytes 0x10 0x98 0xF7 0x7F hold (low, high) = (0,1) (-8,-7) (7,-1) (-1,7);
    byte 32 = 0x21 holds K indices 64, 65 = (1, 2) in the second group."""
    q = np.zeros(64, np.uint8)
    q[:4] = [0x10, 0x98, 0xF7, 0x7F]
    q[32] = 0x21
    s = np.array([0.5, 0.25], np.float32)
    out = oracle.dequant_row(q, s)
    expect = np.zeros(128)
    expect[:8] = np.array([0, 1, -8, -7, 7, -1, -1, 7]) * 0.5
    expect[64:66] = np.array([1, 2]) * 0.25
    assert np.array_equal(out, expect)


def test_dequant_grid_exhaustive():
    """Every byte value decodes to the integer pair its two nibbles spell."""
    q = np.arange(256, dtype=np.uint8)
    q = np.concatenate([q, q])                  # K = 1024
    s = np.full(16, 1.0, np.float32)
    out = oracle.dequant_row(q, s)
    lo = np.array([(b & 15) - 16 * ((b & 15) >= 8) for b in range(256)] * 2)
    hi = np.array([(b >> 4) - 16 * ((b >> 4) >= 8) for b in range(256)] * 2)
    assert np.array_equal(out[0::2], lo) and np.array_equal(out[1::2], hi)


# --------------------------------------------------------------- top-k --

@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("E,k", [(4, 1), (5, 2), (6, 3), (8, 2), (8, 3)])
def test_topk_matches_bruteforce(mode, E, k):
    """Selection and slot order: the chosen set is the k-subset with the
    largest key sum (keys distinct), listed by descending key."""
    rng = np.random.default_rng(100 * E + k + mode)
    L = small_layout(E=E, k=k, mode=mode, rsf=2.5 if mode else 1.0)
    z = rng.normal(0, 1.5, size=(40, E))
    b = rng.normal(0, 0.1, size=E).astype(np.float32)
    idx, w, key, gap = oracle.route_from_logits(L, b, z)
    keys = z + b.astype(np.float64) if mode == 0 else logistic(z) + b.astype(np.float64)
    for t in range(z.shape[0]):
        best = max(itertools.combinations(range(E), k), key=lambda S: sum(keys[t, list(S)]))
        order = sorted(best, key=lambda e: -keys[t, e])
        assert list(idx[t]) == order
        srt = np.sort(keys[t])[::-1]
        top = k + 1 if k < E else E
        assert gap[t] == pytest.approx(np.min(srt[:top - 1] - srt[1:top]), rel=1e-12)


@pytest.mark.parametrize("mode,E,k", [(1, 256, 8), (1, 1024, 16), (0, 1024, 16), (0, 64, 8)])
def test_topk_large_E_matches_library_sort(mode, E, k):
    """At the sizes the GPU serves (up to 1024 experts, 16 slots) the selection
    is the first k of numpy's stable sort of (-key, id) over the oracle's own
    keys, which match their definition (z + b, or sigmoid(z) + b).  Softmax
    logits are rounded so that equal keys occur: ties go to the lower id.
    Catches a wrong slot order, a lost tie rule or an off-by-one at large E."""
    rng = np.random.default_rng(1000 + E + k + 7 * mode)
    L = small_layout(E=E, k=k, mode=mode, rsf=2.5 if mode else 1.0)
    z = np.round(rng.normal(0, 1.0, size=(48, E)), 2)
    b = rng.normal(0, 0.1, size=E).astype(np.float32) if mode else None
    idx, _, key, _ = oracle.route_from_logits(L, b, z)
    want = logistic(z) + b.astype(np.float64) if mode else z
    np.testing.assert_allclose(key, want, rtol=1e-14, atol=1e-15)
    ties = 0
    for t in range(z.shape[0]):
        order = np.lexsort((np.arange(E), -key[t]))[:k]   # key descending, then id ascending
        assert list(idx[t]) == list(order)
        ties += len(key[t][order]) - len(np.unique(key[t][order]))
    if mode == 0:
        assert ties > 0   # the rounding produced equal keys among the selected slots


def test_topk_ties_go_to_lowest_index():
    L = small_layout(E=6, k=3)
    z = np.array([[1.0, 2.0, 2.0, 0.5, 2.0, 1.0]])
    idx, _, _, gap = oracle.route_from_logits(L, None, z)
    assert list(idx[0]) == [1, 2, 4]
    assert gap[0] == 0.0


@pytest.mark.parametrize("mode,rsf", [(0, 1.0), (1, 2.5), (1, 1.0), (0, 3.0)])
def test_weights_sum_to_rsf(mode, rsf):
    rng = np.random.default_rng(7)
    L = small_layout(E=16, k=4, mode=mode, rsf=rsf)
    z = rng.normal(0, 2, size=(64, 16))
    b = rng.normal(0, 0.1, 16).astype(np.float32)
    _, w, _, _ = oracle.route_from_logits(L, b, z)
    assert np.all(w > 0)
    assert np.max(np.abs(w.sum(1) - rsf)) < 1e-12


def test_softmax_two_selected_is_logistic_of_difference():
    """Renormalised softmax over two selected logits = logistic(z0 - z1)."""
    L = small_layout(E=5, k=2)
    z = np.array([[0.3, -1.0, 2.0, 1.1, -0.2]])
    idx, w, _, _ = oracle.route_from_logits(L, None, z)
    assert list(idx[0]) == [2, 3]
    assert w[0, 0] == pytest.approx(1.0 / (1.0 + math.exp(1.1 - 2.0)), rel=1e-14)
    assert w[0, 1] == pytest.approx(1.0 / (1.0 + math.exp(2.0 - 1.1)), rel=1e-14)


def test_softmax_full_k_is_library_softmax():
    """k = E, no bias: the weights are the plain softmax of the logits."""
    rng = np.random.default_rng(3)
    L = small_layout(E=7, k=7)
    z = rng.normal(0, 2, size=(10, 7))
    idx, w, _, _ = oracle.route_from_logits(L, None, z)
    p = scipy.special.softmax(z, axis=1)
    for t in range(10):
        assert np.allclose(w[t], p[t, idx[t]], rtol=1e-13, atol=0)


def test_softmax_logit_bias_enters_weights():
    """A softmax-mode bias is a logit offset: softmax(z + b) restricted to the selection."""
    L = small_layout(E=3, k=3)
    z = np.array([[0.0, 0.0, 0.0]])
    b = np.array([math.log(2.0), 0.0, math.log(5.0)], np.float32)
    idx, w, _, _ = oracle.route_from_logits(L, b, z)
    assert list(idx[0]) == [2, 0, 1]
    assert np.allclose(w[0], [5 / 8, 2 / 8, 1 / 8], rtol=1e-7)


def test_sigmoid_bias_selects_but_does_not_weigh():
    """noaux_tc: the bias picks the experts, the unbiased sigmoid weighs them.
    sigmoid(ln 3) = 3/4 and sigmoid(0) = 1/2, so with rsf 2.5 the weights are
    2.5 * (3/4, 1/2) / (5/4) = (1.5, 1.0); expert 2 has the largest logit but
    its bias of -5 keeps it out."""
    L = small_layout(E=4, k=2, mode=1, rsf=2.5)
    z = np.array([[math.log(3.0), 0.0, 2.0, -1.0]])
    b = np.array([0.0, 0.0, -5.0, 0.0], np.float32)
    idx, w, _, _ = oracle.route_from_logits(L, b, z)
    assert list(idx[0]) == [0, 1]
    assert np.allclose(w[0], [1.5, 1.0], rtol=1e-14)


def test_sigmoid_equal_scores_split_rsf_evenly():
    L = small_layout(E=6, k=3, mode=1, rsf=2.5)
    z = np.zeros((1, 6))
    b = np.array([0.1, 0.5, -0.2, 0.3, 0.0, 0.2], np.float32)
    idx, w, _, _ = oracle.route_from_logits(L, b, z)
    assert list(idx[0]) == [1, 3, 5]
    assert np.allclose(w[0], [2.5 / 3] * 3, rtol=1e-14)


def test_router_logits_one_hot():
    """z = x . Wr with Wr laid out [H][E]: a one-hot x picks a row of Wr."""
    L = small_layout(E=5, k=1, H=64, I=64)
    rng = np.random.default_rng(1)
    Wr = rng.normal(0, 0.02, (64, 5)).astype(np.float32)
    x = np.zeros((2, 64), np.float32)
    x[0, 17] = 1.0
    x[1, 40] = -2.0
    z = oracle.router_logits(L, oracle.weights(L, Wr), x)
    assert np.array_equal(z[0], Wr[17].astype(np.float64))
    assert np.array_equal(z[1], -2.0 * Wr[40].astype(np.float64))


def test_router_logits_bf16_input():
    """bf16 activations are read exactly (upper half of an f32)."""
    L = small_layout(E=3, k=1, H=64, I=64, x_dtype=1)
    Wr = np.ones((64, 3), np.float32)
    x = np.zeros((1, 64), np.uint16)
    x[0, 0] = 0x3FC0   # 1.5
    x[0, 1] = 0xC010   # -2.25
    z = oracle.router_logits(L, oracle.weights(L, Wr), x)
    assert np.array_equal(z[0], [-0.75] * 3)


# ------------------------------------------------------------ dispatch --

def read_golden(name):
    d = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *vals = line.split()
            d[key] = [int(v) for v in vals]
    return d


def test_dispatch_worked_example():
    g = read_golden("grouping_example.txt")
    idx = np.array(g["routes"], np.int32).reshape(-1, g["top_k"][0])
    counts, offsets, perm, inv = oracle.dispatch(idx, g["num_experts"][0])
    assert list(counts) == g["counts"]
    assert list(offsets) == g["offsets"]
    assert list(perm) == g["perm"]
    assert list(perm[inv]) == list(range(6))


@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (7, 2, 8), (64, 8, 64), (300, 8, 256), (0, 2, 4)])
def test_dispatch_invariants(T, k, E):
    rng = np.random.default_rng(T + k + E)
    idx = np.array([rng.choice(E, k, replace=False) for _ in range(T)], np.int32).reshape(T, k)
    counts, offsets, perm, inv = oracle.dispatch(idx, E)
    assert counts.sum() == T * k
    assert offsets[0] == 0 and np.all(np.diff(offsets) == counts)
    assert sorted(perm) == list(range(T * k))
    assert np.array_equal(perm[inv], np.arange(T * k))
    flat = idx.ravel()
    for e in range(E):
        grp = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[grp] == e)
        assert np.all(np.diff(grp // k) > 0)           # ascending token, stable


# -------------------------------------------------------------- experts --

def test_swiglu_closed_form_one_hot():
    """One-hot x and diagonal weights: g_n = q1*s1*c, u_n = q3*s3*c,
    h_n = g_n * logistic(g_n) * u_n, y_n = q2*s2*h_n."""
    H = I = 64
    j, c = 5, 1.5
    q1 = np.zeros((I, H), np.int64)
    q3 = np.zeros((I, H), np.int64)
    q2 = np.zeros((H, I), np.int64)
    vals1 = np.array([(n % 15) - 7 for n in range(I)])
    vals3 = np.array([((3 * n) % 16) - 8 for n in range(I)])
    vals2 = np.array([((5 * n) % 13) - 6 for n in range(H)])
    q1[:, j] = vals1
    q3[:, j] = vals3
    q2[np.arange(H), np.arange(I)] = vals2

    def pack(qm):
        u = (qm & 0xF).astype(np.uint8)
        return (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)

    s1 = np.full((I, 1), 0.25, np.float32)
    s3 = np.full((I, 1), 0.5, np.float32)
    s2 = np.full((H, 1), 0.125, np.float32)
    x = np.zeros((1, H))
    x[0, j] = c
    y = oracle.expert_ffn(H, I, (pack(q1), s1, pack(q3), s3, pack(q2), s2), x)
    for n in range(H):
        g = vals1[n] * 0.25 * c
        u = vals3[n] * 0.5 * c
        h = g / (1.0 + math.exp(-g)) * u
        assert y[0, n] == pytest.approx(vals2[n] * 0.125 * h, rel=1e-14, abs=1e-300)


def test_expert_ffn_matches_numpy_dense():
    """Transposed operand or dropped gate: the oracle's row-by-row FFN against
    numpy matmuls on the dequantised matrices (H != I)."""
    H, I = 128, 192
    w = rand_expert(11, 0, H, I)
    x = np.random.default_rng(0).normal(size=(3, H))
    assert np.allclose(oracle.expert_ffn(H, I, w, x), numpy_swiglu(w, x), rtol=1e-12, atol=1e-12)


def _layer(L, rng_seed, E, H, I, identical=False, shared=False, bias=None, T=12, x_dtype=0):
    rng = np.random.default_rng(rng_seed)
    Wr = rng.normal(0, 0.1, (H, E)).astype(np.float32)
    ex = {e: rand_expert(rng_seed, 0 if identical else e, H, I) for e in range(E)}
    sh = rand_expert(rng_seed, 999, H, L.shared_intermediate) if shared else None
    x = rng.normal(0, 1, (T, H)).astype(np.float32)
    return Wr, ex, sh, x


@pytest.mark.parametrize("mode,rsf", [(0, 1.0), (1, 2.5)])
def test_identical_experts_equal_dense_ffn(mode, rsf):
    """E identical experts: the output is one dense SwiGLU(x) times sum(w) = rsf."""
    E, H, I = 4, 128, 128
    L = small_layout(E=E, k=2, H=H, I=I, mode=mode, rsf=rsf)
    Wr, ex, _, x = _layer(L, 5, E, H, I, identical=True)
    b = np.zeros(E, np.float32) if mode == 1 else None
    out, _, _ = oracle.moe_forward(L, oracle.weights(L, Wr, b, ex), x)
    ref = rsf * numpy_swiglu(ex[0], x.astype(np.float64))
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-11 * np.abs(ref).max())


def test_topk_equal_E_is_dense_mixture():
    """k = E softmax: out = sum_e softmax(x Wr)_e * FFN_e(x)."""
    E, H, I = 4, 128, 128
    L = small_layout(E=E, k=E, H=H, I=I)
    Wr, ex, _, x = _layer(L, 6, E, H, I)
    out, _, _ = oracle.moe_forward(L, oracle.weights(L, Wr, None, ex), x)
    xd = x.astype(np.float64)
    p = scipy.special.softmax(xd @ Wr.astype(np.float64), axis=1)
    ref = sum(p[:, [e]] * numpy_swiglu(ex[e], xd) for e in range(E))
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-11 * np.abs(ref).max())


def test_layer_is_weighted_sum_of_selected_experts():
    """Grouping, scatter and combine: out[t] = sum_j w[t,j] FFN_idx[t,j](x_t) + shared."""
    E, H, I = 6, 128, 128
    L = small_layout(E=E, k=3, H=H, I=I, mode=1, rsf=2.5, shared=1, I_shared=192)
    Wr, ex, sh, x = _layer(L, 8, E, H, I, shared=True, T=20)
    b = np.random.default_rng(9).normal(0, 0.1, E).astype(np.float32)
    out, idx, w = oracle.moe_forward(L, oracle.weights(L, Wr, b, ex, sh), x)
    xd = x.astype(np.float64)
    ref = numpy_swiglu(sh, xd)
    for t in range(x.shape[0]):
        for j in range(3):
            ref[t] += w[t, j] * numpy_swiglu(ex[idx[t, j]], xd[t:t + 1])[0]
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-11 * np.abs(ref).max())


def test_shared_expert_added_with_weight_one():
    E, H, I = 5, 128, 128
    L1 = small_layout(E=E, k=2, H=H, I=I, mode=1, rsf=2.5, shared=1, I_shared=128)
    L0 = small_layout(E=E, k=2, H=H, I=I, mode=1, rsf=2.5, shared=0)
    Wr, ex, sh, x = _layer(L1, 12, E, H, I, shared=True)
    b = np.zeros(E, np.float32)
    o1, _, _ = oracle.moe_forward(L1, oracle.weights(L1, Wr, b, ex, sh), x)
    o0, _, _ = oracle.moe_forward(L0, oracle.weights(L0, Wr, b, ex), x)
    ref = numpy_swiglu(sh, x.astype(np.float64))
    assert np.allclose(o1 - o0, ref, rtol=1e-10, atol=1e-10 * np.abs(ref).max())


def test_token_permutation_equivariance():
    E, H, I = 6, 128, 128
    L = small_layout(E=E, k=2, H=H, I=I)
    Wr, ex, _, x = _layer(L, 13, E, H, I, T=16)
    W = oracle.weights(L, Wr, None, ex)
    out, idx, _ = oracle.moe_forward(L, W, x)
    pi = np.random.default_rng(0).permutation(16)
    out2, idx2, _ = oracle.moe_forward(L, W, x[pi])
    assert np.array_equal(idx2, idx[pi])
    assert np.allclose(out2, out[pi], rtol=1e-13, atol=1e-13 * np.abs(out).max())


def test_expert_id_permutation_invariance():
    """Relabelling experts consistently in Wr, bias and weights changes nothing."""
    E, H, I = 6, 128, 128
    L = small_layout(E=E, k=2, H=H, I=I, mode=1, rsf=2.5)
    Wr, ex, _, x = _layer(L, 14, E, H, I, T=16)
    b = np.random.default_rng(2).normal(0, 0.1, E).astype(np.float32)
    out, idx, _ = oracle.moe_forward(L, oracle.weights(L, Wr, b, ex), x)
    sigma = np.random.default_rng(1).permutation(E)       # new id of old expert e = sigma[e]
    Wr2 = np.empty_like(Wr)
    b2 = np.empty_like(b)
    ex2 = {}
    for e in range(E):
        Wr2[:, sigma[e]] = Wr[:, e]
        b2[sigma[e]] = b[e]
        ex2[sigma[e]] = ex[e]
    out2, idx2, _ = oracle.moe_forward(L, oracle.weights(L, Wr2, b2, ex2), x)
    assert np.array_equal(idx2, sigma[idx])
    assert np.allclose(out2, out, rtol=1e-13, atol=1e-13 * np.abs(out).max())


def test_dense_weight_helper_agrees_with_oracle_dequant():
    """The numpy unpack used by the pins and the oracle's dequant agree."""
    w = rand_expert(21, 3, 128, 64)
    D = dense_weight(w[0], w[1])
    for r in (0, 17, 63):
        assert np.array_equal(oracle.dequant_row(w[0][r], w[1][r]), D[r])
    assert unpack_int4(np.array([0x98], np.uint8)).tolist() == [-8, -7]


# --------------------------------------------------------------- norm --

def test_rmsnorm_closed_form():
    c, eps, H = 3.0, 1e-6, 64
    x = np.tile(np.array([c, -c], np.float32), H // 2)[None, :]
    out = oracle.rmsnorm(x, eps)
    r = c / math.sqrt(c * c + eps)
    assert np.allclose(out[0], np.tile([r, -r], H // 2), rtol=1e-15)


# ---------------------------------------------------------- boundaries --

def test_empty_and_bad_arguments():
    L = small_layout(E=4, k=2, H=64, I=64)
    z = np.zeros((0, 4))
    idx, w, _, _ = oracle.route_from_logits(L, None, z)
    assert idx.shape == (0, 2)
    bad = small_layout(E=4, k=5, H=64, I=64)
    with pytest.raises(RuntimeError, match="-2"):
        oracle.route_from_logits(bad, None, np.zeros((1, 4)))
    with pytest.raises(RuntimeError, match="-2"):
        oracle.dispatch(np.array([[0, 7]], np.int32), 4)

"""Test-side helpers: seeded workload inputs with top-k margin control, and an
independent numpy restatement of dense pieces used only to pin the oracle."""
import numpy as np

import oracle
import synth

MARGIN = 1e-4


def unpack_int4(q):
    """Packed bytes [..., K/2] -> int8 [..., K]; the even K index is the low
    nibble and a nibble is two's complement."""
    q = np.asarray(q, np.uint8)
    lo = (q & 0x0F).astype(np.int16)
    hi = (q >> 4).astype(np.int16)
    v = np.stack([lo, hi], axis=-1).reshape(*q.shape[:-1], q.shape[-1] * 2)
    return np.where(v >= 8, v - 16, v).astype(np.int8)


def dense_weight(q, s):
    """[N][K/2] packed + [N][K/64] scales -> [N][K] f64."""
    v = unpack_int4(q).astype(np.float64)
    return v * np.repeat(np.asarray(s, np.float64), 64, axis=-1)


def numpy_swiglu(w, x):
    """y = W2 (silu(W1 x) * W3 x) with numpy matmuls; x [n][H] f64."""
    W1 = dense_weight(w[0], w[1])
    W3 = dense_weight(w[2], w[3])
    W2 = dense_weight(w[4], w[5])
    g = x @ W1.T
    u = x @ W3.T
    h = g * (0.5 * (1.0 + np.tanh(0.5 * g))) * u   # g * logistic(g), via tanh
    return h @ W2.T


def margin_x(wl, T, Wr, bias, margin=MARGIN, max_attempts=256):
    """x rows whose oracle top-(k+1) keys are separated by >= margin; a row that
    fails is redrawn from the next attempt stream.  Returns (x, attempts)."""
    L = oracle.layout(wl)
    W = oracle.weights(L, Wr, bias)
    attempts = np.zeros(T, np.int64)
    x = synth.x_rows(wl, T, attempts)
    if T == 0:
        return x, attempts
    _, _, _, gap = oracle.route(L, W, x)
    bad = np.nonzero(gap < margin)[0]
    while bad.size:
        attempts[bad] += 1
        if attempts.max() > max_attempts:
            raise RuntimeError("margin rejection did not converge")
        for t in bad:
            x[t] = _row(wl, t, attempts[t])
        _, _, _, g2 = oracle.route(L, W, x[bad])
        bad = bad[g2 < margin]
    return x, attempts


def _row(wl, t, attempt):
    fill = synth.normal_bf16 if wl.x_dtype == synth.workloads.X_BF16 else synth.normal_f32
    return fill(wl.seed, 0, synth.T_X, int(attempt), wl.H, 1.0, start=t * wl.H)


def oracle_weights_for(wl, layer, Wr, bias, experts_needed, shared=True):
    L = oracle.layout(wl)
    ex = {int(e): synth.expert_weights(wl, layer, int(e)) for e in experts_needed}
    sh = synth.expert_weights(wl, layer, synth.SHARED_EXPERT) if (wl.n_shared and shared) else None
    return L, oracle.weights(L, Wr, bias, ex, sh), ex, sh

"""ctypes wrapper of the f64 oracle (moe_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the test suite, the package smoke check
and the benchmark's CPU-baseline leg, never by the CUDA path.
"""
import ctypes

import numpy as np

from . import _build

_lib = None


class Layout(ctypes.Structure):
    _fields_ = [("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("shared_intermediate", ctypes.c_int32),
                ("router_mode", ctypes.c_int32), ("x_dtype", ctypes.c_int32),
                ("routed_scaling_factor", ctypes.c_double), ("n_group", ctypes.c_int32),
                ("topk_group", ctypes.c_int32), ("top_p", ctypes.c_double)]


_PP = ctypes.POINTER(ctypes.c_void_p)


class Weights(ctypes.Structure):
    _fields_ = [("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("w1_q", _PP), ("w1_s", _PP), ("w3_q", _PP), ("w3_s", _PP),
                ("w2_q", _PP), ("w2_s", _PP),
                ("sw1_q", ctypes.c_void_p), ("sw3_q", ctypes.c_void_p), ("sw2_q", ctypes.c_void_p),
                ("sw1_s", ctypes.c_void_p), ("sw3_s", ctypes.c_void_p), ("sw2_s", ctypes.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(_build.build())
        P = ctypes.c_void_p
        i = ctypes.c_int
        _lib.oracle_router_logits.argtypes = [P, P, P, i, P]
        _lib.oracle_route.argtypes = [P, P, P, i, P, P, P, P]
        _lib.oracle_route_from_logits.argtypes = [P, P, P, i, P, P, P, P]
        _lib.oracle_dispatch.argtypes = [P, i, i, i, P, P, P, P]
        _lib.oracle_dequant_row.argtypes = [P, P, i, P]
        _lib.oracle_expert_ffn.argtypes = [i, i, P, P, P, P, P, P, P, i, P]
        _lib.oracle_moe_forward.argtypes = [P, P, P, i, P, P, P]
        _lib.oracle_rmsnorm.argtypes = [P, i, i, ctypes.c_double, P]
        _lib.oracle_rmsnorm.restype = ctypes.c_int
        for f in ("oracle_router_logits", "oracle_route", "oracle_route_from_logits",
                  "oracle_dispatch", "oracle_dequant_row", "oracle_expert_ffn",
                  "oracle_moe_forward"):
            getattr(_lib, f).restype = ctypes.c_int
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError("%s returned %d" % (what, rc))


def layout(wl=None, **kw):
    """Layout from a synth Workload (or keyword fields)."""
    if wl is not None:
        kw = dict(num_experts=wl.E, top_k=wl.k, hidden=wl.H, intermediate=wl.I,
                  n_shared=wl.n_shared, shared_intermediate=wl.I_shared,
                  router_mode=wl.router_mode, x_dtype=wl.x_dtype,
                  routed_scaling_factor=wl.rsf, n_group=wl.n_group,
                  topk_group=wl.topk_group, top_p=wl.top_p) | kw
    return Layout(**kw)


class _Holder:
    """Keeps numpy arrays and ctypes arrays alive while a Weights struct is in use."""

    def __init__(self):
        self.keep = []


def weights(L, router_w, router_bias=None, experts=None, shared=None):
    """experts: dict e -> (w1q, w1s, w3q, w3s, w2q, w2s) canonical arrays (only
    the experts that are needed); shared: the same tuple or None."""
    hold = _Holder()
    E = L.num_experts
    router_w = np.ascontiguousarray(router_w, np.float32)
    hold.keep.append(router_w)
    if router_bias is not None:
        router_bias = np.ascontiguousarray(router_bias, np.float32)
        hold.keep.append(router_bias)
    arrs = []
    for slot in range(6):
        a = (ctypes.c_void_p * E)()
        for e, tup in (experts or {}).items():
            t = np.ascontiguousarray(tup[slot])
            hold.keep.append(t)
            a[e] = t.ctypes.data
        hold.keep.append(a)
        arrs.append(ctypes.cast(a, _PP))
    sh = [None] * 6
    if shared is not None:
        for slot in range(6):
            t = np.ascontiguousarray(shared[slot])
            hold.keep.append(t)
            sh[slot] = t.ctypes.data
    W = Weights(router_w.ctypes.data, None if router_bias is None else router_bias.ctypes.data,
                arrs[0], arrs[1], arrs[2], arrs[3], arrs[4], arrs[5],
                sh[0], sh[2], sh[4], sh[1], sh[3], sh[5])
    W._hold = hold
    return W


def router_logits(L, W, x):
    x = np.ascontiguousarray(x)
    T = x.shape[0]
    z = np.zeros((T, L.num_experts), np.float64)
    _check(lib().oracle_router_logits(ctypes.byref(L), ctypes.byref(W), _p(x), T, _p(z)),
           "oracle_router_logits")
    return z


def route(L, W, x):
    """-> idx [T][k] i32, w [T][k] f64, key [T][E] f64, gap [T] f64."""
    x = np.ascontiguousarray(x)
    T = x.shape[0]
    idx = np.zeros((T, L.top_k), np.int32)
    w = np.zeros((T, L.top_k), np.float64)
    key = np.zeros((T, L.num_experts), np.float64)
    gap = np.zeros(T, np.float64)
    _check(lib().oracle_route(ctypes.byref(L), ctypes.byref(W), _p(x), T, _p(idx), _p(w),
                              _p(key), _p(gap)), "oracle_route")
    return idx, w, key, gap


def route_from_logits(L, router_bias, z):
    z = np.ascontiguousarray(z, np.float64)
    T = z.shape[0]
    b = None if router_bias is None else np.ascontiguousarray(router_bias, np.float32)
    idx = np.zeros((T, L.top_k), np.int32)
    w = np.zeros((T, L.top_k), np.float64)
    key = np.zeros((T, L.num_experts), np.float64)
    gap = np.zeros(T, np.float64)
    _check(lib().oracle_route_from_logits(ctypes.byref(L), _p(b), _p(z), T, _p(idx), _p(w),
                                          _p(key), _p(gap)), "oracle_route_from_logits")
    return idx, w, key, gap


def dispatch(idx, E):
    """-> counts [E], offsets [E+1], perm [T*k], inv [T*k] (all i32)."""
    idx = np.ascontiguousarray(idx, np.int32)
    T, k = idx.shape
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(T * k, np.int32)
    inv = np.zeros(T * k, np.int32)
    _check(lib().oracle_dispatch(_p(idx), T, k, E, _p(counts), _p(offsets), _p(perm), _p(inv)),
           "oracle_dispatch")
    return counts, offsets, perm, inv


def dequant_row(q, s):
    q = np.ascontiguousarray(q, np.uint8)
    s = np.ascontiguousarray(s, np.float32)
    K = 2 * q.size
    out = np.zeros(K, np.float64)
    _check(lib().oracle_dequant_row(_p(q), _p(s), K, _p(out)), "oracle_dequant_row")
    return out


def expert_ffn(H, I, w, x):
    """w = (w1q, w1s, w3q, w3s, w2q, w2s); x [n][H] f64 -> y [n][H] f64."""
    x = np.ascontiguousarray(x, np.float64)
    n = x.shape[0]
    y = np.zeros((n, H), np.float64)
    ws = [np.ascontiguousarray(a) for a in w]
    _check(lib().oracle_expert_ffn(H, I, *[_p(a) for a in ws], _p(x), n, _p(y)),
           "oracle_expert_ffn")
    return y


def moe_forward(L, W, x):
    """-> out [T][H] f64, idx [T][k], w [T][k]."""
    x = np.ascontiguousarray(x)
    T = x.shape[0]
    out = np.zeros((T, L.hidden), np.float64)
    idx = np.zeros((T, L.top_k), np.int32)
    w = np.zeros((T, L.top_k), np.float64)
    _check(lib().oracle_moe_forward(ctypes.byref(L), ctypes.byref(W), _p(x), T, _p(out),
                                    _p(idx), _p(w)), "oracle_moe_forward")
    return out, idx, w


def rmsnorm(x, eps=1e-6):
    """x [T][H] f32 -> x / sqrt(mean(x^2) + eps) in f64."""
    x = np.ascontiguousarray(x, np.float32)
    T, H = x.shape
    out = np.zeros((T, H), np.float64)
    _check(lib().oracle_rmsnorm(_p(x), T, H, float(eps), _p(out)), "oracle_rmsnorm")
    return out

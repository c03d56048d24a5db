"""Seeded synthetic inputs for the MoE layer (see synth.h for the definitions).

Host-side fills come from libsynth.so; weights too large for a host round-trip
are filled in HBM by libsynth_dev.so with identical bits.  Nothing here
computes any part of the layer.
"""
import ctypes
import os

import numpy as np

from . import workloads
from .workloads import Workload, BY_NAME, ALL  # noqa: F401

T_X, T_WR, T_BIAS = 1, 2, 3
T_W1Q, T_W1S, T_W3Q, T_W3S, T_W2Q, T_W2S = 4, 5, 6, 7, 8, 9
SHARED_EXPERT = 0xFFFFFFFF

_HERE = os.path.dirname(os.path.abspath(__file__))
_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        from . import _build
        so = _build.build_host()
        lib = ctypes.CDLL(so)
        u64, u32 = ctypes.c_uint64, ctypes.c_uint32
        for name, outp, extra in (("synth_fill_int4", ctypes.c_void_p, []),
                                  ("synth_fill_scales", ctypes.c_void_p, []),
                                  ("synth_fill_normal_f32", ctypes.c_void_p, [ctypes.c_double]),
                                  ("synth_fill_normal_bf16", ctypes.c_void_p, [ctypes.c_double])):
            f = getattr(lib, name)
            f.restype = None
            f.argtypes = [u64, u32, u32, u32, u64, u64] + extra + [outp]
        lib.synth_draw_at.restype = u64
        lib.synth_draw_at.argtypes = [u64, u32, u32, u32, u64]
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        so = os.path.join(_HERE, "libsynth_dev.so")
        if not os.path.exists(so):
            raise RuntimeError("synth/libsynth_dev.so is not built; run __graft_entry__.build()")
        lib = ctypes.CDLL(so)
        for name in ("synth_dev_fill_int4", "synth_dev_fill_scales"):
            f = getattr(lib, name)
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                          ctypes.c_uint64, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p]
        _dev = lib
    return _dev


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


# ----------------------------------------------------------------- fills --

def int4(seed, layer, tensor, expert, n_bytes, start=0):
    out = np.empty(n_bytes, np.uint8)
    _host_lib().synth_fill_int4(seed, layer, tensor, expert, start, n_bytes, _ptr(out))
    return out


def scales(seed, layer, tensor, expert, n, start=0):
    out = np.empty(n, np.float32)
    _host_lib().synth_fill_scales(seed, layer, tensor, expert, start, n, _ptr(out))
    return out


def normal_f32(seed, layer, tensor, expert, n, sigma, start=0):
    out = np.empty(n, np.float32)
    _host_lib().synth_fill_normal_f32(seed, layer, tensor, expert, start, n, float(sigma), _ptr(out))
    return out


def normal_bf16(seed, layer, tensor, expert, n, sigma, start=0):
    out = np.empty(n, np.uint16)
    _host_lib().synth_fill_normal_bf16(seed, layer, tensor, expert, start, n, float(sigma), _ptr(out))
    return out


def draw(seed, layer, tensor, expert, i):
    return int(_host_lib().synth_draw_at(seed, layer, tensor, expert, i))


def bf16_to_f32(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(f):
    """Round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(f, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


# ------------------------------------------------------ workload tensors --

def router_w(wl: Workload, layer=0):
    """Wr[H][E] f32 ~ N(0, router_sigma)."""
    return normal_f32(wl.seed, layer, T_WR, 0, wl.H * wl.E, wl.router_sigma).reshape(wl.H, wl.E)


def zipf_bias_path(wl: Workload):
    return os.path.join(_HERE, "zipf_bias_%s.txt" % wl.name)


def router_bias(wl: Workload, layer=0):
    """b[E] f32, or None.  "zipf" biases are stored values written by the
    calibration script beside the oracle (see zipf_bias_*.txt headers)."""
    if wl.bias == "none":
        return None
    if wl.bias == "normal":
        return normal_f32(wl.seed, layer, T_BIAS, 0, wl.E, wl.bias_sigma)
    if wl.bias == "zipf":
        p = zipf_bias_path(wl)
        if not os.path.exists(p):
            raise FileNotFoundError("%s missing: run oracle/calibrate_zipf.py" % p)
        b = np.loadtxt(p, dtype=np.float64, comments="#").astype(np.float32)
        assert b.shape == (wl.E,)
        return b
    raise ValueError(wl.bias)


def x_rows(wl: Workload, T, attempts=None, sigma=1.0):
    """x[T][H] ~ N(0, 1) as f32 (x_dtype 0) or bf16 bits (x_dtype 1).
    Row t uses rejection attempt attempts[t] (default 0) as its stream's expert id."""
    if attempts is None:
        attempts = np.zeros(T, np.int64)
    fill = normal_bf16 if wl.x_dtype == workloads.X_BF16 else normal_f32
    rows = [fill(wl.seed, 0, T_X, int(attempts[t]), wl.H, sigma, start=t * wl.H) for t in range(T)]
    dt = np.uint16 if wl.x_dtype == workloads.X_BF16 else np.float32
    return np.stack(rows).astype(dt) if T else np.zeros((0, wl.H), dt)


def x_as_f64(wl: Workload, x):
    if wl.x_dtype == workloads.X_BF16:
        return bf16_to_f32(x).astype(np.float64)
    return np.asarray(x, np.float64)


def expert_weights(wl: Workload, layer, e):
    """Canonical packed weights of routed expert e (or SHARED_EXPERT):
    (w1q [I][H/2] u8, w1s [I][H/64] f32, w3q, w3s, w2q [H][I/2] u8, w2s [H][I/64] f32)."""
    H = wl.H
    I = wl.I_shared if e == SHARED_EXPERT else wl.I
    s = wl.seed
    w1q = int4(s, layer, T_W1Q, e, I * H // 2).reshape(I, H // 2)
    w1s = scales(s, layer, T_W1S, e, I * H // 64).reshape(I, H // 64)
    w3q = int4(s, layer, T_W3Q, e, I * H // 2).reshape(I, H // 2)
    w3s = scales(s, layer, T_W3S, e, I * H // 64).reshape(I, H // 64)
    w2q = int4(s, layer, T_W2Q, e, H * I // 2).reshape(H, I // 2)
    w2s = scales(s, layer, T_W2S, e, H * I // 64).reshape(H, I // 64)
    return w1q, w1s, w3q, w3s, w2q, w2s


def dev_fill_int4(seed, layer, tensor, expert0, per_expert, n_experts, ptr, stream=0):
    rc = _dev_lib().synth_dev_fill_int4(seed, layer, tensor, expert0, per_expert, n_experts,
                                        ctypes.c_void_p(ptr), ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError("synth_dev_fill_int4 failed: %d" % rc)


def dev_fill_scales(seed, layer, tensor, expert0, per_expert, n_experts, ptr, stream=0):
    rc = _dev_lib().synth_dev_fill_scales(seed, layer, tensor, expert0, per_expert, n_experts,
                                          ctypes.c_void_p(ptr), ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError("synth_dev_fill_scales failed: %d" % rc)

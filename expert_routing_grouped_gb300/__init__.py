"""Python binding of libmoe.so, the GB300 (sm_103a) MoE-layer forward library.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch is used for device memory and streams.  The names mirror
include/moe.h.  Importing this module loads the library and raises if it is
missing -- there is no fallback.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK, MOE_ERR_NOMEM, MOE_ERR_ROUTING, MOE_ERR_DEVICE, MOE_ERR_ARG = 0, -1, -2, -3, -4
MOE_ERR_IO, MOE_ERR_ENGINE = -5, -6
MOE_OPT_REGIME, MOE_OPT_SMALL_T_MAX, MOE_OPT_PROFILE, MOE_OPT_USAGE, MOE_OPT_PDL = 1, 2, 3, 4, 5
MOE_OPT_WAIT_LIMIT_US = 6
REGIME_AUTO, REGIME_GEMV, REGIME_TC, REGIME_TC_EXACT = 0, 1, 2, 3
ROUTER_SOFTMAX, ROUTER_SIGMOID, ROUTER_SOFTMAX_RAW = 0, 1, 2
X_F32, X_BF16 = 0, 1

MOE_DBG_IDX, MOE_DBG_W, MOE_DBG_COUNTS, MOE_DBG_OFFSETS, MOE_DBG_PERM, MOE_DBG_INV = range(6)

EXPORTS = ("moe_init", "moe_route", "moe_forward", "moe_forward_residual",
           "moe_forward_residual_norm", "moe_forward_host",
           "moe_rmsnorm_bf16", "moe_set_option", "moe_debug_view", "moe_debug_read",
           "moe_stage_times", "moe_status", "moe_device_bytes", "moe_free", "moe_strerror",
           "moe_route_noalloc", "moe_usage_read", "moe_usage_reset", "moe_engine_id",
           "moe_route_trace_write", "moe_route_trace_read", "moe_set_next_layer")


class MoeLayout(ctypes.Structure):
    _fields_ = [("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("shared_intermediate", ctypes.c_int32),
                ("router_mode", ctypes.c_int32), ("routed_scaling_factor", ctypes.c_float),
                ("x_dtype", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("n_group", ctypes.c_int32), ("topk_group", ctypes.c_int32),
                ("top_p", ctypes.c_float)]


class MoeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "router_w", "router_bias", "w1_q", "w1_s", "w3_q", "w3_s", "w2_q", "w2_s",
        "sw1_q", "sw1_s", "sw3_q", "sw3_s", "sw2_q", "sw2_s")]


class MoeDebug(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("idx", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("counts", ctypes.c_void_p), ("offsets", ctypes.c_void_p),
                ("perm", ctypes.c_void_p), ("inv", ctypes.c_void_p),
                ("status", ctypes.c_void_p), ("regime", ctypes.c_int32),
                ("launches", ctypes.c_int64)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libmoe.so is not built (run __graft_entry__.build()); "
                          "the MoE layer has no other implementation")
    lib = ctypes.CDLL(LIB_PATH)
    P, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    sig = {
        "moe_init": (i, [P, P, P]),
        "moe_forward": (i, [P, P, i, P, P]),
        "moe_route": (i, [P, P, i, P]),
        "moe_forward_residual": (i, [P, P, i, P, P]),
        "moe_forward_residual_norm": (i, [P, P, i, P, f, P, P]),
        "moe_forward_host": (i, [P, P, i, P, P]),
        "moe_rmsnorm_bf16": (i, [P, i, i, f, P, P]),
        "moe_set_option": (i, [P, i, i]),
        "moe_debug_view": (i, [P, P]),
        "moe_debug_read": (i, [P, i, P, ctypes.c_size_t]),
        "moe_stage_times": (i, [P, P, P, i, P]),
        "moe_status": (i, [P, P]),
        "moe_device_bytes": (ctypes.c_size_t, [P]),
        "moe_free": (None, [P]),
        "moe_strerror": (ctypes.c_char_p, [i]),
        "moe_route_noalloc": (i, [P, i, i, i, i, i, i, f, P, P, P, P, P]),
        "moe_usage_read": (i, [P, P, i]),
        "moe_usage_reset": (i, [P]),
        "moe_set_next_layer": (i, [P, P]),
        "moe_engine_id": (ctypes.c_uint32, [ctypes.c_char_p]),
        "moe_route_trace_write": (i, [ctypes.c_char_p, i, i, ctypes.c_uint32, P]),
        "moe_route_trace_read": (i, [ctypes.c_char_p, i, i, ctypes.c_uint32, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class MoeError(RuntimeError):
    def __init__(self, code, what):
        super().__init__("%s failed: %d (%s)" % (what, code, lib.moe_strerror(code).decode()))
        self.code = code


def _check(rc, what):
    if rc != MOE_OK:
        raise MoeError(rc, what)
    return rc


def _ptr(t):
    """Device or host address of a torch tensor / numpy array (or None)."""
    if t is None:
        return None
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    return t.ctypes.data


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


class MoELayer:
    """One MoE layer: moe_init on construction, moe_forward per call, moe_free on close."""

    def __init__(self, layout: MoeLayout, weights: dict):
        self.layout = layout
        self._handle = ctypes.c_void_p()
        W = MoeWeights(**{k: _ptr(v) for k, v in weights.items()})
        _check(lib.moe_init(ctypes.byref(layout), ctypes.byref(W), ctypes.byref(self._handle)),
               "moe_init")

    @property
    def handle(self):
        return self._handle

    def forward(self, x, T, out, stream=None):
        return _check(lib.moe_forward(self._handle, _ptr(x), T, _ptr(out), _stream(stream)),
                      "moe_forward")

    def route(self, x, T, stream=None):
        return _check(lib.moe_route(self._handle, _ptr(x), T, _stream(stream)), "moe_route")

    def forward_residual(self, x, T, resid, stream=None):
        return _check(lib.moe_forward_residual(self._handle, _ptr(x), T, _ptr(resid),
                                               _stream(stream)), "moe_forward_residual")

    def forward_residual_norm(self, x, T, resid, eps, norm_out, stream=None):
        return _check(lib.moe_forward_residual_norm(self._handle, _ptr(x), T, _ptr(resid),
                                                    float(eps), _ptr(norm_out), _stream(stream)),
                      "moe_forward_residual_norm")

    def forward_host(self, x_host, T, out_host, stream=None):
        return _check(lib.moe_forward_host(self._handle, _ptr(x_host), T, _ptr(out_host),
                                           _stream(stream)), "moe_forward_host")

    def set_option(self, option, value):
        return _check(lib.moe_set_option(self._handle, option, value), "moe_set_option")

    def set_next_layer(self, nxt):
        """moe_set_next_layer: prefetch nxt's router and shared expert into L2
        during this layer's forwards (None clears the link)."""
        self._next = nxt
        return _check(lib.moe_set_next_layer(self._handle, nxt.handle if nxt is not None else None),
                      "moe_set_next_layer")

    def debug_view(self):
        d = MoeDebug()
        _check(lib.moe_debug_view(self._handle, ctypes.byref(d)), "moe_debug_view")
        return d

    def debug_read(self, field):
        """numpy copy of one field of the last forward (see MOE_DBG_*)."""
        import numpy as np
        L = self.layout
        T = self.debug_view().T
        n = {MOE_DBG_IDX: T * L.top_k, MOE_DBG_W: T * L.top_k, MOE_DBG_COUNTS: L.num_experts,
             MOE_DBG_OFFSETS: L.num_experts + 1, MOE_DBG_PERM: T * L.top_k,
             MOE_DBG_INV: T * L.top_k}[field]
        a = np.zeros(n, np.float32 if field == MOE_DBG_W else np.int32)
        _check(lib.moe_debug_read(self._handle, field, a.ctypes.data, a.nbytes), "moe_debug_read")
        return a

    def stage_times(self):
        """[(stage name, ms)] of the last forward (needs MOE_OPT_PROFILE = 1)."""
        ms = (ctypes.c_float * 8)()
        names = (ctypes.c_char_p * 8)()
        n = ctypes.c_int()
        _check(lib.moe_stage_times(self._handle, ms, names, 8, ctypes.byref(n)), "moe_stage_times")
        return [(names[i].decode(), ms[i]) for i in range(n.value)]

    def status(self):
        s = ctypes.c_int32()
        _check(lib.moe_status(self._handle, ctypes.byref(s)), "moe_status")
        return s.value

    def device_bytes(self):
        return lib.moe_device_bytes(self._handle)

    def usage(self):
        """numpy int64 [E]: assignments per expert over the forwards counted
        since init or the last reset (needs MOE_OPT_USAGE = 1)."""
        import numpy as np
        a = np.zeros(self.layout.num_experts, np.int64)
        _check(lib.moe_usage_read(self._handle, a.ctypes.data, a.size), "moe_usage_read")
        return a

    def usage_reset(self):
        return _check(lib.moe_usage_reset(self._handle), "moe_usage_reset")

    def close(self):
        if self._handle:
            lib.moe_free(self._handle)
            self._handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def rmsnorm_bf16(x, T, H, eps, out, stream=None):
    return _check(lib.moe_rmsnorm_bf16(_ptr(x), T, H, eps, _ptr(out), _stream(stream)),
                  "moe_rmsnorm_bf16")


def layout_for(wl, max_tokens):
    """moe_layout from a synthetic workload description (synth.workloads.Workload)."""
    return MoeLayout(num_experts=wl.E, top_k=wl.k, hidden=wl.H, intermediate=wl.I,
                     n_shared=wl.n_shared, shared_intermediate=wl.I_shared,
                     router_mode=wl.router_mode, routed_scaling_factor=wl.rsf,
                     x_dtype=wl.x_dtype, max_tokens=max_tokens, n_group=wl.n_group,
                     topk_group=wl.topk_group, top_p=wl.top_p)


def route_noalloc(x, T, hidden, num_experts, top_k, x_dtype, router_mode, rsf, router_w_eh,
                  router_bias, idx, w, stream=None):
    """moe_route_noalloc: routing with no device allocation (see include/moe.h)."""
    return _check(lib.moe_route_noalloc(_ptr(x), T, hidden, num_experts, top_k, x_dtype,
                                        router_mode, rsf, _ptr(router_w_eh), _ptr(router_bias),
                                        _ptr(idx), _ptr(w), _stream(stream)), "moe_route_noalloc")


def engine_id(name):
    """FNV-1a 32-bit id of an engine name (moe_engine_id)."""
    return lib.moe_engine_id(name.encode())


def route_trace_write(path, counts, engine):
    """Writes counts (int64 [n_layers][n_experts]) as a route_trace usage
    history; engine is a name or a 32-bit id."""
    import numpy as np
    c = np.ascontiguousarray(counts, dtype=np.int64)
    if c.ndim != 2:
        raise ValueError("counts must be [n_layers][n_experts]")
    eid = engine_id(engine) if isinstance(engine, str) else int(engine)
    return _check(lib.moe_route_trace_write(os.fsencode(path), c.shape[0], c.shape[1], eid,
                                            c.ctypes.data), "moe_route_trace_write")


def route_trace_read(path, n_layers, n_experts, engine=0):
    """Reads a route_trace usage history: (counts int64 [n_layers][n_experts],
    engine id found in the file, 0 if none).  engine 0 accepts any writer."""
    import numpy as np
    c = np.zeros((n_layers, n_experts), np.int64)
    found = ctypes.c_uint32()
    eid = engine_id(engine) if isinstance(engine, str) else int(engine)
    _check(lib.moe_route_trace_read(os.fsencode(path), n_layers, n_experts, eid, c.ctypes.data,
                                    ctypes.byref(found)), "moe_route_trace_read")
    return c, found.value

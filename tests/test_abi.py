"""The C ABI without a GPU: the library loads, exports every function that
include/moe.h declares, and rejects bad arguments on the host before any CUDA
call (the pages' return codes: pure-C Colibri tutorial, trdm.cn, §4.2)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_api():
    names = declared_functions()
    for must in ("moe_init", "moe_forward", "moe_free"):
        assert must in names


def test_library_exports_every_declared_symbol():
    import expert_routing_grouped_gb300 as moe
    lib = ctypes.CDLL(moe.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(declared_functions()) == set(moe.EXPORTS)


def _layout(**kw):
    import expert_routing_grouped_gb300 as moe
    base = dict(num_experts=8, top_k=2, hidden=512, intermediate=1024, n_shared=0,
                shared_intermediate=0, router_mode=0, routed_scaling_factor=1.0, x_dtype=0,
                max_tokens=16)
    base.update(kw)
    return moe.MoeLayout(**base)


def _init(layout, weights=True):
    import expert_routing_grouped_gb300 as moe
    dummy = ctypes.c_void_p(16)   # never dereferenced: validation fails first
    W = moe.MoeWeights(**({n: dummy.value for n, _ in moe.MoeWeights._fields_} if weights else {}))
    h = ctypes.c_void_p(1234)
    rc = moe.lib.moe_init(ctypes.byref(layout), ctypes.byref(W), ctypes.byref(h))
    return rc, h


@pytest.mark.parametrize("kw,code", [
    (dict(top_k=0), -2), (dict(top_k=9), -2), (dict(num_experts=0), -2),
    (dict(num_experts=2000, top_k=2), -2), (dict(router_mode=3), -2),
    (dict(routed_scaling_factor=0.0), -2), (dict(top_k=33, num_experts=64), -2),
    (dict(hidden=500), -4), (dict(hidden=0), -4), (dict(intermediate=1000), -4),
    (dict(n_shared=1, shared_intermediate=0), -4), (dict(n_shared=2), -4),
    (dict(x_dtype=5), -4), (dict(max_tokens=0), -4),
    (dict(router_mode=2, n_group=2, topk_group=1), -2),              # groups need sigmoid
    (dict(router_mode=1, n_group=3, topk_group=1), -2),              # 8 % 3
    (dict(router_mode=1, n_group=8, topk_group=2), -2),              # groups of one
    (dict(router_mode=1, n_group=4, topk_group=0), -2),
    (dict(router_mode=1, n_group=4, topk_group=5), -2),
    (dict(router_mode=1, n_group=4, topk_group=1, top_k=3), -2),     # k > 1 group of 2
    (dict(router_mode=1, n_group=64, topk_group=1, num_experts=128), -2),   # > 32 groups
    (dict(n_group=-1), -2), (dict(top_p=-0.5), -2), (dict(top_p=float("nan")), -2),
    (dict(router_mode=4), -2),
])
def test_init_rejects_bad_layout(kw, code):
    rc, h = _init(_layout(**kw))
    assert rc == code
    assert h.value is None


def test_init_rejects_missing_weights():
    rc, h = _init(_layout(), weights=False)
    assert rc == -4 and h.value is None


def test_init_sigmoid_needs_bias():
    import expert_routing_grouped_gb300 as moe
    W = moe.MoeWeights(**{n: 16 for n, _ in moe.MoeWeights._fields_})
    W.router_bias = None
    h = ctypes.c_void_p()
    rc = moe.lib.moe_init(ctypes.byref(_layout(router_mode=1)), ctypes.byref(W), ctypes.byref(h))
    assert rc == -4


def test_null_handle_calls():
    import expert_routing_grouped_gb300 as moe
    assert moe.lib.moe_forward(None, None, 1, None, None) == -4
    assert moe.lib.moe_forward_host(None, None, 1, None, None) == -4
    assert moe.lib.moe_set_option(None, 1, 0) == -4
    assert moe.lib.moe_debug_view(None, None) == -4
    assert moe.lib.moe_device_bytes(None) == 0
    assert moe.lib.moe_usage_read(None, None, 8) == -4
    assert moe.lib.moe_usage_reset(None) == -4
    moe.lib.moe_free(None)
    assert moe.lib.moe_forward_residual_norm(None, None, 1, None, 1e-6, None, None) == -4
    assert moe.lib.moe_rmsnorm_bf16(None, 0, 64, 1e-6, None, None) == 0     # dry run
    assert moe.lib.moe_rmsnorm_bf16(None, 2, 64, 1e-6, None, None) == -4


def test_rmsnorm_rejects_misaligned_pointers():
    """x and out are accessed 16 bytes at a time: an address off the 16-byte
    grid is refused before anything is launched (no device is needed)."""
    import ctypes
    import expert_routing_grouped_gb300 as moe
    P = ctypes.c_void_p
    assert moe.lib.moe_rmsnorm_bf16(P(0x10004), 2, 64, 1e-6, P(0x20000), None) == -4
    assert moe.lib.moe_rmsnorm_bf16(P(0x10000), 2, 64, 1e-6, P(0x20008), None) == -4


def test_strerror():
    import expert_routing_grouped_gb300 as moe
    assert moe.lib.moe_strerror(0) == b"ok"
    assert b"max_tokens" in moe.lib.moe_strerror(-1)
    assert moe.lib.moe_strerror(-2) == b"invalid routing layout"
    assert b"usage-history" in moe.lib.moe_strerror(-5)
    assert b"another engine" in moe.lib.moe_strerror(-6)


@pytest.mark.parametrize("x,w_eh", [(0x1008, 0x2000), (0x1000, 0x2004), (0x1001, 0x2001)])
def test_route_noalloc_rejects_misaligned_pointers(x, w_eh):
    """x and the router rows are read with 16-byte vector loads: a pointer off
    a 16-byte boundary is refused on the host, before any CUDA call (the
    pointers here are never dereferenced)."""
    import expert_routing_grouped_gb300 as moe
    rc = moe.lib.moe_route_noalloc(x, 4, 512, 8, 2, 0, 0, 1.0, w_eh, None, 0x3000, 0x4000,
                                   None)
    assert rc == moe.MOE_ERR_ARG

"""The 8-layer decode stack on the GPU against the f64 oracle.

Each layer: xn = bf16(rmsnorm(x_l)) (`moe_rmsnorm_bf16`), then
x_{l+1} = x_l + MoE_l(xn) (`moe_forward_residual`), as the decode bench runs it.

Only layer 0's input is margin-controlled, so parity is teacher-forced per
layer: the oracle consumes the GPU's own bf16 layer input.  Routing must then
match exactly for every token whose oracle top-(k+1) keys are >= 1e-4 apart;
a token inside that margin may pick either side of the near-tie, so its GPU
choice is only checked to be legal (every expert it differs in sits within the
margin of the oracle's k-th key) and its output is not compared.  The layer
output matches within the GEMV tolerance.  The free-running stack (the oracle
on its own residual stream, f64 with the same bf16 rounding of each layer's
input) is compared by tolerance only."""
import numpy as np
import pytest

import oracle
import synth
from gpu_inputs import make_layer, oracle_layer, rel_l2
from synth.workloads import Workload
from inputs import MARGIN, margin_x

pytestmark = pytest.mark.gpu

GEMV_TOL = 1e-4
FREE_TOL = 1e-3


def legal_choice(gpu_ids, ref_ids, key, margin):
    """Every expert the GPU picked differently lies within `margin` of the
    oracle's k-th key."""
    kth = np.sort(key)[::-1][len(ref_ids) - 1]
    diff = set(gpu_ids) ^ set(ref_ids)
    return all(abs(key[e] - kth) < margin for e in diff)


def test_decode_stack_teacher_forced_and_free_running():
    import torch
    import expert_routing_grouped_gb300 as moe
    dev = torch.device("cuda:0")
    wl = synth.BY_NAME["glm_decode"]
    T, H = 2, wl.H
    # layer 0's input: the decode bench's token rows, margin-controlled for layer 0
    h0, Wr0, b0 = make_layer(wl, 0, 4, dev)
    x0_bits, _ = margin_x(wl, T, Wr0, b0)
    x0 = synth.bf16_to_f32(x0_bits).astype(np.float32)
    resid = torch.from_numpy(x0.copy()).to(dev)
    ox = x0.astype(np.float64)                    # the oracle's free-running residual
    xn = torch.empty(T, H, dtype=torch.int16, device=dev)
    near_ties = 0
    for l in range(wl.layers):
        h, Wr, bias = (h0, Wr0, b0) if l == 0 else make_layer(wl, l, 4, dev)
        moe.rmsnorm_bf16(resid, T, H, 1e-6, xn)
        before = resid.clone()
        h.forward_residual(xn, T, resid)
        torch.cuda.synchronize()
        assert h.status() == 0
        delta = (resid - before).cpu().numpy().astype(np.float64)
        xn_bits = xn.cpu().numpy().view(np.uint16)
        # teacher forcing: the oracle on the GPU's layer input
        ref = oracle_layer(wl, l, xn_bits, Wr, bias)
        gpu_idx = h.debug_read(moe.MOE_DBG_IDX).reshape(T, wl.k)
        same = np.ones(T, bool)
        for t in range(T):
            if ref["gap"][t] >= MARGIN:
                assert np.array_equal(gpu_idx[t], ref["idx"][t]), (l, t)
            elif not np.array_equal(np.sort(gpu_idx[t]), np.sort(ref["idx"][t])):
                assert legal_choice(gpu_idx[t], ref["idx"][t], ref["key"][t], MARGIN), (l, t)
                same[t] = False
                near_ties += 1
        # the residual add rounds to f32: allow its rounding on top of the layer's
        scale = np.abs(ox).max() * 2.0 ** -23 * np.sqrt(H)
        err = np.linalg.norm(delta[same] - ref["out"][same])
        assert err <= GEMV_TOL * np.linalg.norm(ref["out"][same]) + scale, (l, err)
        # free-running oracle on its own stream
        oxn = synth.f32_to_bf16(oracle.rmsnorm(ox.astype(np.float32), 1e-6).astype(np.float32))
        ox = ox + oracle_layer(wl, l, oxn, Wr, bias)["out"]
        if l > 0:
            h.close()
    h0.close()
    got = resid.cpu().numpy()
    assert np.all(np.isfinite(got))
    assert rel_l2(got, ox) <= FREE_TOL, (rel_l2(got, ox), near_ties)


@pytest.mark.parametrize("T", [1, 4])
def test_decode_stack_graph_replay_and_prefetch_bitwise(T):
    """The decode bench times the 8-layer stack as one captured CUDA graph with
    next-layer L2 prefetch links (moe_set_next_layer).  Both must leave the
    results untouched: the eager stack without links, the eager stack with
    links, and two replays of the captured stack with links agree bit for bit
    (the eager stack itself is checked against the oracle above).  So do the
    stack whose pre-norms after the first come from the previous layer's
    combine (moe_forward_residual_norm), eager and replayed: that is the form
    the bench times.  T = 1 runs the GEMV path, whose W13 pass streams the
    shared expert before it waits for the routing kernel; T = 4 the exact
    decode tensor-core kernel."""
    import torch
    import expert_routing_grouped_gb300 as moe
    dev = torch.device("cuda:0")
    wl = synth.BY_NAME["glm_decode"]
    H = wl.H
    layers = [make_layer(wl, l, 4, dev)[0] for l in range(wl.layers)]
    x0 = torch.from_numpy(synth.bf16_to_f32(synth.x_rows(wl, T))).to(dev)
    resid = torch.empty(T, H, device=dev)
    xn = torch.empty(T, H, dtype=torch.int16, device=dev)
    stream = torch.cuda.Stream()

    def stack():
        resid.copy_(x0)
        for lay in layers:
            moe.rmsnorm_bf16(resid, T, H, 1e-6, xn, stream)
            lay.forward_residual(xn, T, resid, stream)

    def stack_fused():
        resid.copy_(x0)
        moe.rmsnorm_bf16(resid, T, H, 1e-6, xn, stream)
        for i, lay in enumerate(layers):
            if i + 1 < len(layers):
                lay.forward_residual_norm(xn, T, resid, 1e-6, xn, stream)
            else:
                lay.forward_residual(xn, T, resid, stream)

    try:
        with torch.cuda.stream(stream):
            stack()
        torch.cuda.synchronize()
        plain = resid.cpu().numpy()
        assert np.all(np.isfinite(plain))
        assert all(lay.status() == 0 for lay in layers)
        for a, b in zip(layers[:-1], layers[1:]):
            a.set_next_layer(b)
        with torch.cuda.stream(stream):
            stack()
        torch.cuda.synchronize()
        assert np.array_equal(resid.cpu().numpy(), plain)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            stack()
        for _ in range(2):
            resid.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(resid.cpu().numpy(), plain)
        assert all(lay.status() == 0 for lay in layers)
        del g
        with torch.cuda.stream(stream):
            stack_fused()
        torch.cuda.synchronize()
        assert np.array_equal(resid.cpu().numpy(), plain)
        gf = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gf, stream=stream):
            stack_fused()
        for _ in range(2):
            resid.zero_()
            xn.zero_()
            gf.replay()
            torch.cuda.synchronize()
            assert np.array_equal(resid.cpu().numpy(), plain)
        assert all(lay.status() == 0 for lay in layers)
        del gf
    finally:
        for lay in layers:
            lay.set_next_layer(None)
        for lay in layers:
            lay.close()


@pytest.mark.parametrize("T", [1, 4, 16])
def test_forward_residual_norm_matches_separate_norm(T):
    """moe_forward_residual_norm = moe_forward_residual followed by
    moe_rmsnorm_bf16 of the updated residual, bit for bit, on each expert path
    (T = 1 GEMV, T = 4 exact decode tensor-core kernel, T = 16 tensor-core
    grouped GEMM), in place (norm_out = x) as the stacked layers use it; and a
    null, misaligned or resid-overlapping norm_out, or a negative eps, is
    rejected before anything is launched."""
    import ctypes
    import torch
    import expert_routing_grouped_gb300 as moe
    dev = torch.device("cuda:0")
    wl = synth.BY_NAME["glm_decode"]
    H = wl.H
    layers = [make_layer(wl, l, 16, dev)[0] for l in range(2)]
    try:
        x0 = torch.from_numpy(synth.bf16_to_f32(synth.x_rows(wl, T))).to(dev)
        xn = torch.empty(T, H, dtype=torch.int16, device=dev)
        # separate calls
        resid = x0.clone()
        moe.rmsnorm_bf16(resid, T, H, 1e-6, xn)
        layers[0].forward_residual(xn, T, resid)
        moe.rmsnorm_bf16(resid, T, H, 1e-6, xn)
        torch.cuda.synchronize()
        r1, n1 = resid.cpu().numpy(), xn.cpu().numpy()
        layers[1].forward_residual(xn, T, resid)
        torch.cuda.synchronize()
        r2 = resid.cpu().numpy()
        # fused, in place
        resid.copy_(x0)
        xn.zero_()
        moe.rmsnorm_bf16(resid, T, H, 1e-6, xn)
        layers[0].forward_residual_norm(xn, T, resid, 1e-6, xn)
        torch.cuda.synchronize()
        assert np.array_equal(resid.cpu().numpy(), r1)
        assert np.array_equal(xn.cpu().numpy(), n1)
        layers[1].forward_residual(xn, T, resid)
        torch.cuda.synchronize()
        assert np.array_equal(resid.cpu().numpy(), r2)
        assert all(lay.status() == 0 for lay in layers)
        assert np.all(np.isfinite(r2))
        # argument checks: nothing launched, resid untouched
        h = layers[0]._handle
        big = torch.empty(T * H + 16, dtype=torch.int16, device=dev)
        P = ctypes.c_void_p
        call = moe.lib.moe_forward_residual_norm
        assert call(h, P(xn.data_ptr()), T, P(resid.data_ptr()), ctypes.c_float(1e-6), None,
                    None) == moe.MOE_ERR_ARG
        assert call(h, P(xn.data_ptr()), T, P(resid.data_ptr()), ctypes.c_float(1e-6),
                    P(big.data_ptr() + 2), None) == moe.MOE_ERR_ARG
        assert call(h, P(xn.data_ptr()), T, P(resid.data_ptr()), ctypes.c_float(1e-6),
                    P(resid.data_ptr() + 16), None) == moe.MOE_ERR_ARG
        assert call(h, P(xn.data_ptr()), T, P(resid.data_ptr()), ctypes.c_float(-1.0),
                    P(big.data_ptr()), None) == moe.MOE_ERR_ARG
        torch.cuda.synchronize()
        assert np.array_equal(resid.cpu().numpy(), r2)
    finally:
        for lay in layers:
            lay.close()


@pytest.mark.parametrize("T", [1, 2])
def test_forward_residual_norm_wide_rows(T):
    """The fused combine and norm on rows longer than 8192 elements (H =
    10240: the norm reads the row's float4s past 2048 back from resid), on
    the GEMV path: bit for bit the separate calls, and the layer output
    within the GEMV tolerance of the oracle."""
    import torch
    import expert_routing_grouped_gb300 as moe
    dev = torch.device("cuda:0")
    wl = Workload("wide_rows", H=10240, E=8, k=2, I=1024, n_shared=1, I_shared=1024,
                  router_mode=1, rsf=2.5, x_dtype=1, tokens=(T,), seed=77, bias="normal",
                  bias_sigma=0.1)
    H = wl.H
    h, Wr, bias = make_layer(wl, 0, 4, dev)
    try:
        h.set_option(moe.MOE_OPT_REGIME, moe.REGIME_GEMV)
        x_bits, _ = margin_x(wl, T, Wr, bias)
        x0 = torch.from_numpy(synth.bf16_to_f32(x_bits).astype(np.float32)).to(dev)
        xn = torch.empty(T, H, dtype=torch.int16, device=dev)
        resid = x0.clone()
        moe.rmsnorm_bf16(resid, T, H, 1e-6, xn)
        xn_in = xn.cpu().numpy().view(np.uint16).copy()
        h.forward_residual(xn, T, resid)
        moe.rmsnorm_bf16(resid, T, H, 1e-6, xn)
        torch.cuda.synchronize()
        r1, n1 = resid.cpu().numpy(), xn.cpu().numpy()
        resid.copy_(x0)
        moe.rmsnorm_bf16(resid, T, H, 1e-6, xn)
        h.forward_residual_norm(xn, T, resid, 1e-6, xn)
        torch.cuda.synchronize()
        assert h.status() == 0
        assert np.array_equal(resid.cpu().numpy(), r1)
        assert np.array_equal(xn.cpu().numpy(), n1)
        ref = oracle_layer(wl, 0, xn_in, Wr, bias)
        delta = r1.astype(np.float64) - x0.cpu().numpy().astype(np.float64)
        scale = np.abs(r1).max() * 2.0 ** -23 * np.sqrt(H)
        assert np.linalg.norm(delta - ref["out"]) <= GEMV_TOL * np.linalg.norm(ref["out"]) + scale
    finally:
        h.close()

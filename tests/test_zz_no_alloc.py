"""moe_route_noalloc: routing with no device allocation, for callers that
cannot call cudaMalloc (inside stream capture, in hot loops that must not
synchronise the device, or under another allocator).  It must give the same
routing as the regular entry point.  This file sorts last so that a run
stopping at the first failure has run every other test already."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

W_TOL = 5e-5   # the routing-weight tolerance of the other GPU tests


@pytest.mark.parametrize("name", ["glm_decode", "olmoe"])
def test_noalloc_routing_matches_moe_route(name):
    import torch
    import expert_routing_grouped_gb300 as moe
    from synth.device import device_weights
    dev = torch.device("cuda:0")
    wl = synth.BY_NAME[name]
    t, Wr, bias = device_weights(wl, 0, dev)
    layer = moe.MoELayer(moe.layout_for(wl, 64), t)
    del t
    torch.cuda.empty_cache()
    w_eh = torch.from_numpy(np.ascontiguousarray(Wr.T)).to(dev)       # [E][H]
    b = torch.from_numpy(bias).to(dev) if bias is not None else None
    # two calls in a row with different sizes (the split-K and the tiled router)
    for T in (1, 64):
        x = torch.from_numpy(synth.x_rows(wl, T)).to(dev)
        layer.route(x, T)
        ref_idx = layer.debug_read(moe.MOE_DBG_IDX).reshape(T, wl.k)
        ref_w = layer.debug_read(moe.MOE_DBG_W).reshape(T, wl.k)
        idx = torch.full((T, wl.k), -1, dtype=torch.int32, device=dev)
        w = torch.zeros((T, wl.k), dtype=torch.float32, device=dev)
        moe.route_noalloc(x, T, wl.H, wl.E, wl.k, wl.x_dtype, wl.router_mode, wl.rsf, w_eh, b,
                          idx, w)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), ref_idx)
        assert np.max(np.abs(w.cpu().numpy() - ref_w) / ref_w) <= W_TOL
    layer.close()


def test_noalloc_rejects_oversized_calls():
    import torch
    import expert_routing_grouped_gb300 as moe
    dev = torch.device("cuda:0")
    E, H, T = 1024, 512, 2048          # T * E = 2 M logits > the 1 M-float scratch
    x = torch.zeros(T, H, dtype=torch.float32, device=dev)
    w_eh = torch.zeros(E, H, dtype=torch.float32, device=dev)
    idx = torch.zeros(T, 2, dtype=torch.int32, device=dev)
    w = torch.zeros(T, 2, dtype=torch.float32, device=dev)
    rc = moe.lib.moe_route_noalloc(x.data_ptr(), T, H, E, 2, 0, 0, 1.0, w_eh.data_ptr(), None,
                                   idx.data_ptr(), w.data_ptr(), None)
    assert rc == moe.MOE_ERR_NOMEM
    assert moe.lib.moe_route_noalloc(None, 0, H, E, 2, 0, 0, 1.0, None, None, None, None,
                                     None) == moe.MOE_OK

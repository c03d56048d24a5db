"""GPU-test helpers: build a layer from device-generated weights (same bits as
the host generator the oracle uses), run it through the C ABI, and build the
matching oracle result."""
import numpy as np

import oracle
import synth
from inputs import margin_x, oracle_weights_for

from synth.device import device_weights


def make_layer(wl, layer, max_tokens, dev):
    """moe_init on device-generated weights; the canonical copies are freed after."""
    import torch
    import expert_routing_grouped_gb300 as moe
    t, Wr, bias = device_weights(wl, layer, dev)
    h = moe.MoELayer(moe.layout_for(wl, max_tokens), t)
    del t
    torch.cuda.empty_cache()
    return h, Wr, bias


def to_device_x(wl, x, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev)


def oracle_layer(wl, layer, x, Wr, bias, rows=None):
    """Oracle routing/dispatch for all rows, and the layer output for `rows`
    (all by default; outputs are per-token independent given the routing)."""
    L = oracle.layout(wl)
    W0 = oracle.weights(L, Wr, bias)
    idx, w, key, gap = oracle.route(L, W0, x)
    counts, offsets, perm, inv = oracle.dispatch(idx, wl.E)
    rows = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    needed = np.unique(idx[rows])
    needed = needed[needed >= 0]          # -1: a slot the top-p trim dropped
    L, W, _, _ = oracle_weights_for(wl, layer, Wr, bias, needed)
    out, _, _ = oracle.moe_forward(L, W, x[rows])
    return dict(idx=idx, w=w, key=key, gap=gap, counts=counts, offsets=offsets, perm=perm,
                inv=inv, out=out, rows=rows)


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


__all__ = ["device_weights", "make_layer", "to_device_x", "oracle_layer", "rel_l2", "margin_x"]

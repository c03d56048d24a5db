"""Canonical weights of one synthetic layer generated directly in HBM.

Same bits as the host generator (synth.expert_weights), without a host
round-trip: a 256-expert layer holds 5.5 GB of packed weights and scales.
Returns torch device tensors keyed by the moe_weights field names.
"""
from . import (SHARED_EXPERT, T_W1Q, T_W1S, T_W2Q, T_W2S, T_W3Q, T_W3S, dev_fill_int4,
               dev_fill_scales, router_bias, router_w)

_Q = (("w1_q", T_W1Q), ("w3_q", T_W3Q), ("w2_q", T_W2Q))
_S = (("w1_s", T_W1S), ("w3_s", T_W3S), ("w2_s", T_W2S))


def device_weights(wl, layer, dev):
    """-> (dict of device tensors, Wr [H][E] f32 numpy, bias [E] f32 numpy or None)."""
    import torch
    H, I, E = wl.H, wl.I, wl.E
    t = {}
    for name, tid in _Q:
        per = I * H // 2
        t[name] = torch.empty(E * per, dtype=torch.uint8, device=dev)
        dev_fill_int4(wl.seed, layer, tid, 0, per, E, t[name].data_ptr())
    for name, tid in _S:
        per = I * H // 64
        t[name] = torch.empty(E * per, dtype=torch.float32, device=dev)
        dev_fill_scales(wl.seed, layer, tid, 0, per, E, t[name].data_ptr())
    if wl.n_shared:
        Is = wl.I_shared
        for name, tid in _Q:
            t["s" + name] = torch.empty(Is * H // 2, dtype=torch.uint8, device=dev)
            dev_fill_int4(wl.seed, layer, tid, SHARED_EXPERT, Is * H // 2, 1, t["s" + name].data_ptr())
        for name, tid in _S:
            t["s" + name] = torch.empty(Is * H // 64, dtype=torch.float32, device=dev)
            dev_fill_scales(wl.seed, layer, tid, SHARED_EXPERT, Is * H // 64, 1,
                            t["s" + name].data_ptr())
    Wr = router_w(wl, layer)
    bias = router_bias(wl, layer)
    t["router_w"] = torch.from_numpy(Wr).to(dev)
    if bias is not None:
        t["router_bias"] = torch.from_numpy(bias).to(dev)
    torch.cuda.synchronize()
    return t, Wr, bias

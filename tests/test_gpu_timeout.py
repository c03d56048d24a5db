"""The bounded-wait recovery path of the pipelined tensor-core kernels, driven
without a fault or a hang.  MOE_OPT_WAIT_LIMIT_US = 0 makes every wait between
their roles that is not complete when first tested give up at once -- the
MMA warp's first wait for a dequantised operand always does -- so each forward
sets the device status word to 2 (a wait ran out), stops its roles, drains its
own copies and MMAs, frees its tensor memory and returns.  The forward call
itself succeeds.  With the limit back at its default, the next forward must
match the oracle: the tensor memory was freed, and the split-K arrival
counters of the decode kernel were left in a state the next launch clears."""
import numpy as np
import pytest
import torch

import synth
from gpu_inputs import make_layer, oracle_layer, rel_l2, to_device_x
from inputs import margin_x

pytestmark = pytest.mark.gpu

TIMEOUT = 2
DEFAULT_LIMIT_US = 2000000


@pytest.mark.parametrize("regime,T,tol", [(2, 16, 5e-3), (3, 4, 1e-4)])
def test_wait_limit_runs_out_and_the_next_forward_is_correct(regime, T, tol):
    import expert_routing_grouped_gb300 as moe
    dev = torch.device("cuda:0")
    wl = synth.BY_NAME["tiny"]
    h, Wr, bias = make_layer(wl, 0, 16, dev)
    try:
        x, _ = margin_x(wl, T, Wr, bias)
        ref = oracle_layer(wl, 0, x, Wr, bias)
        xd = to_device_x(wl, x, dev)
        out = torch.zeros(T, wl.H, device=dev)
        h.set_option(moe.MOE_OPT_REGIME, regime)
        h.set_option(moe.MOE_OPT_WAIT_LIMIT_US, 0)
        for _ in range(3):
            assert moe.lib.moe_forward(h.handle, xd.data_ptr(), T, out.data_ptr(), None) == moe.MOE_OK
            assert h.status() == TIMEOUT
            assert h.debug_view().regime == regime
        h.set_option(moe.MOE_OPT_WAIT_LIMIT_US, DEFAULT_LIMIT_US)
        out.fill_(float("nan"))
        h.forward(xd, T, out)
        torch.cuda.synchronize()
        assert h.status() == 0
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got))
        assert rel_l2(got, ref["out"]) <= tol
    finally:
        h.close()


def test_wait_limit_option_rejects_negative():
    import expert_routing_grouped_gb300 as moe
    dev = torch.device("cuda:0")
    h, _, _ = make_layer(synth.BY_NAME["tiny"], 0, 4, dev)
    try:
        assert moe.lib.moe_set_option(h.handle, moe.MOE_OPT_WAIT_LIMIT_US, -1) == moe.MOE_ERR_ARG
    finally:
        h.close()

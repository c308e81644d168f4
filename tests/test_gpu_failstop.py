"""Fail-stop of the single-launch kernel, on the GPU, with nothing faulting.

The ML4 page's persistent decode kernel ("Specialized decode", "Fail-stop")
bounds every in-kernel wait and reports instead of hanging.  Here the test
hook makes one call's first grid-wide wait (each block polls the router
logits the other blocks publish, tagged with the call number) expect a tag
one call ahead -- words nothing writes: the wait must give up after about a
second, moe_check must report the timeout, and the next call on the same
handle must be correct again."""
import time

import numpy as np
import pytest

import gen
from moe_cases import guarded_case
from gpu_util import check_parity, load_moe, out_to_bits, x_to_device

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = -5


@pytest.fixture(scope="module")
def moe():
    return load_moe()


@pytest.mark.parametrize("T", [1, 8])
def test_grid_wait_gives_up_and_the_handle_recovers(moe, orc, T):
    """One token (the h exchange through tagged words) and eight (through
    plain rows and per-slot counters, which the restart clears too)."""
    import torch
    layer, x, _ = guarded_case(1, gen.BASE_SEED + 11, T=T)
    L = moe.MoELayer(layer, max_tokens=8)
    try:
        assert L.info().single_launch_max_tokens >= 1
        xd = x_to_device(x)
        # a clean call first
        out, ids, w = L.forward(xd)
        torch.cuda.synchronize()
        assert moe.moe_check(L.h) == moe.MOE_OK
        good = out_to_bits(out)
        # the stalled call: returns (launch OK), the wait runs out on the GPU
        moe.moe_debug_inject(L.h, moe.MOE_INJECT_WAIT_STALL, 1)
        t0 = time.time()
        L.forward(xd)
        rc = moe.moe_check(L.h)
        waited = time.time() - t0
        assert rc == MOE_ERR_TIMEOUT, (rc, moe.last_error())
        assert 0.5 < waited < 30.0, waited
        # recovered: the next call is correct and matches the clean one
        out2, ids2, w2 = L.forward(xd)
        torch.cuda.synchronize()
        assert moe.moe_check(L.h) == moe.MOE_OK
        assert np.array_equal(out_to_bits(out2), good)
        check_parity(orc, layer, x, out_to_bits(out2), ids2.cpu().numpy(), w2.cpu().numpy())
    finally:
        L.close()


def test_inject_rejects_bad_arguments(moe):
    layer, x, _ = guarded_case(0, gen.BASE_SEED + 12, T=1)
    L = moe.MoELayer(layer, max_tokens=1)
    try:
        with pytest.raises(moe.MoEError):
            moe.moe_debug_inject(L.h, 99, 1)
        with pytest.raises(moe.MoEError):
            moe.moe_debug_inject(L.h, moe.MOE_INJECT_WAIT_STALL, -1)
        moe.moe_debug_inject(L.h, moe.MOE_INJECT_WAIT_STALL, 0)
    finally:
        L.close()

"""The single launch beside other work on the GPU.

Its blocks hand values to each other through tagged words, so every block
must get an SM while the others wait for it.  Here a second stream keeps the
GPU busy with short, self-terminating matrix products (they end by
themselves within milliseconds) while layers run as one launch, launched
plainly (fused = 0) and as a cooperative grid (fused = 1).  Each call must
finish correctly with a clean status: no in-kernel wait may run into its
one-second limit."""
import numpy as np
import pytest
import torch

import gen
from gpu_util import check_parity, load_moe, out_to_bits, x_to_device
from moe_cases import guarded_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return load_moe()


@pytest.mark.parametrize("fused", [0, 1], ids=["plain", "cooperative"])
@pytest.mark.parametrize("cfg", [1, 2])
def test_single_launch_beside_a_busy_stream(moe, orc, cfg, fused):
    layer, x, _ = guarded_case(cfg, gen.BASE_SEED + 80 + cfg)
    T = x.shape[0]
    L = moe.MoELayer(layer, max_tokens=T, fused=fused)
    try:
        assert L.info().single_launch_max_tokens == T
        xd = x_to_device(x)
        side = torch.cuda.Stream()
        main = torch.cuda.Stream()
        a = torch.randn(2048, 2048, device="cuda", dtype=torch.bfloat16)
        outs = []
        torch.cuda.synchronize()
        for rep in range(4):
            with torch.cuda.stream(side):
                for _ in range(8):
                    a = (a @ a).clamp_(-1.0, 1.0)
            with torch.cuda.stream(main):
                out = torch.empty((T, layer["cfg"]["H"]), dtype=torch.bfloat16, device="cuda")
                ids = torch.empty((T, layer["cfg"]["k"]), dtype=torch.int32, device="cuda")
                w = torch.empty((T, layer["cfg"]["k"]), dtype=torch.float32, device="cuda")
                moe.moe_decode_forward(L.h, xd, T, out, ids, w, main)
                outs.append((out, ids, w))
        torch.cuda.synchronize()
        assert moe.moe_check(L.h, main) == moe.MOE_OK, moe.last_error()
        first = out_to_bits(outs[0][0])
        for out, ids, w in outs:
            assert np.array_equal(out_to_bits(out), first)     # every call the same, bit for bit
        check_parity(orc, layer, x, first, outs[0][1].cpu().numpy(), outs[0][2].cpu().numpy())
    finally:
        L.close()

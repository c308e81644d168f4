"""Row a6: the grouped tensor-core path (tcgen05) for steps with more than 8
tokens, against the oracle.

grouped_min_tokens selects which slots take it: -1 none (GEMV kernels only),
1 every slot, 8 the library default (the experts many tokens chose, and the
shared expert)."""
import numpy as np
import pytest

import gen
from moe_cases import guarded_case
from gpu_util import check_parity, load_moe, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return load_moe()


@pytest.mark.parametrize("gmin", [-1, 8, 1], ids=["gemv", "default", "all_grouped"])
def test_zipf64_full_size(moe, orc, gmin):
    """The 64-token Zipf-routed Flint layer: hot experts hold up to ~46 tokens."""
    layer, x, _ = guarded_case(3, gen.BASE_SEED + 3)
    gout, gids, gw = run_gpu(moe, layer, x, grouped_min_tokens=gmin)
    check_parity(orc, layer, x, gout, gids, gw)


SHAPES = [
    # H, E, k, I, S, Is, T
    (256, 17, 2, 320, 1, 192, 13),
    (384, 64, 6, 128, 1, 128, 37),
    (128, 8, 3, 64, 2, 64, 64),      # every slot holds many tokens
    (256, 4, 4, 128, 0, 128, 24),    # no shared expert, all experts selected by all tokens
]


@pytest.mark.parametrize("gmin", [1, 4])
@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_ragged_grouped(moe, orc, shape, gmin):
    H, E, k, I, S, Is, T = shape
    c = dict(name="ragged", T=T, H=H, E=E, k=k, I=I, S=S, Is=Is, zipf=False, normalize=1, routed_scale=1.0)
    layer, x, _ = guarded_case(c, 2000 + H + E + T, full=True)
    gout, gids, gw = run_gpu(moe, layer, x, grouped_min_tokens=gmin)
    check_parity(orc, layer, x, gout, gids, gw)


def test_grouped_large_activations(moe, orc):
    """x * 2^20 (router rows * 2^-20 keep the routing): the power-of-two
    prescales of x and h keep the f16 operands exact."""
    c = dict(name="ragged", T=24, H=256, E=8, k=3, I=128, S=1, Is=128, zipf=False, normalize=1, routed_scale=1.0)
    layer, x, _ = guarded_case(c, 77, full=True)
    import torch
    xs = (x.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** 20)
    xb = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    big = dict(layer)
    big["router_w"] = layer["router_w"] * np.float32(2.0 ** -20)
    gout, gids, gw = run_gpu(moe, big, xb, grouped_min_tokens=1)
    check_parity(orc, big, xb, gout, gids, gw)


def test_grouped_repeatable(moe):
    """Two calls on one handle give identical bits (fixed reduction order)."""
    layer, x, _ = guarded_case(3, gen.BASE_SEED + 31, T=40)
    L = moe.MoELayer(layer, max_tokens=64, grouped_min_tokens=2)
    try:
        a = run_gpu(moe, layer, x, layer_obj=L)[0]
        b = run_gpu(moe, layer, x, layer_obj=L)[0]
        assert np.array_equal(a, b)
    finally:
        L.close()

"""The load-time repack is lossless: decoding the repacked weights with the
kernels' own decoder gives, bit for bit, the oracle's FP32 dequantisation of
the canonical weights (every expert of the tiny layer; sampled experts and the
shared expert of the Flint- and ML4-shaped layers)."""
import numpy as np
import pytest

import gen
from gpu_util import load_moe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return load_moe()


def _check_expert(moe, orc, L, layer, which, e):
    got = L.dequant(which, e).cpu().numpy()
    if which in (0, 2):
        pre = "" if which == 0 else "s"
        codes, sf, gs = layer[pre + "w13"][e], layer[pre + "w13_sf"][e], layer[pre + "w13_gs"][e]
        I = codes.shape[0] // 2
        ref = np.concatenate([orc.dequant(codes[:I], sf[:I], float(gs[0])),
                              orc.dequant(codes[I:], sf[I:], float(gs[1]))])
    else:
        pre = "" if which == 1 else "s"
        ref = orc.dequant(layer[pre + "w2"][e], layer[pre + "w2_sf"][e], float(layer[pre + "w2_gs"][e]))
    assert got.shape == ref.shape
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), (which, e)


def test_tiny_every_expert(moe, orc):
    layer = gen.make_layer(gen.config(0), 12)
    L = moe.MoELayer(layer, max_tokens=1)
    try:
        for e in range(layer["cfg"]["E"]):
            _check_expert(moe, orc, L, layer, 0, e)
            _check_expert(moe, orc, L, layer, 1, e)
        _check_expert(moe, orc, L, layer, 2, 0)
        _check_expert(moe, orc, L, layer, 3, 0)
    finally:
        L.close()


@pytest.mark.parametrize("cfg,experts", [(1, [0, 97, 255]), (4, [5, 127])])
def test_sampled_experts(moe, orc, cfg, experts):
    c = gen.config(cfg)
    layer = gen.make_layer(c, 40 + cfg, experts=experts)
    L = moe.MoELayer(layer, max_tokens=1)
    try:
        for e in experts:
            _check_expert(moe, orc, L, layer, 0, e)
            _check_expert(moe, orc, L, layer, 1, e)
        _check_expert(moe, orc, L, layer, 2, 0)
        _check_expert(moe, orc, L, layer, 3, 0)
    finally:
        L.close()

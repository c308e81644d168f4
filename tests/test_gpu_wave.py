"""The one-wave chain kernels at up to 8 tokens, against the oracle: gate/up
(when H is a multiple of 512) and down + combine (when I is) stream units of
every slot from one 16-warp block per SM.  Shapes where a block's unit range
spans one slot, several slots, the shared expert and routed ones, with and
without a K split, and the full-size ML4- and Inkling-shaped layers run
through the chain ("Day 0 support for Mistral Large 4 on vLLM"; "Inkling 2
Small on vLLM: Day-0 Support")."""
import pytest

from gpu_util import check_parity, load_moe, run_gpu
from moe_cases import guarded_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return load_moe()


SHAPES = [
    # H, E, k, I, S, Is, T
    (512, 8, 2, 512, 1, 512, 1),
    (256, 32, 4, 512, 1, 1024, 8),
    (1024, 64, 6, 1024, 1, 512, 5),
    (128, 16, 3, 2048, 0, 2048, 8),
    (512, 40, 8, 1536, 2, 512, 3),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_wave_kernels_parity(moe, orc, shape):
    H, E, k, I, S, Is, T = shape
    c = dict(name="wave", T=T, H=H, E=E, k=k, I=I, S=S, Is=Is, zipf=False, normalize=1, routed_scale=1.0)
    layer, x, _ = guarded_case(c, 7100 + H + E + T)
    gout, gids, gw = run_gpu(moe, layer, x, fused=-1)
    check_parity(orc, layer, x, gout, gids, gw)


@pytest.mark.parametrize("cfg", [4, 6])
def test_wave_kernels_full_size_repeatable(moe, orc, cfg):
    layer, x, _ = guarded_case(cfg, 808 + cfg)
    L = moe.MoELayer(layer, max_tokens=8, fused=-1)
    try:
        a = run_gpu(moe, layer, x, layer_obj=L)
        b = run_gpu(moe, layer, x, layer_obj=L)
    finally:
        L.close()
    assert (a[0] == b[0]).all()
    check_parity(orc, layer, x, *a)

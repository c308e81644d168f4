"""Softmax routing (score_func = "softmax": the Mistral Large 4 page, section
"Specialized decode", runs a softmax top-4 router) on the GPU against the
oracle, through the C ABI.

Every case runs through moe_decode_forward twice: as the single launch where
the shape allows it (up to 8 tokens: the routing warps' softmax weights) and as
the three-kernel chain (fused = -1).  The chain cases cover the router's
paths: one token group with the router rows split along K (logits summed in
shared memory), several token groups (global expert masks and the second
ticket), the grouped tensor-core path above 8 tokens, and both
normalisations."""
import numpy as np
import pytest

import gen
from gpu_util import check_parity, load_moe, run_gpu
from moe_cases import guarded_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return load_moe()


CASES = [
    # H, E, k, I, S, Is, T, normalize
    (256, 16, 2, 128, 1, 128, 1, 1),     # tiny-shaped, one token
    (1024, 32, 4, 128, 1, 128, 8, 1),    # one token group, router split along K
    (1024, 32, 4, 128, 1, 128, 8, 0),    # the same, weights = full softmax scores
    (384, 64, 6, 128, 1, 128, 37, 1),    # several token groups, grouped path for hot experts
    (256, 128, 4, 256, 1, 256, 5, 0),    # ML4-like: 128 experts, top-4
]


@pytest.mark.parametrize("fused", [0, -1], ids=["single", "chain"])
@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_softmax_routing_parity(moe, orc, case, fused):
    H, E, k, I, S, Is, T, norm = case
    c = dict(name="softmax", T=T, H=H, E=E, k=k, I=I, S=S, Is=Is, zipf=False, normalize=norm,
             routed_scale=1.0 if norm else 1.5, score_func="softmax")
    layer, x, _ = guarded_case(c, 4000 + H + E + T, full=True)
    gout, gids, gw = run_gpu(moe, layer, x, fused=fused)
    check_parity(orc, layer, x, gout, gids, gw)
    if not norm:
        # unnormalised softmax weights are probabilities (times the routed
        # scale 1.5): below 1.5 in total
        assert np.all(gw.sum(axis=1) <= 1.5 * (1.0 + 1e-6))


def test_softmax_ml4_workload(moe, orc):
    """The Mistral-Large-4-shaped layer at T = 8 with its page's softmax router."""
    c = gen.config(4, score_func="softmax")
    layer, x, _ = guarded_case(c, gen.BASE_SEED + 40)
    gout, gids, gw = run_gpu(moe, layer, x)
    check_parity(orc, layer, x, gout, gids, gw)


@pytest.mark.parametrize("T", [1, 2, 8])
def test_softmax_flint_single_launch(moe, orc, T):
    """A Flint-shaped layer with softmax routing runs as one launch (each
    token-count instance) and matches the oracle."""
    c = gen.config(2, score_func="softmax", T=T)
    layer, x, _ = guarded_case(c, gen.BASE_SEED + 41 + T)
    L = moe.MoELayer(layer, max_tokens=T)
    try:
        assert L.info().single_launch_max_tokens == T
        gout, gids, gw = run_gpu(moe, layer, x, layer_obj=L)
    finally:
        L.close()
    check_parity(orc, layer, x, gout, gids, gw)


def test_softmax_layers_take_the_single_launch(moe):
    c = gen.config(0, score_func="softmax")
    layer = gen.make_layer(c, 3)
    L = moe.MoELayer(layer, max_tokens=4)
    try:
        assert L.info().single_launch_max_tokens == 4
    finally:
        L.close()

"""Pins for the oracle's Four-Over-Six NVFP4 activation quantiser and its W4A4
layer (no GPU).  "Inkling 2 Small on vLLM: Day-0 Support", "Mixed-precision
MoE and Four-Over-Six NVFP4": a per-token global scale plus, per 16-element
block, the block maximum scaled to 6 and to 4, keeping the lower mean
absolute reconstruction error; "MoE with fused activation quantisation": the
tokens are quantised before gate/up and the SwiGLU output before down.

The roundings are pinned to their definitions (E2M1 grid midpoints worked by
hand; E4M3 against torch's float8_e4m3fn cast, a library routine); the 6-vs-4
choice to blocks worked by hand (one where 4 reconstructs exactly, one where 6
does, an all-zero tie); the W4A4 layer of one expert to a dense FP64 MLP fed
the quantiser's output (weights from torch's E4M3 decoder).
"""
import math

import numpy as np
import pytest
import torch

from test_oracle_layer import E2M1, bf16_bits, bits_to_f64, dense, pack, random_expert

pytestmark = pytest.mark.filterwarnings("ignore")


@pytest.mark.parametrize("v,code", [
    (0.0, 0), (0.24, 0), (0.25, 0), (0.26, 1), (0.75, 2), (1.25, 2), (1.3, 3), (1.75, 4), (2.5, 4),
    (2.6, 5), (3.5, 6), (5.0, 6), (5.1, 7), (6.0, 7), (100.0, 7), (-0.25, 0), (-0.75, 10), (-5.0, 14),
    (-7.0, 15),
])
def test_e2m1_round_to_nearest_even(orc, v, code):
    # grid 0, .5, 1, 1.5, 2, 3, 4, 6; on a midpoint the code with mantissa bit 0
    assert orc.e2m1_from_f32(v) == code


def test_e4m3_round_matches_torch(orc):
    rng = np.random.default_rng(41)
    vals = np.concatenate([
        np.exp2(rng.uniform(-12, np.log2(448), 4000)),
        # exact midpoints between neighbouring E4M3 values
        np.array([(orc.e4m3(c) + orc.e4m3(c + 1)) / 2 for c in range(0, 0x7E)]),
    ]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for v, r in zip(vals, ref):
        assert orc.e4m3_from_f32(float(v)) == int(r), (float(v), int(r))
    assert orc.e4m3_from_f32(1000.0) == 0x7E       # saturates at 448


def _row(blocks):
    return bf16_bits(np.concatenate([np.asarray(b, np.float64) for b in blocks]))


def test_four_wins_where_it_is_exact(orc):
    # global max 1792 = 4 * 448, so gs = 1: candidate 4 has block scale 448
    # and reconstructs 1792, 896, 448 exactly; candidate 6 has scale
    # e4m3(298.67) = 288: 6.22 -> 6, 3.11 -> 3, 1.56 -> 1.5, error 64+32+16
    blk = [1792, 896, 448] + [0] * 13
    codes, sf, ch, gs, deq = orc.quant_fos(_row([blk]))
    assert gs == 1.0 and ch[0] == 4 and orc.e4m3(int(sf[0])) == 448.0
    assert list(codes[:3]) == [6, 4, 2] and np.array_equal(deq[:3], [1792, 896, 448])


def test_six_wins_where_it_is_exact(orc):
    # block 1 sets gs = 1; block 2 has max 1728 = 6 * 288: candidate 6 (scale
    # 288) is exact, candidate 4 (432, a tie between 416 and 448 -> 448)
    # reconstructs 1728 as 1792 and 864 as 896
    codes, sf, ch, gs, deq = orc.quant_fos(_row([[1792] + [0] * 15, [1728, 864] + [0] * 14]))
    assert gs == 1.0 and ch[1] == 6 and orc.e4m3(int(sf[1])) == 288.0
    assert np.array_equal(deq[16:18], [1728, 864])


def test_tie_goes_to_six_and_zero_rows(orc):
    codes, sf, ch, gs, deq = orc.quant_fos(_row([[1792] + [0] * 15, [0] * 16]))
    assert ch[1] == 6 and np.all(deq[16:] == 0)
    codes, sf, ch, gs, deq = orc.quant_fos(_row([[0] * 32]))
    assert gs == 1.0 and np.all(ch == 6) and np.all(deq == 0)


def test_quantised_values_are_on_the_grid(orc):
    rng = np.random.default_rng(42)
    row = bf16_bits(rng.standard_normal(256) * np.exp2(rng.integers(-4, 5, 256)))
    codes, sf, ch, gs, deq = orc.quant_fos(row)
    v = bits_to_f64(row)
    for b in range(16):
        s = orc.e4m3(int(sf[b]))
        assert s <= 448
        np.testing.assert_array_equal(deq[16 * b:16 * b + 16], E2M1[codes[16 * b:16 * b + 16]] * s * gs)
    # the choice is the lower error (FP32 accumulation in element order)
    assert set(ch.tolist()) <= {4, 6}
    assert np.abs(v - deq).max() <= np.abs(v).max() / 4


def test_w4a4_single_expert_equals_dense_mlp_on_quantised_activations(orc):
    rng = np.random.default_rng(43)
    H, I = 128, 64
    c13, s13, c2, s2 = random_expert(rng, H, I)
    gs13 = np.array([[0.125, 0.25]], np.float32)
    gs2 = np.array([0.5], np.float32)
    c = dict(H=H, E=1, k=1, I=I, S=0, Is=I, normalize=1, routed_scale=1.0, w4a4=1)
    layer = {"cfg": c, "router_w": rng.standard_normal((1, H)).astype(np.float32), "router_b": None,
             "w13": pack(c13)[None], "w13_sf": s13[None], "w13_gs": gs13,
             "w2": pack(c2)[None], "w2_sf": s2[None], "w2_gs": gs2}
    xb = bf16_bits(rng.standard_normal((2, H)))
    out, pre, ids, w = orc.forward(layer, xb)
    W13 = dense(c13, s13, 1.0)
    Wg, Wu, Wd = W13[:I] * 0.125, W13[I:] * 0.25, dense(c2, s2, 0.5)
    for t in range(2):
        xq = orc.quant_fos(xb[t])[4]
        g, u = Wg @ xq, Wu @ xq
        h = np.array([orc.bf16_round(v) for v in (g / (1 + np.exp(-g))) * u])
        hq = orc.quant_fos(bf16_bits(h))[4]
        assert np.allclose(pre[t], Wd @ hq, rtol=1e-12, atol=1e-12)
    # and it differs from the W4A16 layer (the quantisation is on)
    out16, pre16, _, _ = orc.forward(dict(layer, cfg=dict(c, w4a4=0)), xb)
    assert not np.allclose(pre, pre16, rtol=1e-6)

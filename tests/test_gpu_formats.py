"""The other expert formats on the GPU, through the C ABI, against the oracle:
MXFP4 ("Day 0 support for Mistral Large 4 on vLLM", "MXFP4 experts at load,
one layer at a time"), FP8 with 128 x 128 block scales (the same page,
"Highlights": the shared experts of its NVFP4 checkpoint) and MXFP8 ("Inkling 2
Small on vLLM: Day-0 Support", "Mixed-precision MoE and Four-Over-Six NVFP4").

The repack is checked bit for bit with the kernels' own decoders; layers run
as one launch and as the three-kernel chain on ragged shapes (T up to 37:
the grouped tensor-core kernels above 8 tokens for MXFP4, which becomes NVFP4,
the GEMV kernels for the FP8 formats), then the full-size workloads of these
formats.  MXFP4 layers draw their unselected experts as zeros (a NaN scale
code is refused at initialisation, see the last test)."""
import numpy as np
import pytest

import gen
from gpu_util import check_parity, load_moe, run_gpu
from moe_cases import guarded_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return load_moe()


def _fill(*fmts):
    return "zero" if "mxfp4" in fmts else "poison"


@pytest.mark.parametrize("efmt,sfmt", [("mxfp4", "mxfp4"), ("fp8_block", "fp8_block"), ("mxfp8", "mxfp8"),
                                       ("nvfp4", "fp8_block")])
def test_dequant_bit_exact(moe, orc, efmt, sfmt):
    c = dict(name="fmt", T=1, H=384, E=3, k=1, I=192, S=1, Is=320, zipf=False, normalize=1, routed_scale=1.0,
             efmt=efmt, sfmt=sfmt)
    layer = gen.make_layer(c, 51)
    L = moe.MoELayer(layer, max_tokens=1)
    try:
        for which in range(4):
            pre = "" if which < 2 else "s"
            fmt = efmt if which < 2 else sfmt
            I = c["I"] if which < 2 else c["Is"]
            for e in ([0, 2] if which < 2 else [0]):
                got = L.dequant(which, e).cpu().numpy()
                if which in (0, 2):
                    codes, sf = layer[pre + "w13"][e], layer[pre + "w13_sf"][e]
                    gs = layer[pre + "w13_gs"][e] if fmt == "nvfp4" else (1.0, 1.0)
                    rows = 2 * I
                    if fmt == "fp8_block":   # blocks tile the whole [2I, H] matrix
                        ref = orc.dequant_fmt(fmt, codes, sf, 1.0, rows, c["H"])
                    else:
                        cu = codes[:I], codes[I:]
                        su = sf[:I], sf[I:]
                        ref = np.concatenate([orc.dequant_fmt(fmt, cu[h], su[h], float(gs[h]), I, c["H"])
                                              for h in range(2)])
                else:
                    gs = float(layer[pre + "w2_gs"][e]) if fmt == "nvfp4" else 1.0
                    ref = orc.dequant_fmt(fmt, layer[pre + "w2"][e], layer[pre + "w2_sf"][e], gs, c["H"], I)
                assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), (which, e)
    finally:
        L.close()


SHAPES = [
    # H, E, k, I, S, Is, T
    (128, 6, 2, 64, 1, 128, 1),
    (192, 9, 3, 128, 1, 64, 2),
    (320, 33, 4, 192, 1, 128, 7),
    (256, 17, 2, 320, 1, 192, 13),
    (384, 64, 6, 128, 1, 128, 37),
]
FMTS = [("mxfp4", "mxfp4"), ("nvfp4", "fp8_block"), ("mxfp8", "mxfp8"), ("fp8_block", "nvfp4")]


@pytest.mark.parametrize("fused", [0, -1], ids=["auto", "chain"])
@pytest.mark.parametrize("fmts", FMTS, ids=["-".join(f) for f in FMTS])
@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_format_parity_shapes(moe, orc, shape, fmts, fused):
    H, E, k, I, S, Is, T = shape
    c = dict(name="fmt", T=T, H=H, E=E, k=k, I=I, S=S, Is=Is, zipf=False, normalize=1, routed_scale=1.0,
             efmt=fmts[0], sfmt=fmts[1])
    layer, x, _ = guarded_case(c, 6000 + H + E + T, fill=_fill(*fmts))
    gout, gids, gw = run_gpu(moe, layer, x, fused=fused)
    check_parity(orc, layer, x, gout, gids, gw)


@pytest.mark.parametrize("cfg", [5, 6, 7, 8])
def test_format_workloads_full_size(moe, orc, cfg):
    """ML4 with its FP8 block-scaled shared expert, the Inkling-2-Small-shaped
    layer in NVFP4 and in MXFP8, and the Flint-shaped layer in MXFP4, as the
    benchmark runs them."""
    c = gen.config(cfg)
    layer, x, _ = guarded_case(cfg, gen.BASE_SEED + 60 + cfg, fill=_fill(c["efmt"], c["sfmt"]))
    gout, gids, gw = run_gpu(moe, layer, x)
    check_parity(orc, layer, x, gout, gids, gw)


def test_flint_mxfp4_takes_the_single_launch(moe):
    layer = gen.make_layer(gen.config(8), 3, experts=[0], fill="zero")
    L = moe.MoELayer(layer, max_tokens=8)
    try:
        assert L.info().single_launch_max_tokens == 8
    finally:
        L.close()


def test_mxfp4_scales_that_do_not_convert_are_refused(moe):
    c = dict(name="fmt", T=1, H=128, E=2, k=1, I=64, S=0, Is=64, zipf=False, normalize=1, routed_scale=1.0,
             efmt="mxfp4", sfmt="nvfp4")
    layer = gen.make_layer(c, 5, fill="zero")
    sf = layer["w2_sf"].copy()
    sf[1] = 118
    sf[1, 0, 0] = 100                          # 18 octaves apart in expert 1's down matrix
    layer["w2_sf"] = sf
    with pytest.raises(moe.MoEError) as ei:
        moe.MoELayer(layer, max_tokens=1)
    assert ei.value.status == moe.moe.MOE_ERR_UNSUPPORTED
    assert "expert 1 down" in str(ei.value) and "18 octaves" in str(ei.value)
    sf[1, 0, 0] = 255                          # NaN
    layer["w2_sf"] = sf
    with pytest.raises(moe.MoEError) as ei:
        moe.MoELayer(layer, max_tokens=1)
    assert "NaN" in str(ei.value)

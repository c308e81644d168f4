"""Pins for the oracle's other expert formats (no GPU): MXFP4 (E2M1 + one E8M0
scale per 32 values: "Day 0 support for Mistral Large 4 on vLLM", "MXFP4
experts at load, one layer at a time"), FP8 with one FP32 scale per 128 x 128
block (the same page, "Highlights": FP8 block-scaled shared experts; the block
size is a reading) and MXFP8 (E4M3 + one E8M0 scale per 32: "Inkling 2 Small
on vLLM: Day-0 Support", "Mixed-precision MoE and Four-Over-Six NVFP4").

E8M0 is pinned to torch's float8_e8m0fnu decoder (a library routine).  The
placement of the MX and block scales is pinned against the NVFP4 path, which
the other pin files tie to the pages: a layer whose weights are representable
in both formats (E2M1 values, power-of-two scales within E4M3's range) must
give bit-identical results in both.  An FP8-block layer of one expert is also
checked against a dense FP64 MLP whose weights come from torch's E4M3 decoder.
"""
import math

import numpy as np
import pytest
import torch

from test_oracle_layer import bf16_bits, bits_to_f64, pack

pytestmark = pytest.mark.filterwarnings("ignore")


def test_e8m0_exhaustive_vs_torch(orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    for c in range(256):
        v = orc.e8m0(c)
        if c == 255:
            assert math.isnan(v) and math.isnan(ref[c])
        else:
            assert v == ref[c] == 2.0 ** (c - 127), c


def e4m3_code_of(orc, value):
    """The E4M3 code whose value is `value` (exact)."""
    for c in range(256):
        v = orc.e4m3(c)
        if v == value and math.copysign(1.0, v) == math.copysign(1.0, value):
            return c
    raise ValueError(value)


def nvfp4_scale_code(orc, j):
    """E4M3 code of 2^j (exact for -9 <= j <= 8)."""
    return e4m3_code_of(orc, 2.0 ** j)


def both_formats(orc, rng, fmt, rows, cols):
    """A random [rows, cols] matrix representable in `fmt` and in NVFP4 with a
    unit tensor scale: E2M1 values, power-of-two scales (E8M0 per 32 for MX,
    FP32 per 128 x 128 for the FP8 block format).  -> (fmt codes, fmt scales,
    NVFP4 codes, NVFP4 scales)."""
    nib = rng.integers(0, 16, (rows, cols))
    if fmt == "nvfp4":
        j = rng.integers(-9, 9, (rows, cols // 16))
        nv_sf = np.vectorize(lambda v: nvfp4_scale_code(orc, int(v)))(j).astype(np.uint8)
        return pack(nib), nv_sf, pack(nib), nv_sf
    if fmt in ("mxfp4", "mxfp8"):
        j = rng.integers(-9, 9, (rows, cols // 32))           # distinct per block
        sf = (j + 127).astype(np.uint8)
        nv_j = np.repeat(j, 2, axis=1)                         # two 16-blocks per 32-block
    else:
        nbr, nbc = (rows + 127) // 128, (cols + 127) // 128
        j = rng.integers(-9, 9, (nbr, nbc))
        sf = np.ldexp(1.0, j).astype(np.float32)
        nv_j = np.kron(j, np.ones((128, 8), np.int64))[:rows, :cols // 16]
    nv_sf = np.vectorize(lambda v: nvfp4_scale_code(orc, int(v)))(nv_j).astype(np.uint8)
    if fmt == "mxfp4":
        codes = pack(nib)
    else:
        lut = np.array([e4m3_code_of(orc, orc.e2m1(c)) for c in range(16)], np.uint8)
        codes = lut[nib]
    return codes, sf, pack(nib), nv_sf


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp8", "fp8_block"])
def test_dequant_matches_nvfp4_on_shared_values(orc, fmt):
    rng = np.random.default_rng(31)
    rows, cols = 256, 384
    codes, sf, nv_codes, nv_sf = both_formats(orc, rng, fmt, rows, cols)
    a = orc.dequant_fmt(fmt, codes, sf, 1.0, rows, cols)
    b = orc.dequant(nv_codes, nv_sf, 1.0)
    assert np.array_equal(a, b)
    assert orc.dequant_fmt("nvfp4", nv_codes, nv_sf, 1.0, rows, cols).tobytes() == b.tobytes()


def layer_pair(orc, rng, efmt, sfmt, H=256, I=128, E=4, k=2, S=1):
    """The same layer in (efmt, sfmt) and in NVFP4."""
    c = dict(H=H, E=E, k=k, I=I, S=S, Is=I, normalize=1, routed_scale=1.0)
    a = {"cfg": dict(c, efmt=efmt, sfmt=sfmt), "router_w": rng.standard_normal((E, H)).astype(np.float32),
         "router_b": None}
    b = {"cfg": dict(c), "router_w": a["router_w"], "router_b": None}
    for pre, n, fmt in (("", E, efmt), ("s", S, sfmt)):
        parts = {}
        for m, (rows, cols) in (("w13", (2 * I, H)), ("w2", (H, I))):
            mats = [both_formats(orc, rng, fmt, rows, cols) for _ in range(n)]
            a[pre + m] = np.stack([q[0] for q in mats])
            a[pre + m + "_sf"] = np.stack([q[1] for q in mats])
            b[pre + m] = np.stack([q[2] for q in mats])
            b[pre + m + "_sf"] = np.stack([q[3] for q in mats])
        ones13, ones2 = np.ones((n, 2), np.float32), np.ones((n,), np.float32)
        a[pre + "w13_gs"], b[pre + "w13_gs"] = (None if fmt != "nvfp4" else ones13), ones13
        a[pre + "w2_gs"], b[pre + "w2_gs"] = (None if fmt != "nvfp4" else ones2), ones2
    return a, b


@pytest.mark.parametrize("efmt,sfmt", [("mxfp4", "nvfp4"), ("mxfp8", "mxfp8"), ("nvfp4", "fp8_block"),
                                       ("fp8_block", "mxfp4")])
def test_layer_matches_nvfp4_on_shared_values(orc, efmt, sfmt):
    rng = np.random.default_rng(32)
    a, b = layer_pair(orc, rng, efmt, sfmt)
    xb = bf16_bits(rng.standard_normal((3, 256)))
    oa, pa, ia, wa = orc.forward(a, xb)
    ob, pb, ib, wb = orc.forward(b, xb)
    assert np.array_equal(ia, ib) and np.array_equal(wa, wb)
    assert np.array_equal(pa, pb) and np.array_equal(oa, ob)


def test_fp8_block_single_expert_equals_dense_mlp(orc):
    """One FP8-block expert, top-1, no shared expert: the layer is the dense
    SwiGLU MLP of the weights torch's E4M3 decoder and the block scales give."""
    rng = np.random.default_rng(33)
    H, I = 256, 192
    def mat(rows, cols):
        codes = rng.integers(0, 0x7F, (rows, cols)).astype(np.uint8) | (rng.integers(0, 2, (rows, cols)) << 7).astype(np.uint8)
        bs = rng.uniform(0.5, 1.0, ((rows + 127) // 128, (cols + 127) // 128)).astype(np.float32) / 64
        vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        W = vals * np.kron(bs.astype(np.float64), np.ones((128, 128)))[:rows, :cols]
        return codes, bs, W
    c13, s13, W13 = mat(2 * I, H)
    c2, s2, W2 = mat(H, I)
    c = dict(H=H, E=1, k=1, I=I, S=0, Is=I, normalize=1, routed_scale=1.0, efmt="fp8_block")
    layer = {"cfg": c, "router_w": rng.standard_normal((1, H)).astype(np.float32), "router_b": None,
             "w13": c13[None], "w13_sf": s13[None], "w13_gs": None, "w2": c2[None], "w2_sf": s2[None],
             "w2_gs": None}
    xb = bf16_bits(rng.standard_normal((2, H)))
    out, pre, ids, w = orc.forward(layer, xb)
    for t in range(2):
        x = bits_to_f64(xb[t])
        g, u = W13[:I] @ x, W13[I:] @ x
        h = np.array([orc.bf16_round(v) for v in (g / (1 + np.exp(-g))) * u])
        y = W2 @ h
        assert np.allclose(pre[t], y, rtol=1e-12, atol=1e-12)

"""Pins for the oracle's number formats (no GPU).

E2M1 is pinned to its value table {0, 0.5, 1, 1.5, 2, 3, 4, 6} (largest 6 with
4 representable: Inkling 2 Small page, "Mixed-precision MoE and Four-Over-Six
NVFP4"); E4M3 to torch's float8_e4m3fn decoder (a library routine) and to
closed-form values; the BF16 rounding to torch's float32->bfloat16 cast on
float32-representable inputs and to hand-worked ties; the dequantised weight to
an FP32 computation done another way (numpy float32 products).
"""
import math
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.filterwarnings("ignore")

E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_e2m1_golden_file(orc):
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "e2m1_values.txt"))
            if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 16
    for code, val in rows:
        v = orc.e2m1(int(code))
        assert v == float(val) and math.copysign(1.0, v) == math.copysign(1.0, float(val))


def test_e2m1_table_exhaustive(orc):
    for c in range(8):
        assert orc.e2m1(c) == E2M1_TABLE[c]
        neg = orc.e2m1(c + 8)
        assert neg == -E2M1_TABLE[c]
    # code 0x8 is negative zero
    assert math.copysign(1.0, orc.e2m1(8)) == -1.0
    assert max(abs(orc.e2m1(c)) for c in range(16)) == 6.0


def test_e4m3_exhaustive_vs_torch(orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = orc.e4m3(c)
        if c in (0x7F, 0xFF):
            assert math.isnan(v) and math.isnan(ref[c])
        else:
            assert v == ref[c], (c, v, ref[c])


@pytest.mark.parametrize("code,val", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
    (0x20, 0.125), (0x38, 1.0), (0x39, 1.125), (0x7E, 448.0), (0xB8, -1.0),
    (0xFE, -448.0), (0x30, 0.5),
])
def test_e4m3_closed_forms(orc, code, val):
    assert orc.e4m3(code) == val


def test_bf16_round_matches_torch_on_float32_inputs(orc):
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),    # BF16 subnormal range
        np.array([1.0, -1.0, 65504.0, 3.0e38, 1e-45], dtype=np.float32),
    ])
    ref = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float64).numpy()
    for v, r in zip(vals, ref):
        assert orc.bf16_round(float(v)) == r, (v, r)


def test_bf16_round_ties_and_edges(orc):
    u = 2.0 ** -7                           # BF16 ulp at 1
    assert orc.bf16_round(1 + u / 2) == 1.0                   # tie -> even (down)
    assert orc.bf16_round(1 + 3 * u / 2) == 1 + 2 * u          # tie -> even (up)
    assert orc.bf16_round(1 + u / 2 + 2.0 ** -40) == 1 + u     # single rounding from FP64
    assert orc.bf16_round(-(1 + u / 2)) == -1.0
    sub = 2.0 ** -133                                          # smallest BF16 subnormal
    assert orc.bf16_round(sub) == sub
    assert orc.bf16_round(sub / 2) == 0.0                       # tie -> even (zero)
    assert orc.bf16_round(0.75 * sub) == sub
    bmax = (2 - u) * 2.0 ** 127
    assert orc.bf16_round(bmax) == bmax
    assert math.isinf(orc.bf16_round((2 - u / 2) * 2.0 ** 127))   # tie to even overflows
    assert orc.bf16_round(0.0) == 0.0
    assert orc.to_bf16_bits(1.0) == 0x3F80
    assert orc.to_bf16_bits(-2.0) == 0xC000
    assert orc.bf16_bits_to_float(0x3FC0) == 1.5


def _np_pack(vals_codes: np.ndarray) -> np.ndarray:
    """Pack a [rows, cols] array of 4-bit codes: element 2j -> low nibble of
    byte j, 2j+1 -> high nibble (the packing reading used throughout)."""
    lo = vals_codes[:, 0::2].astype(np.uint8)
    hi = vals_codes[:, 1::2].astype(np.uint8)
    return (lo | (hi << 4)).astype(np.uint8)


def test_dequant_matches_float32_products(orc):
    rng = np.random.default_rng(3)
    rows, cols = 24, 96
    codes = rng.integers(0, 16, (rows, cols))
    sf = rng.integers(0, 256, (rows, cols // 16)).astype(np.uint8)
    sf[sf == 0x7F] = 0x38
    sf[sf == 0xFF] = 0xB8
    gs = np.float32(1.0 / math.sqrt(cols))
    e2m1 = np.array(E2M1_TABLE + [-v for v in E2M1_TABLE], dtype=np.float32)
    e4m3 = torch.from_numpy(sf).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    # FP32: the first product is exact in FP32 (<= 6 significant bits), so one
    # FP32 multiply by gs is the single rounding of the exact value.
    expect = (e2m1[codes] * np.repeat(e4m3, 16, axis=1)).astype(np.float32) * gs
    got = orc.dequant(_np_pack(codes), sf, float(gs))
    assert got.dtype == np.float32
    assert np.array_equal(got.view(np.uint32), expect.astype(np.float32).view(np.uint32))


def test_dequant_packing_order(orc):
    # Row 0: element 0 = code 1 (0.5), element 1 = code 7 (6.0) -> byte 0x71.
    codes = np.zeros((1, 16), np.uint8)
    codes[0, 0] = 0x71
    sf = np.full((1, 2), 0x38, np.uint8)     # scale 1.0 for both blocks of 16
    out = orc.dequant(codes, sf, 1.0)
    assert out[0, 0] == 0.5 and out[0, 1] == 6.0
    assert np.all(out[0, 2:] == 0.0)
    # block scale applies to 16 consecutive elements along K
    codes = np.full((1, 16), 0x22, np.uint8)   # every element 1.0
    sf = np.array([[0x30, 0x40]], np.uint8)   # 0.5 then 2.0
    out = orc.dequant(codes, sf, 1.0)
    assert np.all(out[0, :16] == 0.5) and np.all(out[0, 16:] == 2.0)

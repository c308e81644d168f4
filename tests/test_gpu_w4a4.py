"""W4A4 on the GPU, through the C ABI, against the oracle: the activations
quantised to NVFP4 with "Four Over Six" block scales before each GEMM
("Inkling 2 Small on vLLM: Day-0 Support", "Mixed-precision MoE and
Four-Over-Six NVFP4"; "Day 0 support for Mistral Large 4 on vLLM", "MoE with
fused activation quantisation").

The quantiser takes every decision in FP32 on both sides from the same BF16
row, so it is compared bit for bit (values and global scales) on rows built to
reach each branch: both candidates, zero blocks and rows, the E2M1 midpoints,
rows far from 1 in magnitude.  Layers are then compared with the usual
tolerance: the tokens' quantisation is identical on both sides, while the
SwiGLU output h can differ by one BF16 rounding (FP32 GPU accumulation vs the
oracle's FP64), which may move an element, rarely, to a neighbouring code."""
import numpy as np
import pytest
import torch

import gen
import oracle
from gpu_util import check_parity, load_moe, run_gpu, x_to_device
from moe_cases import guarded_case

pytestmark = pytest.mark.gpu

E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


@pytest.fixture(scope="module")
def moe():
    return load_moe()


def _bf16_bits(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _rows(kind: str, n: int, rng: np.random.Generator) -> np.ndarray:
    """Four BF16 rows of length n of one kind."""
    nb = n // 16
    if kind == "normal":
        v = rng.standard_normal((4, n))
    elif kind == "wide":            # every block at its own octave, 2^-20 .. 2^20
        v = rng.standard_normal((4, n)) * np.repeat(2.0 ** rng.integers(-20, 21, (4, nb)), 16, axis=1)
    elif kind == "grid":            # E2M1 values times a power of two per block: 6 and 4 both exact at times
        g = E2M1_GRID[rng.integers(0, 8, (4, n))] * rng.choice([-1.0, 1.0], (4, n))
        v = g * np.repeat(2.0 ** rng.integers(-6, 7, (4, nb)), 16, axis=1)
    elif kind == "midpoints":       # values on the E2M1 decision points of a block maximum of 6
        mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
        v = mids[rng.integers(0, len(mids), (4, n))] * rng.choice([-1.0, 1.0], (4, n))
        v[:, ::16] = 6.0
        v *= np.repeat(2.0 ** rng.integers(-3, 4, (4, nb)), 16, axis=1)
    elif kind == "sparse":          # zero rows, zero blocks, single elements
        v = rng.standard_normal((4, n))
        v[0] = 0.0
        v[1, : 16 * (nb // 2)] = 0.0
        v[2] = 0.0
        v[2, rng.integers(0, n)] = -3.0
        v[3, rng.random(n) < 0.9] = 0.0
    elif kind == "huge":
        v = rng.standard_normal((4, n)) * 2.0 ** 100
    elif kind == "tiny":            # the global scale below FP32's normal range on the last rows
        v = rng.standard_normal((4, n)) * np.array([2.0 ** -100, 2.0 ** -110, 2.0 ** -122, 2.0 ** -126])[:, None]
    else:
        raise ValueError(kind)
    return _bf16_bits(v.astype(np.float32))


KINDS = ["normal", "wide", "grid", "midpoints", "sparse", "huge", "tiny"]


# 1040, 4112 and 40960 split a row over 4 and 8 CTAs with a shorter last
# share; 40960 takes two rounds of 1024 threads in each of its 8 CTAs
@pytest.mark.parametrize("n", [16, 48, 768, 1040, 2560, 4112, 7168, 40960])
@pytest.mark.parametrize("kind", KINDS)
def test_quantiser_bit_exact(moe, kind, n):
    rng = np.random.default_rng(1000 * KINDS.index(kind) + n)
    rows = _rows(kind, n, rng)
    x = x_to_device(rows)
    deq = torch.empty_like(x)
    gs = torch.empty(rows.shape[0], dtype=torch.float32, device="cuda")
    moe.moe_quant_fos(x, rows.shape[0], n, deq, gs)
    torch.cuda.synchronize()
    got = _bits_to_f64(deq.view(torch.int16).cpu().numpy().view(np.uint16))
    ggs = gs.cpu().numpy()
    for r in range(rows.shape[0]):
        _, _, _, ogs, odeq = oracle.quant_fos(rows[r])
        assert np.float32(ogs).view(np.uint32) == ggs[r].view(np.uint32), (r, ogs, ggs[r])
        # the oracle's values carry the global scale; the products e2m1 * e4m3
        # times an FP32 number are exact in FP64, so is the division
        want = odeq / ogs
        bad = np.flatnonzero(got[r] != want)
        assert bad.size == 0, (r, bad[:8], got[r][bad[:8]], want[bad[:8]], rows[r][bad[:8]])


def test_quantiser_in_place_and_stream(moe):
    rng = np.random.default_rng(7)
    rows = _rows("wide", 2048, rng)
    x = x_to_device(rows)
    ref = torch.empty_like(x)
    gs0 = torch.empty(4, dtype=torch.float32, device="cuda")
    moe.moe_quant_fos(x, 4, 2048, ref, gs0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    gs1 = torch.empty_like(gs0)
    with torch.cuda.stream(s):
        moe.moe_quant_fos(x, 4, 2048, x, gs1, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(x.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(gs0, gs1)


SHAPES = [
    # H, E, k, I, S, Is, T
    (128, 6, 2, 64, 1, 128, 1),
    (192, 9, 3, 128, 1, 64, 2),
    (320, 33, 4, 192, 1, 128, 7),
    (256, 17, 2, 320, 1, 192, 13),
    (384, 64, 6, 128, 1, 128, 37),
    (256, 8, 2, 256, 0, 256, 64),
]


@pytest.mark.parametrize("grouped", [0, -1], ids=["grouped", "gemv"])
@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_w4a4_parity_shapes(moe, orc, shape, grouped):
    """Ragged shapes through the chain; above 8 tokens the hot experts take
    the grouped tensor-core kernels ("grouped") or stay on the GEMV kernels."""
    H, E, k, I, S, Is, T = shape
    c = dict(name="w4a4", T=T, H=H, E=E, k=k, I=I, S=S, Is=Is, zipf=False, normalize=1, routed_scale=1.0,
             w4a4=1)
    layer, x, _ = guarded_case(c, 9100 + H + E + T)
    gout, gids, gw = run_gpu(moe, layer, x, grouped_min_tokens=grouped if grouped else 2)
    check_parity(orc, layer, x, gout, gids, gw)


def test_w4a4_differs_from_w4a16(moe, orc):
    """The option changes the result (by the quantisation error, a few
    percent) and the oracle agrees on which result it is."""
    c = dict(name="w4a4", T=3, H=256, E=8, k=2, I=128, S=1, Is=128, zipf=False, normalize=1, routed_scale=1.0)
    layer, x, _ = guarded_case(c, 5, full=True)
    q = dict(layer, cfg=dict(layer["cfg"], w4a4=1))
    g16, _, _ = run_gpu(moe, layer, x)
    g4, gids, gw = run_gpu(moe, q, x)
    check_parity(orc, q, x, g4, gids, gw)
    a, b = _bits_to_f64(g16), _bits_to_f64(g4)
    rel = np.abs(a - b).max() / np.abs(a).max()
    assert 1e-3 < rel < 0.5, rel


def test_w4a4_runs_the_chain(moe):
    layer = gen.make_layer(gen.config(9), 3, experts=[0])
    L = moe.MoELayer(layer, max_tokens=8)
    try:
        assert L.info().single_launch_max_tokens == 0
    finally:
        L.close()


@pytest.mark.parametrize("cfg", [9, 10])
def test_w4a4_workloads_full_size(moe, orc, cfg):
    """The Inkling-2-Small-shaped layer at 8 tokens and the Zipf-routed
    Flint-shaped layer at 64 tokens with W4A4, as the benchmark runs them."""
    layer, x, _ = guarded_case(cfg, gen.BASE_SEED + 90 + cfg)
    gout, gids, gw = run_gpu(moe, layer, x)
    check_parity(orc, layer, x, gout, gids, gw)


@pytest.mark.parametrize("T", [5, 37])
def test_w4a4_stage_entry_points_repeat(moe, orc, T):
    """The stages called one by one, twice in a row on one handle, equal the
    chained forward bit for bit: the token quantiser reads x while the router
    still runs and waits for it last, and a second step's quantiser must not
    overtake the first step's consumers of its outputs."""
    c = dict(name="w4a4", T=T, H=320, E=33, k=4, I=192, S=1, Is=128, zipf=False, normalize=1, routed_scale=1.0,
             w4a4=1)
    layer, x, _ = guarded_case(c, 9300 + T)
    L = moe.MoELayer(layer, max_tokens=T, grouped_min_tokens=2)
    try:
        xd = x_to_device(x)
        H, k = layer["cfg"]["H"], layer["cfg"]["k"]
        outs = []
        for _ in range(2):
            out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
            ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
            w = torch.empty((T, k), dtype=torch.float32, device="cuda")
            moe.moe_stage_route(L.h, xd, T, ids, w)
            moe.moe_stage_gate_up(L.h, xd, T)
            moe.moe_stage_down(L.h, T, out)
            outs.append((out, ids, w))
        torch.cuda.synchronize()
        fout, fids, fw = run_gpu(moe, layer, x, layer_obj=L)
        for out, ids, w in outs:
            assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), fout)
            assert np.array_equal(ids.cpu().numpy(), fids)
            assert np.array_equal(w.cpu().numpy(), fw)
        check_parity(orc, layer, x, fout, fids, fw)
    finally:
        L.close()

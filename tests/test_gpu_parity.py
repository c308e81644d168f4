"""GPU vs oracle parity through the C ABI.

Routing ids must match as sets (and in order where the scores are separated by
the margin), weights within 1e-5 relative, outputs within
|gpu - oracle| <= 1e-2 + 1e-2 |oracle| per element.  The five workloads run at
their full sizes in the launch configuration the benchmark uses; smaller
shapes cover several tiles with ragged ends, the degenerate cases and large
activations."""
import numpy as np
import pytest
import torch

import gen
from gpu_util import check_parity, load_moe, out_to_bits, run_gpu, x_to_device
from moe_cases import guarded_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return load_moe()


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
def test_workload_full_size(moe, orc, cfg):
    """moe_decode_forward as the benchmark runs it (single launch where the
    shape allows it)."""
    layer, x, _ = guarded_case(cfg, gen.BASE_SEED + cfg)
    gout, gids, gw = run_gpu(moe, layer, x)
    check_parity(orc, layer, x, gout, gids, gw)


@pytest.mark.parametrize("cfg", [0, 1, 2])
def test_workload_three_kernel_chain(moe, orc, cfg):
    """The same workloads through the moe_stage_* chain (fused = -1)."""
    layer, x, _ = guarded_case(cfg, gen.BASE_SEED + 10 + cfg)
    gout, gids, gw = run_gpu(moe, layer, x, fused=-1)
    check_parity(orc, layer, x, gout, gids, gw)


def test_single_launch_is_used_for_small_steps(moe):
    layer = gen.make_layer(gen.config(1), 3, experts=[0])
    L = moe.MoELayer(layer, max_tokens=8)
    try:
        assert L.info().single_launch_max_tokens >= 1
    finally:
        L.close()
    L = moe.MoELayer(layer, max_tokens=8, fused=-1)
    try:
        assert L.info().single_launch_max_tokens == 0
    finally:
        L.close()


def test_tiny_all_experts_real(moe, orc):
    layer, x, _ = guarded_case(0, 7, T=8, full=True)
    gout, gids, gw = run_gpu(moe, layer, x)
    check_parity(orc, layer, x, gout, gids, gw)


SHAPES = [
    # H, E, k, I, S, Is, T
    (64, 5, 1, 64, 0, 64, 1),
    (192, 9, 3, 128, 1, 64, 3),
    (320, 33, 4, 192, 2, 128, 7),
    (128, 4, 4, 64, 1, 64, 8),        # every expert selected
    (512, 40, 8, 256, 1, 256, 5),
    (256, 17, 2, 320, 1, 192, 13),    # T > 8: grouped token path
    (384, 64, 6, 128, 1, 128, 37),
    (128, 8, 3, 64, 2, 64, 64),
    (128, 1, 1, 64, 0, 64, 4),        # a single expert
    (192, 48, 5, 128, 2, 64, 2),      # two tokens: each warp gathers its own pieces' h
    (256, 300, 6, 128, 1, 128, 2),    # more than 256 experts: the chain's router
    (128, 256, 8, 64, 1, 128, 8),     # top-8 of 256 at T = 8, shared expert wider than the routed ones
]


@pytest.mark.parametrize("fused", [0, -1], ids=["auto", "chain"])
@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_ragged_shapes(moe, orc, shape, fused):
    H, E, k, I, S, Is, T = shape
    c = dict(name="ragged", T=T, H=H, E=E, k=k, I=I, S=S, Is=Is, zipf=False, normalize=1, routed_scale=1.0)
    layer, x, _ = guarded_case(c, 1000 + H + E + T, full=True)
    gout, gids, gw = run_gpu(moe, layer, x, fused=fused)
    check_parity(orc, layer, x, gout, gids, gw)


@pytest.mark.parametrize("fused", [0, -1], ids=["auto", "chain"])
def test_no_normalisation_and_routed_scale(moe, orc, fused):
    c = gen.config(0, normalize=0, routed_scale=2.5)
    layer, x, _ = guarded_case(c, 31, T=4, full=True)
    gout, gids, gw = run_gpu(moe, layer, x, fused=fused)
    check_parity(orc, layer, x, gout, gids, gw)


def test_router_bias_zipf_small(moe, orc):
    c = gen.config(3)
    layer, x, _ = guarded_case(c, 77, T=16)
    gout, gids, gw = run_gpu(moe, layer, x)
    check_parity(orc, layer, x, gout, gids, gw)


@pytest.mark.parametrize("fused", [0, -1], ids=["auto", "chain"])
def test_large_activations_prescale(moe, orc, fused):
    """Activations far outside the f16 range (x * 2^20, so h ~ 2^40): the
    kernels' power-of-two prescale must keep the result exact up to the usual
    rounding.  The router rows are scaled by 2^-20 so the logits, hence the
    routing, are exactly those of the unscaled input."""
    layer, x, _ = guarded_case(0, 5, T=3, full=True)
    xs = (x.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** 20)
    xb = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    big = dict(layer)
    big["router_w"] = layer["router_w"] * np.float32(2.0 ** -20)
    gout, gids, gw = run_gpu(moe, big, xb, fused=fused)
    err_abs, err_rel = check_parity(orc, big, xb, gout, gids, gw)
    assert np.abs((gout.astype(np.uint32) << 16).view(np.float32)).max() > 1e9


@pytest.mark.parametrize("fused", [0, -1], ids=["auto", "chain"])
def test_zero_input(moe, orc, fused):
    layer, x, _ = guarded_case(0, 3, T=2, full=True)
    xz = np.zeros_like(x)
    gout, gids, gw = run_gpu(moe, layer, xz, fused=fused)
    oout, _, oids, _ = orc.forward(layer, xz)
    assert np.array_equal(gout, oout)


@pytest.mark.parametrize("fused", [0, -1], ids=["auto", "chain"])
def test_handle_reuse_varying_T_and_determinism(moe, orc, fused):
    layer, x, _ = guarded_case(2, 11, T=8)
    L = moe.MoELayer(layer, max_tokens=8, fused=fused)
    try:
        first = None
        for T in (8, 1, 5, 8):
            gout, gids, gw = run_gpu(moe, layer, x[:T], layer_obj=L)
            check_parity(orc, layer, x[:T], gout, gids, gw)
            if T == 8:
                if first is None:
                    first = gout
                else:
                    assert np.array_equal(first, gout), "run-to-run difference"
    finally:
        L.close()


def test_many_calls_keep_tags_in_step(moe, orc):
    """The single launch tags exchanged words with the call number: after a
    long run of calls with changing T (stale words of larger steps stay
    behind), every call still matches the oracle."""
    layer, x, _ = guarded_case(0, 17, T=8, full=True)
    L = moe.MoELayer(layer, max_tokens=8)
    try:
        xd = x_to_device(x)
        for i in range(300):
            T = (1, 8, 2, 5)[i % 4]
            out, ids, w = L.forward(xd[:T])
        torch.cuda.synchronize()
        assert moe.moe_check(L.h) == moe.MOE_OK
        for T in (8, 1):
            gout, gids, gw = run_gpu(moe, layer, x[:T], layer_obj=L)
            check_parity(orc, layer, x[:T], gout, gids, gw)
    finally:
        L.close()


@pytest.mark.parametrize("cfg,T,pinned", [(1, 1, True), (1, 1, False), (1, 2, True), (1, 8, True), (0, 12, True),
                                          (0, 12, False)])
def test_host_buffer_entry_point(moe, orc, cfg, T, pinned):
    """Host buffers: pinned output is written through its device alias (the
    single launch at T=1, 2 and 8, the chain's down kernel at T=12), pageable
    output is copied back; a pinned x is read in place by the single launch
    at T <= 2 and copied up otherwise; all equal the device-buffer call bit
    for bit."""
    layer, x, _ = guarded_case(cfg, 13, T=T)
    L = moe.MoELayer(layer, max_tokens=T)
    try:
        H, k = layer["cfg"]["H"], layer["cfg"]["k"]
        pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
        xh = pin(torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16))
        oh = pin(torch.full((T, H), 7.0, dtype=torch.bfloat16))
        ih = pin(torch.empty((T, k), dtype=torch.int32))
        wh = pin(torch.empty((T, k), dtype=torch.float32))
        moe.moe_decode_forward_host(L.h, xh, T, oh, ih, wh)
        torch.cuda.synchronize()
        dout, dids, dw = run_gpu(moe, layer, x, layer_obj=L)
        assert np.array_equal(out_to_bits(oh), dout)
        assert np.array_equal(ih.numpy(), dids) and np.array_equal(wh.numpy(), dw)
        check_parity(orc, layer, x, dout, dids, dw)
    finally:
        L.close()


def test_stage_entry_points(moe, orc):
    """moe_stage_route / _gate_up / _down called one by one equal the chained
    forward of a handle built with fused = -1 bit for bit, and match the
    oracle."""
    layer, x, _ = guarded_case(2, 17)
    L = moe.MoELayer(layer, max_tokens=8, fused=-1)
    try:
        xd = x_to_device(x)
        T, H, k = x.shape[0], layer["cfg"]["H"], layer["cfg"]["k"]
        out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        moe.moe_stage_route(L.h, xd, T, ids, w)
        moe.moe_stage_gate_up(L.h, xd, T)
        moe.moe_stage_down(L.h, T, out)
        torch.cuda.synchronize()
        fout, fids, fw = run_gpu(moe, layer, x, layer_obj=L)
        assert np.array_equal(out_to_bits(out), fout)
        assert np.array_equal(ids.cpu().numpy(), fids)
        check_parity(orc, layer, x, fout, fids, fw)
    finally:
        L.close()


def test_invalid_calls_enqueue_nothing(moe):
    layer, x, _ = guarded_case(0, 3, T=2, full=True)
    L = moe.MoELayer(layer, max_tokens=2)
    try:
        xd = x_to_device(x)
        out = torch.empty_like(xd)
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_decode_forward(L.h, xd, 3, out)
        assert ei.value.status == moe.moe.MOE_ERR_INVALID_ARG
        with pytest.raises(moe.MoEError):
            moe.moe_decode_forward(L.h, xd, 0, out)
        with pytest.raises(moe.MoEError):
            moe.moe_decode_forward(L.h, xd, 2, xd)          # out aliases x
        with pytest.raises(moe.MoEError):
            moe.moe_decode_forward(L.h, xd.view(-1)[1:], 1, out)  # 2-byte offset: misaligned
        assert moe.moe_check(L.h) == moe.MOE_OK
    finally:
        L.close()


def _wide_rows(orc, c, router, rng, T):
    """T activation rows whose magnitudes span about 2^40 within each row:
    sixteen elements ~N(0,1), the others ~N(0,1) * 2^-40 (BF16 holds both),
    each row redrawn until its routing clears the margin (at most 200 draws)."""
    from moe_cases import MARGIN
    rows = []
    for _ in range(200 * T):
        if len(rows) == T:
            break
        v = rng.standard_normal(c["H"]) * 2.0 ** -40
        big = rng.choice(c["H"], 16, replace=False)
        v[big] = rng.standard_normal(16)
        xb = gen.synth._to_bf16_bits(v.astype(np.float32))
        _, _, s, _ = orc.route({"cfg": c, **router}, xb[None, :])
        srt = np.sort(s[0])[::-1]
        if srt[c["k"] - 1] - srt[c["k"]] >= MARGIN:
            rows.append(xb)
    assert len(rows) == T, "no admissible rows"
    return np.stack(rows)


@pytest.mark.parametrize("T", [1, 8])
@pytest.mark.parametrize("fused", [0, -1], ids=["single", "chain"])
def test_activation_rows_spanning_2_pow_40(moe, orc, T, fused):
    """The exact power-of-two prescale of activation rows to f16 (row maximum
    in [2^14, 2^15)) on rows spanning ~2^40: the large elements stay exact,
    only elements far below the row maximum lose bits, and their share of
    every dot product is far inside the tolerance."""
    c = gen.config(2, T=T)
    seed = gen.BASE_SEED + 70 + T
    router = gen.make_router(c, seed)
    x = _wide_rows(orc, c, router, np.random.default_rng(seed), T)
    xv = (x.astype(np.uint32) << 16).view(np.float32)
    a = np.abs(xv[xv != 0])
    assert np.log2(a.max() / a.min()) > 38
    ids, *_ = orc.route({"cfg": c, **router}, x)
    layer = {"cfg": c, **router, **gen.make_experts(c, seed, np.unique(ids))}
    gout, gids, gw = run_gpu(moe, layer, x, fused=fused)
    check_parity(orc, layer, x, gout, gids, gw)

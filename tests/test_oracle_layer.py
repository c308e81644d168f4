"""Pins for the oracle's expert MLP and combine (no GPU).

Special cases that reduce to dense linear algebra (numpy FP64 matmuls over
weights built from a dense value matrix and packed by the test), closed-form
layers worked by hand, and invariants: batch independence, expert permutation,
power-of-two scale linearity, thread-count independence.
"""
import math

import numpy as np
import pytest
import torch

import gen

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                 -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def pack(codes):
    lo = codes[..., 0::2].astype(np.uint8)
    hi = codes[..., 1::2].astype(np.uint8)
    return (lo | (hi << 4)).astype(np.uint8)


def e4m3_vals(sf):
    return torch.from_numpy(np.ascontiguousarray(sf)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def dense(codes, sf, gs):
    """[rows, cols] codes (unpacked), [rows, cols/16] scales -> exact FP64 weights."""
    return E2M1[codes] * np.repeat(e4m3_vals(sf), 16, axis=-1) * float(gs)


def bf16_bits(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def random_expert(rng, H, I):
    c13 = rng.integers(0, 16, (2 * I, H))
    s13 = rng.integers(0x20, 0x39, (2 * I, H // 16)).astype(np.uint8)
    c2 = rng.integers(0, 16, (H, I))
    s2 = rng.integers(0x20, 0x39, (H, I // 16)).astype(np.uint8)
    return c13, s13, c2, s2


def dense_mlp(orc, x, c13, s13, gs13, c2, s2, gs2):
    I = c13.shape[0] // 2
    W13 = dense(c13, s13, 1.0)
    Wg = W13[:I] * float(gs13[0])
    Wu = W13[I:] * float(gs13[1])
    Wd = dense(c2, s2, gs2)
    g = Wg @ x
    u = Wu @ x
    h = np.array([orc.bf16_round(v) for v in (g / (1 + np.exp(-g))) * u])
    return Wd @ h


def test_single_expert_equals_dense_mlp(orc):
    rng = np.random.default_rng(21)
    H, I = 64, 48
    c13, s13, c2, s2 = random_expert(rng, H, I)
    gs13 = np.array([[0.125, 0.25]], np.float32)
    gs2 = np.array([0.5], np.float32)
    c = dict(H=H, E=1, k=1, I=I, S=0, Is=I, normalize=1, routed_scale=1.0)
    layer = {"cfg": c, "router_w": rng.standard_normal((1, H)).astype(np.float32), "router_b": None,
             "w13": pack(c13)[None], "w13_sf": s13[None], "w13_gs": gs13,
             "w2": pack(c2)[None], "w2_sf": s2[None], "w2_gs": gs2}
    xb = bf16_bits(rng.standard_normal((3, H)))
    out, pre, ids, w = orc.forward(layer, xb)
    assert np.all(ids == 0) and np.all(w == 1.0)
    for t in range(3):
        y = dense_mlp(orc, bits_to_f64(xb[t]), c13, s13, gs13[0], c2, s2, gs2[0])
        assert np.allclose(pre[t], y, rtol=1e-13, atol=1e-12)
        assert np.array_equal(out[t], np.array([orc.to_bf16_bits(v) for v in y], np.uint16))


def test_shared_expert_only(orc):
    """Routed down codes all zero -> the output is the shared MLP alone."""
    rng = np.random.default_rng(22)
    H, I, E, k = 64, 32, 4, 2
    c = dict(H=H, E=E, k=k, I=I, S=1, Is=I, normalize=1, routed_scale=1.0)
    rc = [random_expert(rng, H, I) for _ in range(E)]
    sc13, ss13, sc2, ss2 = random_expert(rng, H, I)
    layer = {"cfg": c, "router_w": rng.standard_normal((E, H)).astype(np.float32), "router_b": None,
             "w13": np.stack([pack(r[0]) for r in rc]), "w13_sf": np.stack([r[1] for r in rc]),
             "w13_gs": np.full((E, 2), 0.125, np.float32),
             "w2": np.zeros((E, H, I // 2), np.uint8), "w2_sf": np.stack([r[3] for r in rc]),
             "w2_gs": np.full((E,), 0.25, np.float32),
             "sw13": pack(sc13)[None], "sw13_sf": ss13[None], "sw13_gs": np.array([[0.125, 0.25]], np.float32),
             "sw2": pack(sc2)[None], "sw2_sf": ss2[None], "sw2_gs": np.array([0.5], np.float32)}
    xb = bf16_bits(rng.standard_normal((2, H)))
    out, pre, ids, w = orc.forward(layer, xb)
    for t in range(2):
        y = dense_mlp(orc, bits_to_f64(xb[t]), sc13, ss13, [0.125, 0.25], sc2, ss2, 0.5)
        assert np.allclose(pre[t], y, rtol=1e-13, atol=1e-12)


def test_closed_form_tiny_layer(orc):
    """H=I=16, two routed experts (top-1) and no shared expert.
    Expert 1 is selected (router logit 2 vs -2), weight 1 after normalising.
    Gate codes 0x4 (2.0) with gs 1/16: g = sum_k x_k * 2/16 = 2 for x = 1.
    Up codes 0x6 (4.0) with gs 1/16: u = 4.
    h = bf16(silu(2) * 4) = bf16(8 / (1 + e^-2)) = bf16(7.046377) = 7.03125.
    Down codes 0x2 (1.0), gs 1: y_m = 16 * 7.03125 = 112.5.
    Swapping gate and up would give bf16(silu(4) * 2) = 7.84375 instead."""
    H = I = 16
    c = dict(H=H, E=2, k=1, I=I, S=0, Is=I, normalize=1, routed_scale=1.0)
    rw = np.zeros((2, H), np.float32)
    rw[0, 0], rw[1, 0] = -2.0, 2.0
    codes13 = np.zeros((2, 2 * I, H), np.int64)
    codes13[1, :I] = 0x4
    codes13[1, I:] = 0x6
    codes13[0] = 0x7           # expert 0 (not selected) would give a very different output
    codes2 = np.full((2, H, I), 0x2)
    layer = {"cfg": c, "router_w": rw, "router_b": None,
             "w13": pack(codes13), "w13_sf": np.full((2, 2 * I, 1), 0x38, np.uint8),
             "w13_gs": np.full((2, 2), 1 / 16, np.float32),
             "w2": pack(codes2), "w2_sf": np.full((2, H, 1), 0x38, np.uint8),
             "w2_gs": np.ones(2, np.float32)}
    x = np.full((1, H), 0x3F80, np.uint16)      # all ones
    out, pre, ids, w = orc.forward(layer, x)
    h = 8 / (1 + math.exp(-2))
    assert abs(h - 7.0463766) < 1e-6
    assert ids.tolist() == [[1]] and w.tolist() == [[1.0]]
    assert np.all(pre == 112.5)
    assert np.all(bits_to_f64(out) == 112.5)


def test_closed_form_two_experts_and_shared(orc):
    """Top-2 of 3 with a shared expert; every expert maps x = 1 to a constant
    output, so out = w_a * y_a + w_b * y_b + y_s with closed-form weights."""
    H = I = 16
    c = dict(H=H, E=3, k=2, I=I, S=1, Is=I, normalize=1, routed_scale=1.0)
    rw = np.zeros((3, H), np.float32)
    rw[:, 0] = [1.0, -1.0, 0.5]                        # selects experts 0 then 2
    codes13 = np.zeros((3, 2 * I, H), np.int64)
    codes13[:, :I] = 0x4                               # gate 2.0 * 1/16 * 16 = 2
    codes13[:, I:] = 0x6                               # up 4
    codes2 = np.stack([np.full((H, I), 0x2), np.full((H, I), 0x4), np.full((H, I), 0xC)])  # 1, 2, -2
    layer = {"cfg": c, "router_w": rw, "router_b": None,
             "w13": pack(codes13), "w13_sf": np.full((3, 2 * I, 1), 0x38, np.uint8),
             "w13_gs": np.full((3, 2), 1 / 16, np.float32),
             "w2": pack(codes2), "w2_sf": np.full((3, H, 1), 0x38, np.uint8),
             "w2_gs": np.ones(3, np.float32),
             "sw13": pack(np.concatenate([np.full((I, H), 0x4), np.full((I, H), 0x6)])[None]),
             "sw13_sf": np.full((1, 2 * I, 1), 0x38, np.uint8), "sw13_gs": np.full((1, 2), 1 / 16, np.float32),
             "sw2": pack(np.full((1, H, I), 0x3)), "sw2_sf": np.full((1, H, 1), 0x38, np.uint8),
             "sw2_gs": np.ones(1, np.float32)}           # shared down code 0x3 = 1.5
    x = np.full((1, H), 0x3F80, np.uint16)
    out, pre, ids, w = orc.forward(layer, x)
    s0, s2 = 1 / (1 + math.exp(-1.0)), 1 / (1 + math.exp(-0.5))
    w0, w2 = s0 / (s0 + s2), s2 / (s0 + s2)
    hsum = 16 * 7.03125
    expect = w0 * hsum * 1.0 + w2 * hsum * (-2.0) + hsum * 1.5
    assert ids.tolist() == [[0, 2]]
    assert np.allclose(w, [[w0, w2]], rtol=0, atol=1e-15)
    assert np.allclose(pre, expect, rtol=1e-14, atol=0)


@pytest.fixture(scope="module")
def tiny_case(orc):
    from moe_cases import guarded_case
    return guarded_case(0, 99, T=5, full=True)


def test_batch_independence(orc, tiny_case):
    layer, x, _ = tiny_case
    out, pre, ids, w = orc.forward(layer, x)
    for t in range(x.shape[0]):
        o1, p1, i1, w1 = orc.forward(layer, x[t:t + 1])
        assert np.array_equal(o1[0], out[t]) and np.array_equal(p1[0], pre[t])
        assert np.array_equal(i1[0], ids[t]) and np.array_equal(w1[0], w[t])


def test_thread_count_independence(orc, tiny_case):
    layer, x, _ = tiny_case
    a = orc.forward(layer, x, nthreads=1)
    b = orc.forward(layer, x, nthreads=4)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_expert_permutation_invariance(orc, tiny_case):
    layer, x, _ = tiny_case
    out, pre, ids, w = orc.forward(layer, x)
    E = layer["cfg"]["E"]
    perm = np.random.default_rng(3).permutation(E)
    lp = dict(layer)
    for n in ("router_w", "w13", "w13_sf", "w13_gs", "w2", "w2_sf", "w2_gs"):
        lp[n] = layer[n][perm]
    o2, p2, i2, w2 = orc.forward(lp, x)
    assert np.array_equal(perm[i2], ids)
    assert np.array_equal(p2, pre) and np.array_equal(o2, out)


def test_down_scale_linearity(orc, tiny_case):
    layer, x, _ = tiny_case
    out, pre, *_ = orc.forward(layer, x)
    l2 = dict(layer)
    l2["w2_gs"] = layer["w2_gs"] * np.float32(2)
    l2["sw2_gs"] = layer["sw2_gs"] * np.float32(2)
    _, pre2, *_ = orc.forward(l2, x)
    assert np.array_equal(pre2, 2 * pre)


def test_sign_flip_of_up_codes(orc, tiny_case):
    """Flipping every up-projection code's sign bit negates every h exactly
    (BF16 rounding is symmetric), hence negates the output."""
    layer, x, _ = tiny_case
    out, pre, *_ = orc.forward(layer, x)
    c = layer["cfg"]
    I, Is = c["I"], c["Is"]
    l2 = dict(layer)
    w13 = layer["w13"].copy()
    w13[:, I:] ^= 0x88
    sw13 = layer["sw13"].copy()
    sw13[:, Is:] ^= 0x88
    l2["w13"], l2["sw13"] = w13, sw13
    _, pre2, *_ = orc.forward(l2, x)
    assert np.array_equal(pre2, -pre)


def test_generator_is_deterministic_and_subsettable():
    c = gen.config(0)
    a = gen.make_layer(c, 4)
    b = gen.make_layer(c, 4, experts=[3, 7])
    for n in ("w13", "w13_sf", "w2", "w2_sf"):
        assert np.array_equal(a[n][[3, 7]], b[n][[3, 7]])
        assert np.all(b[n][0] == (0x7F if n.endswith("sf") else 0xFF))
    assert np.array_equal(gen.make_x(c, 4, T=3), gen.make_x(c, 4, T=3))
    sf = a["w13_sf"]
    vals = e4m3_vals(sf)
    assert vals.min() >= 0.125 and vals.max() <= 1.0
    assert np.all(a["w13_gs"] == np.float32(1 / 16))

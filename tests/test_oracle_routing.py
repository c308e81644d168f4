"""Pins for the oracle's router (no GPU).

Sigmoid top-k with weights normalised to sum to 1 (Flint page, "Flint model
architecture", MoE bullet), FP32 router decision (Inkling 2 Small page,
"Accuracy evaluation"): sigmoid is strictly increasing, so the ranking is that
of the FP32 logits.  Pinned by brute force over all k-subsets, by closed
forms for the scores and weights, by the tie rule and by a permutation
invariant.
"""
import itertools
import math

import numpy as np

import gen


def _router_layer(E, H, k, w, b=None, normalize=1, routed_scale=1.0):
    c = dict(H=H, E=E, k=k, I=64, S=0, Is=64, normalize=normalize, routed_scale=routed_scale)
    return {"cfg": c, "router_w": w.astype(np.float32), "router_b": b}


def _bf16(a):
    import torch
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bruteforce_topk_subsets(orc):
    rng = np.random.default_rng(11)
    E, H, k = 9, 32, 3
    for trial in range(20):
        w = rng.standard_normal((E, H)).astype(np.float32)
        x = _bf16(rng.standard_normal((1, H)))
        L = _router_layer(E, H, k, w)
        ids, wt, s, z = orc.route(L, x)
        best = max(itertools.combinations(range(E), k), key=lambda sub: sum(s[0][list(sub)]))
        assert sorted(ids[0].tolist()) == sorted(best)
        # selection order is descending score
        assert all(s[0][ids[0][j]] >= s[0][ids[0][j + 1]] for j in range(k - 1))


def test_scores_weights_closed_form(orc):
    # x = one-hot 1.0 at h=0, router column 0 holds the logits -> z_e known exactly.
    E, H, k = 6, 16, 3
    zs = np.array([0.5, -1.0, 2.0, 0.25, 1.5, -0.75], np.float32)
    w = np.zeros((E, H), np.float32)
    w[:, 0] = zs
    x = np.zeros((1, H), np.uint16)
    x[0, 0] = 0x3F80                                   # BF16 1.0
    L = _router_layer(E, H, k, w)
    ids, wt, s, z = orc.route(L, x)
    sig = [1 / (1 + math.exp(-float(v))) for v in zs]
    assert np.allclose(s[0], sig, rtol=0, atol=1e-15)
    assert ids[0].tolist() == [2, 4, 0]
    tot = sig[2] + sig[4] + sig[0]
    assert np.allclose(wt[0], [sig[2] / tot, sig[4] / tot, sig[0] / tot], rtol=0, atol=1e-15)
    # bias adds to the logit
    b = np.array([0, 0, -5, 0, 0, 3], np.float32)
    ids, wt, s, z = orc.route(_router_layer(E, H, k, w, b), x)
    assert np.allclose(z[0], zs.astype(np.float64) + b, rtol=0, atol=0)
    assert ids[0].tolist() == [5, 4, 0]
    # no normalisation: weights are the scores times the routed scale
    ids, wt, s, z = orc.route(_router_layer(E, H, k, w, normalize=0, routed_scale=2.5), x)
    assert np.allclose(wt[0], [2.5 * sig[2], 2.5 * sig[4], 2.5 * sig[0]], rtol=0, atol=1e-15)


def test_ties_lowest_index_first(orc):
    E, H, k = 8, 16, 2
    w = np.zeros((E, H), np.float32)
    w[:, 0] = [0.1, 0.3, 0.7, 0.2, 0.7, 0.7, 0.0, -1]   # experts 2, 4, 5 tie at the top
    x = np.zeros((1, H), np.uint16)
    x[0, 0] = 0x3F80
    ids, *_ = orc.route(_router_layer(E, H, k, w), x)
    assert ids[0].tolist() == [2, 4]


def test_fp32_decision_precision(orc):
    # The decision is taken on FP32 logits.  (1) Logits 20.0 and 19.5 whose
    # sigmoids round to the same FP32 score (1.0) are distinct FP32 logits:
    # the larger logit wins, as it does for the exact scores.
    E, H, k = 3, 16, 1
    z_hi, z_lo = 20.0, 19.5          # sigmoid -> 1 - 2e-9 vs 1 - 3.4e-9: both fl32 = 1.0
    w = np.zeros((E, H), np.float32)
    w[:, 0] = [z_lo, z_hi, -3.0]
    x = np.zeros((1, H), np.uint16)
    x[0, 0] = 0x3F80
    ids, wt, s, _ = orc.route(_router_layer(E, H, k, w), x)
    assert s[0][1] > s[0][0]
    assert np.float32(s[0][1]) == np.float32(s[0][0])
    assert ids[0].tolist() == [1]
    # (2) FP64 logits 1 + 2^-30 (expert 1) and 1 (expert 0) round to the same
    # FP32 logit: a tie, so the lower index wins although expert 1's exact
    # score is larger.
    E, k = 2, 1
    w = np.zeros((E, H), np.float32)
    w[0, 0] = 1.0
    w[1, 0] = 1.0
    w[1, 1] = 1.0
    x = np.zeros((1, H), np.uint16)
    x[0, 0] = 0x3F80                 # 1.0
    x[0, 1] = 0x3080                 # 2^-30
    ids, wt, s, z = orc.route(_router_layer(E, H, k, w), x)
    assert z[0][1] == 1.0 + 2.0 ** -30 and z[0][0] == 1.0
    assert s[0][1] > s[0][0]
    assert np.float32(z[0][1]) == np.float32(z[0][0])
    assert ids[0].tolist() == [0]


def test_weights_sum_to_one_and_permutation(orc):
    c = gen.config(1)
    R = gen.make_router(c, 5)
    L = {"cfg": c, **R}
    x = gen.make_x(c, 5, T=4)
    ids, wt, s, z = orc.route(L, x)
    assert np.allclose(wt.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    perm = np.random.default_rng(1).permutation(c["E"])        # new index p -> old perm[p]
    Lp = {"cfg": c, "router_w": R["router_w"][perm], "router_b": None}
    ids_p, wt_p, s_p, _ = orc.route(Lp, x)
    inv = np.argsort(perm)
    assert np.array_equal(perm[ids_p], ids)
    assert np.array_equal(wt_p, wt)
    assert np.array_equal(s_p[:, inv], s)


def test_zipf_workload_popularity(orc):
    """The skewed workload's router bias gives selection counts with a log-log
    slope near -1.1 over the 64 most popular ranks."""
    c = gen.config(3)
    seed = 20261205
    R = gen.make_router(c, seed)
    L = {"cfg": c, **R}
    counts = np.zeros(c["E"])
    nb = 6
    for b in range(nb):
        ids, *_ = orc.route(L, gen.make_x(c, 1000 + b))
        np.add.at(counts, ids.ravel(), 1)
    perm = np.random.Generator(np.random.SFC64([seed, 3, 0])).permutation(c["E"])
    byrank = np.zeros(c["E"])
    byrank[perm] = counts
    r = np.arange(1, 65)
    y = byrank[:64]
    m = y > 0
    slope = np.polyfit(np.log(r[m]), np.log(y[m]), 1)[0]
    assert -1.3 < slope < -0.9, slope


# ---- softmax routing (Mistral Large 4 page, "Specialized decode": softmax
# top-4 router), score_func = "softmax" ----

def _softmax_layer(E, H, k, w, b=None, normalize=1, routed_scale=1.0):
    L = _router_layer(E, H, k, w, b, normalize, routed_scale)
    L["cfg"]["score_func"] = "softmax"
    return L


def _onehot_x(H):
    x = np.zeros((1, H), np.uint16)
    x[0, 0] = 0x3F80                                   # BF16 1.0
    return x


def test_softmax_two_experts_is_the_logistic_of_the_difference(orc):
    # softmax over two logits a, b gives 1 / (1 + e^(b - a)) and its complement
    H = 16
    for a, b in [(0.5, -1.25), (3.0, 2.75), (-4.0, 1.0)]:
        w = np.zeros((2, H), np.float32)
        w[:, 0] = [a, b]
        ids, wt, s, z = orc.route(_softmax_layer(2, H, 2, w, normalize=0), _onehot_x(H))
        p0 = 1.0 / (1.0 + math.exp(b - a))
        assert abs(s[0][0] - p0) <= 1e-15 and abs(s[0][1] - (1.0 - p0)) <= 1e-15
        hi = 0 if a > b else 1
        assert ids[0].tolist() == [hi, 1 - hi]
        assert abs(wt[0][0] - max(p0, 1 - p0)) <= 1e-15


def test_softmax_normalised_top2_is_the_logistic_of_the_chosen_gap(orc):
    # normalised over the chosen two, the weights only see their logit gap
    E, H, k = 6, 16, 2
    zs = np.array([0.5, -1.0, 2.0, 0.25, 1.5, -0.75], np.float32)
    w = np.zeros((E, H), np.float32)
    w[:, 0] = zs
    ids, wt, s, z = orc.route(_softmax_layer(E, H, k, w), _onehot_x(H))
    assert ids[0].tolist() == [2, 4]
    p = 1.0 / (1.0 + math.exp(float(zs[4]) - float(zs[2])))
    assert abs(wt[0][0] - p) <= 1e-15 and abs(wt[0][1] - (1.0 - p)) <= 1e-15
    # unnormalised, all experts chosen: the scores are a distribution
    ids, wt, s, z = orc.route(_softmax_layer(E, H, E, w, normalize=0, routed_scale=2.0), _onehot_x(H))
    assert abs(wt[0].sum() - 2.0) <= 1e-14
    assert np.all(np.diff(wt[0]) <= 0)


def test_softmax_is_shift_invariant_and_sigmoid_is_not(orc):
    rng = np.random.default_rng(5)
    E, H, k = 12, 64, 3
    w = (rng.standard_normal((E, H)) / 8).astype(np.float32)
    x = _bf16(rng.standard_normal((2, H)))
    shift = np.full(E, 1.5, np.float32)                  # the same bias on every logit
    for norm in (0, 1):
        a = orc.route(_softmax_layer(E, H, k, w, normalize=norm), x)
        b = orc.route(_softmax_layer(E, H, k, w, shift, normalize=norm), x)
        assert np.array_equal(a[0], b[0])
        assert np.allclose(a[1], b[1], rtol=1e-12, atol=0)
    a = orc.route(_router_layer(E, H, k, w, normalize=0), x)
    b = orc.route(_router_layer(E, H, k, w, shift, normalize=0), x)
    assert np.array_equal(a[0], b[0]) and not np.allclose(a[1], b[1], rtol=1e-3, atol=0)


def test_softmax_selects_what_sigmoid_selects(orc):
    rng = np.random.default_rng(9)
    E, H, k = 40, 96, 5
    for trial in range(10):
        w = rng.standard_normal((E, H)).astype(np.float32)
        x = _bf16(rng.standard_normal((3, H)))
        ids_sig = orc.route(_router_layer(E, H, k, w), x)[0]
        ids_sm, wt, s, z = orc.route(_softmax_layer(E, H, k, w), x)
        assert np.array_equal(ids_sig, ids_sm)
        assert np.allclose(s.sum(axis=1), 1.0, rtol=0, atol=1e-12)
        assert np.allclose(wt.sum(axis=1), 1.0, rtol=0, atol=1e-12)

"""Synthetic layers of the pages' shapes, seeded and reproducible.

Workloads (sizes the pages give, plus choices where they give none):

  0 tiny     T=1,  H=256,  E=16,  top-2, I=128,  1 shared (I=128)
  1 flint    T=1,  H=2048, E=256, top-6, I=768,  1 shared (I=768)   Flint page,
             "Flint model architecture": hidden 2048, 256 experts, sigmoid
             top-6 plus one shared expert; I=768 is our choice.
  2 flint8   as flint with T=8 (the low-latency path's limit, Flint page,
             "Optimisation strategy").
  3 zipf64   as flint with T=64 and a router bias that skews expert popularity
             to Zipf(1.1).
  4 ml4      T=8,  H=6144, E=128, top-4, I=2048, 1 shared (I=2048)  Mistral
             Large 4 page, "Highlights"/"Model architecture": hidden 6144, 128
             experts, top-4, one shared expert; I=2048 is our choice.

Recipe (every config):
  x          ~ N(0,1) per element, rounded to BF16 (round to nearest even)
  router W   ~ N(0, 1/H), FP32
  codes      uniform over the 16 E2M1 codes (uniform bytes: two nibbles)
  scales     a real uniform on [2^-3, 2^0], rounded to E4M3 (fn)
  gs         fl32(1/sqrt(fan_in)): H for gate/up, I for down
  streams    one SFC64 stream per (seed, tensor, expert), so any subset of the
             experts can be drawn on its own and gives the same bytes.

Only inputs are made here.  Experts that a test does not need can be filled
with a "poison" pattern (NaN scales) so that a kernel reading them shows up.
"""
from __future__ import annotations

import math

import numpy as np

CONFIGS = {
    0: dict(name="tiny", T=1, H=256, E=16, k=2, I=128, S=1, Is=128, zipf=False),
    1: dict(name="flint", T=1, H=2048, E=256, k=6, I=768, S=1, Is=768, zipf=False),
    2: dict(name="flint8", T=8, H=2048, E=256, k=6, I=768, S=1, Is=768, zipf=False),
    3: dict(name="zipf64", T=64, H=2048, E=256, k=6, I=768, S=1, Is=768, zipf=True),
    4: dict(name="ml4", T=8, H=6144, E=128, k=4, I=2048, S=1, Is=2048, zipf=False),
}

BASE_SEED = 20261202

# Stream tags.
_T_ROUTER, _T_BIAS, _T_PERM, _T_W13, _T_W13SF, _T_W2, _T_W2SF = 1, 2, 3, 4, 5, 6, 7
_T_SW13, _T_SW13SF, _T_SW2, _T_SW2SF, _T_X = 8, 9, 10, 11, 12

# Zipf exponent of the skewed workload, and the logit scale alpha of the bias
# b_e = -alpha * s * ln(rank(e)).  alpha was set so that, for 64-token batches
# of this layer, the realised selection counts follow a log-log slope of about
# -1.1 over ranks 1..64 (checked by a test that routes with the oracle).
ZIPF_S = 1.1
ZIPF_ALPHA = 0.58

POISON_SCALE = 0x7F   # E4M3 NaN
POISON_CODE = 0xFF


def config(idx_or_name, **over) -> dict:
    if isinstance(idx_or_name, str):
        idx = next(i for i, c in CONFIGS.items() if c["name"] == idx_or_name)
    else:
        idx = int(idx_or_name)
    c = dict(CONFIGS[idx])
    c["index"] = idx
    c.setdefault("normalize", 1)
    c.setdefault("routed_scale", 1.0)
    c.update(over)
    return c


def _rng(seed: int, tag: int, idx: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.SFC64([int(seed), int(tag), int(idx)]))


def _bytes(rng: np.random.Generator, n: int) -> np.ndarray:
    return np.frombuffer(rng.bytes(n), dtype=np.uint8).copy()


_SCALE_TABLE = None


def _scale_table() -> np.ndarray:
    """u16 -> E4M3 code of the real 2^-3 + (1 - 2^-3) * (u + 0.5) / 65536,
    rounded to nearest even by torch's float8_e4m3fn cast (a library routine)."""
    global _SCALE_TABLE
    if _SCALE_TABLE is None:
        import torch
        u = np.arange(65536, dtype=np.float64)
        reals = 0.125 + 0.875 * (u + 0.5) / 65536.0
        t = torch.from_numpy(reals.astype(np.float32)).to(torch.float8_e4m3fn)
        _SCALE_TABLE = t.view(torch.uint8).numpy().copy()
    return _SCALE_TABLE


def _scales(rng: np.random.Generator, n: int) -> np.ndarray:
    u = np.frombuffer(rng.bytes(2 * n), dtype=np.uint16)
    return _scale_table()[u]


def _to_bf16_bits(a: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def canonical_shapes(c: dict) -> dict:
    E, H, I, S, Is = c["E"], c["H"], c["I"], c["S"], c["Is"]
    return {
        "router_w": (E, H), "router_b": (E,),
        "w13": (E, 2 * I, H // 2), "w13_sf": (E, 2 * I, H // 16), "w13_gs": (E, 2),
        "w2": (E, H, I // 2), "w2_sf": (E, H, I // 16), "w2_gs": (E,),
        "sw13": (S, 2 * Is, H // 2), "sw13_sf": (S, 2 * Is, H // 16), "sw13_gs": (S, 2),
        "sw2": (S, H, Is // 2), "sw2_sf": (S, H, Is // 16), "sw2_gs": (S,),
    }


def make_router(c: dict, seed: int) -> dict:
    """Router weight [E,H] FP32 ~ N(0,1/H) and, for the Zipf workload, a bias."""
    E, H = c["E"], c["H"]
    w = _rng(seed, _T_ROUTER).standard_normal((E, H), dtype=np.float32)
    w *= np.float32(1.0 / math.sqrt(H))
    b = None
    if c.get("zipf"):
        perm = _rng(seed, _T_PERM).permutation(E)       # perm[e] = rank-1 of expert e
        ranks = perm.astype(np.float64) + 1.0
        b = (-ZIPF_ALPHA * ZIPF_S * np.log(ranks)).astype(np.float32)
    return {"router_w": w, "router_b": b}


def _one_expert(seed, tags, rows13, rows2, H, I):
    t13, t13sf, t2, t2sf, idx = tags
    w13 = _bytes(_rng(seed, t13, idx), rows13 * (H // 2)).reshape(rows13, H // 2)
    w13sf = _scales(_rng(seed, t13sf, idx), rows13 * (H // 16)).reshape(rows13, H // 16)
    w2 = _bytes(_rng(seed, t2, idx), rows2 * (I // 2)).reshape(rows2, I // 2)
    w2sf = _scales(_rng(seed, t2sf, idx), rows2 * (I // 16)).reshape(rows2, I // 16)
    return w13, w13sf, w2, w2sf


def make_experts(c: dict, seed: int, experts=None, fill: str = "poison") -> dict:
    """Routed + shared expert tensors.  `experts` (iterable of ids) limits which
    routed experts are drawn; the others get `fill` ("poison": NaN scales and
    0xFF codes; "zero": all-zero bytes)."""
    E, H, I, S, Is = c["E"], c["H"], c["I"], c["S"], c["Is"]
    sh = canonical_shapes(c)
    want = range(E) if experts is None else sorted(set(int(e) for e in experts))
    if fill == "poison":
        w13 = np.full(sh["w13"], POISON_CODE, np.uint8)
        w13sf = np.full(sh["w13_sf"], POISON_SCALE, np.uint8)
        w2 = np.full(sh["w2"], POISON_CODE, np.uint8)
        w2sf = np.full(sh["w2_sf"], POISON_SCALE, np.uint8)
    else:
        w13 = np.zeros(sh["w13"], np.uint8)
        w13sf = np.zeros(sh["w13_sf"], np.uint8)
        w2 = np.zeros(sh["w2"], np.uint8)
        w2sf = np.zeros(sh["w2_sf"], np.uint8)
    for e in want:
        a, b, d, f = _one_expert(seed, (_T_W13, _T_W13SF, _T_W2, _T_W2SF, e), 2 * I, H, H, I)
        w13[e], w13sf[e], w2[e], w2sf[e] = a, b, d, f
    gs13 = np.full((E, 2), np.float32(1.0 / math.sqrt(H)), np.float32)
    gs2 = np.full((E,), np.float32(1.0 / math.sqrt(I)), np.float32)
    out = {"w13": w13, "w13_sf": w13sf, "w13_gs": gs13, "w2": w2, "w2_sf": w2sf, "w2_gs": gs2}
    sw13 = np.empty(sh["sw13"], np.uint8)
    sw13sf = np.empty(sh["sw13_sf"], np.uint8)
    sw2 = np.empty(sh["sw2"], np.uint8)
    sw2sf = np.empty(sh["sw2_sf"], np.uint8)
    for s in range(S):
        a, b, d, f = _one_expert(seed, (_T_SW13, _T_SW13SF, _T_SW2, _T_SW2SF, s), 2 * Is, H, H, Is)
        sw13[s], sw13sf[s], sw2[s], sw2sf[s] = a, b, d, f
    out.update({
        "sw13": sw13, "sw13_sf": sw13sf,
        "sw13_gs": np.full((S, 2), np.float32(1.0 / math.sqrt(H)), np.float32),
        "sw2": sw2, "sw2_sf": sw2sf,
        "sw2_gs": np.full((S,), np.float32(1.0 / math.sqrt(Is)), np.float32),
    })
    return out


def make_layer(c: dict, seed: int, experts=None, fill: str = "poison") -> dict:
    layer = {"cfg": dict(c)}
    layer.update(make_router(c, seed))
    layer.update(make_experts(c, seed, experts, fill))
    return layer


def make_x_token(c: dict, seed: int, t: int, redraw: int = 0) -> np.ndarray:
    """One token's activation row [H] as BF16 bits, from stream (seed, x, t, redraw)."""
    rng = np.random.Generator(np.random.SFC64([int(seed), _T_X, int(t), int(redraw)]))
    return _to_bf16_bits(rng.standard_normal(c["H"], dtype=np.float32))


def make_x(c: dict, seed: int, T: int | None = None, redraws=None) -> np.ndarray:
    """[T,H] BF16 bits; redraws[t] selects the t-th token's redraw stream."""
    T = c["T"] if T is None else T
    rows = [make_x_token(c, seed, t, 0 if redraws is None else int(redraws[t])) for t in range(T)]
    return np.stack(rows) if rows else np.zeros((0, c["H"]), np.uint16)


def selected_bytes(c: dict, n_unique_routed: int) -> int:
    """Bytes a decode step must read: router (+bias), the selected routed
    experts and the shared experts (codes + block scales + tensor scales), the
    activations in and the output out."""
    E, H, I, S, Is, T = c["E"], c["H"], c["I"], c["S"], c["Is"], c["T"]
    per_routed = 3 * I * H // 2 + 3 * I * H // 16 + 12
    per_shared = 3 * Is * H // 2 + 3 * Is * H // 16 + 12
    router = E * H * 4 + (E * 4 if c.get("zipf") else 0)
    return router + n_unique_routed * per_routed + S * per_shared + T * H * 2 * 2


def make_layer_torch(c: dict, seed: int, device="cuda") -> dict:
    """The same recipe drawn with torch's generator on `device` (fast, for the
    many distinct layer replicas a timing run needs; these replicas are never
    compared with the oracle).  Returns canonical torch tensors."""
    import torch
    E, H, I, S, Is = c["E"], c["H"], c["I"], c["S"], c["Is"]
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))

    def codes(*shape):
        return torch.randint(0, 256, shape, dtype=torch.uint8, device=device, generator=g)

    def scales(*shape):
        u = torch.rand(shape, dtype=torch.float32, device=device, generator=g)
        return (0.125 + 0.875 * u).to(torch.float8_e4m3fn).view(torch.uint8)

    f32 = dict(dtype=torch.float32, device=device)
    layer = {"cfg": dict(c)}
    layer["router_w"] = torch.randn((E, H), generator=g, **f32) * (1.0 / math.sqrt(H))
    layer["router_b"] = None
    if c.get("zipf"):
        perm = torch.randperm(E, generator=g, device=device).to(torch.float64) + 1.0
        layer["router_b"] = (-ZIPF_ALPHA * ZIPF_S * torch.log(perm)).to(torch.float32)
    layer.update({
        "w13": codes(E, 2 * I, H // 2), "w13_sf": scales(E, 2 * I, H // 16),
        "w13_gs": torch.full((E, 2), 1.0 / math.sqrt(H), **f32),
        "w2": codes(E, H, I // 2), "w2_sf": scales(E, H, I // 16),
        "w2_gs": torch.full((E,), 1.0 / math.sqrt(I), **f32),
        "sw13": codes(S, 2 * Is, H // 2), "sw13_sf": scales(S, 2 * Is, H // 16),
        "sw13_gs": torch.full((S, 2), 1.0 / math.sqrt(H), **f32),
        "sw2": codes(S, H, Is // 2), "sw2_sf": scales(S, H, Is // 16),
        "sw2_gs": torch.full((S,), 1.0 / math.sqrt(Is), **f32),
    })
    return layer


def make_x_torch(c: dict, seed: int, T: int | None = None, device="cuda"):
    import torch
    T = c["T"] if T is None else T
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) + 7919)
    return torch.randn((T, c["H"]), generator=g, dtype=torch.float32, device=device).to(torch.bfloat16)

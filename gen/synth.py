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
  5 ml4fp8s  as ml4 with the shared expert in FP8 (E4M3) with one FP32 scale
             per 128 x 128 block (the page's NVFP4 checkpoint keeps its shared
             experts in block-scaled FP8; the block size is a reading).
  6 inkling  T=8, H=4096, E=384, top-8, I=2560, no shared expert: "Inkling 2
             Small on vLLM: Day-0 Support", "TL;DR" and the architecture table
             (48 MoE layers, 384 routed experts, top-8, no shared expert,
             594B parameters, 17B active); H and I are our choice, sized so
             that 48 layers of 384 experts hold ~580B parameters and the
             top-8 ~12B.  NVFP4 experts (layers 0-39 of the model).
  7 inkling_mx8  as inkling with MXFP8 experts (layers 40-47).
  8 flint_mx4    as flint with MXFP4 routed and shared experts (the Mistral
             Large 4 page's MXFP4 expert format on the Flint shape).

Recipe (every config):
  x          ~ N(0,1) per element, rounded to BF16 (round to nearest even)
  router W   ~ N(0, 1/H), FP32
  codes      uniform over the 16 E2M1 codes (uniform bytes: two nibbles)
  scales     a real uniform on [2^-3, 2^0], rounded to E4M3 (fn)
  gs         fl32(1/sqrt(fan_in)): H for gate/up, I for down
Other expert formats (same streams; no tensor scale):
  MXFP4      codes as above; E8M0 scale 2^j, j uniform over the four
             integers floor(log2(1/sqrt(fan_in))) - 3 .. floor(log2(1/sqrt(fan_in)))
  MXFP8      codes uniform over the 254 finite E4M3 codes; E8M0 scale 2^j, j
             uniform over floor(log2(1/(256 sqrt(fan_in)))) - 1 .. + 0
  FP8 block  codes as MXFP8; one FP32 scale per 128 x 128 block, a real
             uniform on [0.5, 1] / (256 sqrt(fan_in)) rounded to FP32
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
    5: dict(name="ml4fp8s", T=8, H=6144, E=128, k=4, I=2048, S=1, Is=2048, zipf=False, sfmt="fp8_block"),
    6: dict(name="inkling", T=8, H=4096, E=384, k=8, I=2560, S=0, Is=2560, zipf=False),
    7: dict(name="inkling_mx8", T=8, H=4096, E=384, k=8, I=2560, S=0, Is=2560, zipf=False, efmt="mxfp8"),
    8: dict(name="flint_mx4", T=1, H=2048, E=256, k=6, I=768, S=1, Is=768, zipf=False, efmt="mxfp4",
            sfmt="mxfp4"),
    # W4A4: activations quantised with Four-Over-Six NVFP4 before each GEMM
    9: dict(name="inkling_w4a4", T=8, H=4096, E=384, k=8, I=2560, S=0, Is=2560, zipf=False, w4a4=1),
    10: dict(name="zipf64_w4a4", T=64, H=2048, E=256, k=6, I=768, S=1, Is=768, zipf=True, w4a4=1),
}

FORMATS = ("nvfp4", "mxfp4", "fp8_block", "mxfp8")

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
    c.setdefault("efmt", "nvfp4")
    c.setdefault("sfmt", "nvfp4")
    c.setdefault("w4a4", 0)
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


def mat_shapes(fmt: str, rows: int, cols: int):
    """(codes shape, scales shape, scale dtype) of one [rows, cols] matrix."""
    if fmt == "nvfp4":
        return (rows, cols // 2), (rows, cols // 16), np.uint8
    if fmt == "mxfp4":
        return (rows, cols // 2), (rows, cols // 32), np.uint8
    if fmt == "mxfp8":
        return (rows, cols), (rows, cols // 32), np.uint8
    if fmt == "fp8_block":
        return (rows, cols), ((rows + 127) // 128, (cols + 127) // 128), np.float32
    raise ValueError(f"unknown expert format {fmt!r}")


def canonical_shapes(c: dict) -> dict:
    E, H, I, S, Is = c["E"], c["H"], c["I"], c["S"], c["Is"]
    ef, sf = c.get("efmt", "nvfp4"), c.get("sfmt", "nvfp4")
    c13, s13, _ = mat_shapes(ef, 2 * I, H)
    c2, s2, _ = mat_shapes(ef, H, I)
    sc13, ss13, _ = mat_shapes(sf, 2 * Is, H)
    sc2, ss2, _ = mat_shapes(sf, H, Is)
    return {
        "router_w": (E, H), "router_b": (E,),
        "w13": (E, *c13), "w13_sf": (E, *s13), "w13_gs": (E, 2),
        "w2": (E, *c2), "w2_sf": (E, *s2), "w2_gs": (E,),
        "sw13": (S, *sc13), "sw13_sf": (S, *ss13), "sw13_gs": (S, 2),
        "sw2": (S, *sc2), "sw2_sf": (S, *ss2), "sw2_gs": (S,),
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


def _fp8_codes(rng: np.random.Generator, n: int) -> np.ndarray:
    """Uniform over the 254 finite E4M3 codes (0x7F and 0xFF are NaN)."""
    u = (np.frombuffer(rng.bytes(2 * n), dtype=np.uint16) % 254).astype(np.int32)
    return (u + (u >= 0x7F)).astype(np.uint8)


def _e8m0_scales(rng: np.random.Generator, n: int, top: int, count: int) -> np.ndarray:
    """E8M0 codes of 2^j, j uniform over the `count` integers ending at `top`."""
    u = np.frombuffer(rng.bytes(n), dtype=np.uint8) % count
    return (127 + top - (count - 1) + u).astype(np.uint8)


def _matrix(fmt, rng_codes, rng_sf, rows, cols):
    """Codes and scales of one [rows, cols] matrix (fan-in cols) in `fmt`."""
    cs, ss, _ = mat_shapes(fmt, rows, cols)
    inv = 1.0 / math.sqrt(cols)
    if fmt == "nvfp4":
        return (_bytes(rng_codes, cs[0] * cs[1]).reshape(cs),
                _scales(rng_sf, ss[0] * ss[1]).reshape(ss))
    if fmt == "mxfp4":
        return (_bytes(rng_codes, cs[0] * cs[1]).reshape(cs),
                _e8m0_scales(rng_sf, ss[0] * ss[1], math.floor(math.log2(inv)), 4).reshape(ss))
    codes = _fp8_codes(rng_codes, cs[0] * cs[1]).reshape(cs)
    if fmt == "mxfp8":
        return codes, _e8m0_scales(rng_sf, ss[0] * ss[1], math.floor(math.log2(inv / 256.0)), 2).reshape(ss)
    u = rng_sf.random(ss[0] * ss[1])
    return codes, ((0.5 + 0.5 * u) * inv / 256.0).astype(np.float32).reshape(ss)


def _one_expert(seed, tags, rows13, rows2, H, I, fmt="nvfp4"):
    t13, t13sf, t2, t2sf, idx = tags
    w13, w13sf = _matrix(fmt, _rng(seed, t13, idx), _rng(seed, t13sf, idx), rows13, H)
    w2, w2sf = _matrix(fmt, _rng(seed, t2, idx), _rng(seed, t2sf, idx), rows2, I)
    return w13, w13sf, w2, w2sf


def make_experts(c: dict, seed: int, experts=None, fill: str = "poison") -> dict:
    """Routed + shared expert tensors.  `experts` (iterable of ids) limits which
    routed experts are drawn; the others get `fill` ("poison": NaN scales and
    0xFF codes; "zero": all-zero bytes)."""
    E, H, I, S, Is = c["E"], c["H"], c["I"], c["S"], c["Is"]
    ef, sfm = c.get("efmt", "nvfp4"), c.get("sfmt", "nvfp4")
    sh = canonical_shapes(c)
    esd = mat_shapes(ef, 1, 128)[2]
    ssd = mat_shapes(sfm, 1, 128)[2]
    want = range(E) if experts is None else sorted(set(int(e) for e in experts))
    # poison: codes 0xFF (E4M3 NaN for the FP8 formats) and NaN scales
    psc = {np.uint8: POISON_SCALE if ef == "nvfp4" else 0xFF, np.float32: np.float32("nan")}[esd]
    if fill == "poison":
        w13 = np.full(sh["w13"], POISON_CODE, np.uint8)
        w13sf = np.full(sh["w13_sf"], psc, esd)
        w2 = np.full(sh["w2"], POISON_CODE, np.uint8)
        w2sf = np.full(sh["w2_sf"], psc, esd)
    else:
        w13 = np.zeros(sh["w13"], np.uint8)
        w13sf = np.zeros(sh["w13_sf"], esd)
        w2 = np.zeros(sh["w2"], np.uint8)
        w2sf = np.zeros(sh["w2_sf"], esd)
    for e in want:
        a, b, d, f = _one_expert(seed, (_T_W13, _T_W13SF, _T_W2, _T_W2SF, e), 2 * I, H, H, I, ef)
        w13[e], w13sf[e], w2[e], w2sf[e] = a, b, d, f
    # tensor scales: NVFP4 only (the other formats have none)
    gs13 = np.full((E, 2), np.float32(1.0 / math.sqrt(H)), np.float32) if ef == "nvfp4" else None
    gs2 = np.full((E,), np.float32(1.0 / math.sqrt(I)), np.float32) if ef == "nvfp4" else None
    out = {"w13": w13, "w13_sf": w13sf, "w13_gs": gs13, "w2": w2, "w2_sf": w2sf, "w2_gs": gs2}
    sw13 = np.empty(sh["sw13"], np.uint8)
    sw13sf = np.empty(sh["sw13_sf"], ssd)
    sw2 = np.empty(sh["sw2"], np.uint8)
    sw2sf = np.empty(sh["sw2_sf"], ssd)
    for s in range(S):
        a, b, d, f = _one_expert(seed, (_T_SW13, _T_SW13SF, _T_SW2, _T_SW2SF, s), 2 * Is, H, H, Is, sfm)
        sw13[s], sw13sf[s], sw2[s], sw2sf[s] = a, b, d, f
    nv = sfm == "nvfp4"
    out.update({
        "sw13": sw13, "sw13_sf": sw13sf,
        "sw13_gs": np.full((S, 2), np.float32(1.0 / math.sqrt(H)), np.float32) if nv else None,
        "sw2": sw2, "sw2_sf": sw2sf,
        "sw2_gs": np.full((S,), np.float32(1.0 / math.sqrt(Is)), np.float32) if nv else None,
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
    per_routed = expert_bytes(c.get("efmt", "nvfp4"), H, I)
    per_shared = expert_bytes(c.get("sfmt", "nvfp4"), H, Is)
    router = E * H * 4 + (E * 4 if c.get("zipf") else 0)
    return router + n_unique_routed * per_routed + S * per_shared + T * H * 2 * 2


def expert_bytes(fmt: str, H: int, I: int) -> int:
    """Bytes of one expert in its own format: codes, block scales and (NVFP4)
    the three FP32 tensor scales."""
    n = 0
    for rows, cols in ((2 * I, H), (H, I)):
        cs, ss, sd = mat_shapes(fmt, rows, cols)
        n += cs[0] * cs[1] + ss[0] * ss[1] * np.dtype(sd).itemsize
    return n + (12 if fmt == "nvfp4" else 0)


def make_layer_torch(c: dict, seed: int, device="cuda") -> dict:
    """The same recipe drawn with torch's generator on `device` (fast, for the
    many distinct layer replicas a timing run needs; these replicas are never
    compared with the oracle).  Returns canonical torch tensors."""
    import torch
    E, H, I, S, Is = c["E"], c["H"], c["I"], c["S"], c["Is"]
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))

    f32 = dict(dtype=torch.float32, device=device)

    def matrix(fmt, n, rows, cols):
        cs, ss, _ = mat_shapes(fmt, rows, cols)
        inv = 1.0 / math.sqrt(cols)
        if fmt in ("nvfp4", "mxfp4"):
            codes = torch.randint(0, 256, (n, *cs), dtype=torch.uint8, device=device, generator=g)
        else:
            u = torch.randint(0, 254, (n, *cs), dtype=torch.int32, device=device, generator=g)
            codes = (u + (u >= 0x7F).to(torch.int32)).to(torch.uint8)
        if fmt == "nvfp4":
            u = torch.rand((n, *ss), generator=g, **f32)
            sf = (0.125 + 0.875 * u).to(torch.float8_e4m3fn).view(torch.uint8)
        elif fmt == "fp8_block":
            sf = (0.5 + 0.5 * torch.rand((n, *ss), generator=g, **f32)) * (inv / 256.0)
        else:
            top, cnt = (math.floor(math.log2(inv)), 4) if fmt == "mxfp4" else (math.floor(math.log2(inv / 256.0)), 2)
            u = torch.randint(0, cnt, (n, *ss), dtype=torch.int32, device=device, generator=g)
            sf = (127 + top - (cnt - 1) + u).to(torch.uint8)
        return codes, sf

    layer = {"cfg": dict(c)}
    layer["router_w"] = torch.randn((E, H), generator=g, **f32) * (1.0 / math.sqrt(H))
    layer["router_b"] = None
    if c.get("zipf"):
        perm = torch.randperm(E, generator=g, device=device).to(torch.float64) + 1.0
        layer["router_b"] = (-ZIPF_ALPHA * ZIPF_S * torch.log(perm)).to(torch.float32)
    ef, sfm = c.get("efmt", "nvfp4"), c.get("sfmt", "nvfp4")
    for pre, n, fmt, Ix in (("", E, ef, I), ("s", S, sfm, Is)):
        layer[pre + "w13"], layer[pre + "w13_sf"] = matrix(fmt, n, 2 * Ix, H)
        layer[pre + "w2"], layer[pre + "w2_sf"] = matrix(fmt, n, H, Ix)
        nv = fmt == "nvfp4"
        layer[pre + "w13_gs"] = torch.full((n, 2), 1.0 / math.sqrt(H), **f32) if nv else None
        layer[pre + "w2_gs"] = torch.full((n,), 1.0 / math.sqrt(Ix), **f32) if nv else None
    return layer


def make_x_torch(c: dict, seed: int, T: int | None = None, device="cuda"):
    import torch
    T = c["T"] if T is None else T
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) + 7919)
    return torch.randn((T, c["H"]), generator=g, dtype=torch.float32, device=device).to(torch.bfloat16)

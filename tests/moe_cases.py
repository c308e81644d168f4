"""Test-side input assembly: seeded layers with a routing-margin guard.

The margin guard needs routing scores, i.e. the layer's arithmetic, so it lives
here (tests may call the oracle) and not in the input generator.  A token whose
k-th and (k+1)-th FP64 sigmoid scores are closer than MARGIN is redrawn from
its next seeded stream, so that FP32 (GPU) and FP64 (oracle) routing cannot
disagree on which experts are selected.
"""
from __future__ import annotations

import numpy as np

import gen
import oracle

MARGIN = 1e-4


def guarded_x(layer: dict, seed: int, T: int, margin: float = MARGIN):
    c = layer["cfg"]
    k = c["k"]
    redraws = []
    for t in range(T):
        r = 0
        while True:
            xt = gen.make_x_token(c, seed, t, r)
            _, _, s, _ = oracle.route(layer, xt[None, :])
            srt = np.sort(s[0])[::-1]
            if k >= c["E"] or srt[k - 1] - srt[k] >= margin:
                break
            r += 1
            if r > 1000:
                raise RuntimeError("margin guard: no admissible redraw")
        redraws.append(r)
    return gen.make_x(c, seed, T, redraws), redraws


def guarded_case(cfg, seed: int, T: int | None = None, full: bool = False,
                 fill: str = "poison", **over):
    """-> (layer, x_bits, info).  Routed experts that no token selects are not
    drawn unless `full` (they get the `fill` pattern instead)."""
    c = gen.config(cfg, **over) if not isinstance(cfg, dict) else dict(cfg)
    T = c["T"] if T is None else T
    router = gen.make_router(c, seed)
    rl = {"cfg": c, **router}
    x, redraws = guarded_x(rl, seed, T)
    ids, w, s, z = oracle.route(rl, x) if T > 0 else (np.zeros((0, c["k"]), np.int32),) * 4
    experts = None if full else np.unique(ids)
    layer = {"cfg": c, **router, **gen.make_experts(c, seed, experts, fill)}
    return layer, x, {"redraws": redraws, "ids": ids, "w": w, "scores": s}


def sorted_gaps_ok(scores_row: np.ndarray, ids_row: np.ndarray, margin: float = MARGIN):
    """Positions j where the order of ids[j], ids[j+1] is decided by a score gap
    of at least `margin` (there the GPU order must match)."""
    s = scores_row[ids_row]
    return np.abs(s[:-1] - s[1:]) >= margin


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)

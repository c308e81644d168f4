"""Helpers shared by the GPU tests: run the CUDA path through the C ABI and
compare it with the oracle."""
from __future__ import annotations

import numpy as np
import torch

from moe_cases import MARGIN, bf16_bits_to_f64, sorted_gaps_ok

ATOL = 1e-2          # |gpu - oracle| <= ATOL + RTOL * |oracle| per output element
RTOL = 1e-2
W_RTOL = 1e-5        # routing weights, relative


def load_moe():
    from nvfp4_weight_only_fp32_gb300 import build
    build.build()
    import nvfp4_weight_only_fp32_gb300 as m
    m.lib()
    return m


def x_to_device(x_bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16).copy()).view(torch.bfloat16).cuda()


def out_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run_gpu(moe, layer, x_bits, max_tokens=None, layer_obj=None, grouped_min_tokens=0, fused=0):
    own = layer_obj is None
    L = layer_obj or moe.MoELayer(layer, max_tokens=max_tokens or x_bits.shape[0],
                                  grouped_min_tokens=grouped_min_tokens, fused=fused)
    x = x_to_device(x_bits)
    out, ids, w = L.forward(x)
    torch.cuda.synchronize()
    assert moe.moe_check(L.h) == moe.MOE_OK, moe.last_error()
    res = out_to_bits(out), ids.cpu().numpy(), w.cpu().numpy()
    if own:
        L.close()
    return res


def check_parity(orc, layer, x_bits, gout, gids, gw, check_order=True):
    oout, opre, oids, ow = orc.forward(layer, x_bits)
    _, _, scores, _ = orc.route(layer, x_bits)
    T = x_bits.shape[0]
    for t in range(T):
        assert sorted(gids[t].tolist()) == sorted(oids[t].tolist()), (t, gids[t], oids[t])
        if check_order:
            ok = sorted_gaps_ok(scores[t], oids[t], MARGIN)
            for j in range(len(ok)):
                if ok[j] and (j == 0 or ok[j - 1]):
                    assert gids[t][j] == oids[t][j], (t, j, gids[t], oids[t])
        for j, e in enumerate(gids[t].tolist()):
            jo = oids[t].tolist().index(e)
            assert abs(gw[t][j] - ow[t][jo]) <= W_RTOL * abs(ow[t][jo]) + 1e-12, (t, j, gw[t][j], ow[t][jo])
    g = bf16_bits_to_f64(gout)
    o = bf16_bits_to_f64(oout)
    assert np.all(np.isfinite(g)), "non-finite GPU output"
    err = np.abs(g - o)
    tol = ATOL + RTOL * np.abs(o)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{bad.sum()} of {bad.size} outputs outside tolerance; worst at {i}: "
                             f"gpu={g[i]} oracle={o[i]} pre={opre[i]}")
    return float(err.max()), float((err / (np.abs(o) + 1e-30)).max())

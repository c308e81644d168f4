"""moe_route_topk_static: routing with no device allocation.

Callers that cannot call cudaMalloc where they route (an engine whose free
device memory already belongs to its KV cache, an allocator that forbids raw
allocations after start-up, code that must not risk an allocation's implicit
synchronisation) use this entry point: its scratch is a static array inside
the library.  This test calls it through the C ABI twice in a row -- a T=8
Flint-shaped layer, then a T=64 layer with a router bias, the largest T the
static scratch holds -- and checks each result against the routing that the
handle-based entry point (moe_decode_forward) returns for the same inputs: ids
exactly, weights within 1e-5 relative.  Each result is also checked against
the oracle's routing of the same guarded inputs (the id set exactly, the order
where neighbouring scores differ by at least the margin, weights within 1e-5
relative).  It also checks that sizes beyond the static limit are refused with
a message naming the limit.  The file is named so that pytest collects it
last."""
import numpy as np
import pytest
import torch

from gpu_util import W_RTOL, load_moe, x_to_device
from moe_cases import MARGIN, guarded_case, sorted_gaps_ok

pytestmark = pytest.mark.gpu


def _handle_routing(moe, layer, x):
    L = moe.MoELayer(layer, max_tokens=x.shape[0])
    try:
        out, ids, w = L.forward(x_to_device(x))
        torch.cuda.synchronize()
        return ids.cpu().numpy(), w.cpu().numpy()
    finally:
        L.close()


def test_static_routing_matches_handle_path_twice():
    moe = load_moe()
    cases = [guarded_case(2, 9101), guarded_case(3, 9102)]
    for layer, x, info in cases:
        c = layer["cfg"]
        ref_ids, ref_w = _handle_routing(moe, layer, x)
        T, k = x.shape[0], c["k"]
        rw = torch.from_numpy(layer["router_w"]).cuda()
        rb = None if layer["router_b"] is None else torch.from_numpy(layer["router_b"]).cuda()
        ids = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
        moe.moe_route_topk_static(rw, rb, c["E"], c["H"], k, c["normalize"], c["routed_scale"],
                                  x_to_device(x), T, ids, w)
        torch.cuda.synchronize()
        got_ids, got_w = ids.cpu().numpy(), w.cpu().numpy()
        assert np.array_equal(got_ids, ref_ids)
        assert np.all(np.abs(got_w - ref_w) <= W_RTOL * np.abs(ref_w) + 1e-12)
        # against the oracle (FP64 routing of the same inputs)
        oids, ow, scores = info["ids"], info["w"], info["scores"]
        for t in range(T):
            assert sorted(got_ids[t].tolist()) == sorted(oids[t].tolist()), (t, got_ids[t], oids[t])
            ok = sorted_gaps_ok(scores[t], oids[t], MARGIN)
            for j in range(len(ok)):
                if ok[j] and (j == 0 or ok[j - 1]):
                    assert got_ids[t][j] == oids[t][j], (t, j, got_ids[t], oids[t])
            for j, e in enumerate(got_ids[t].tolist()):
                jo = oids[t].tolist().index(e)
                assert abs(got_w[t][j] - ow[t][jo]) <= W_RTOL * abs(ow[t][jo]) + 1e-12, (t, j)


def test_static_routing_refuses_sizes_beyond_its_scratch():
    moe = load_moe()
    rw = torch.zeros((600, 64), dtype=torch.float32, device="cuda")
    x = torch.zeros((65, 64), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((65, 2), dtype=torch.int32, device="cuda")
    w = torch.empty((65, 2), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_route_topk_static(rw, None, 600, 64, 2, 1, 1.0, x, 65, ids, w)
    assert ei.value.status == moe.moe.MOE_ERR_UNSUPPORTED
    msg = str(ei.value)
    assert "T=65" in msg and "num_experts=600" in msg and "64 tokens x 512 experts" in msg

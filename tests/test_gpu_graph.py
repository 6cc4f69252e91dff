"""The whole path captured once in a CUDA graph and replayed with new routing.

Live counts, offsets and page allocation stay on the device, so one capture
serves every replay even though each replay routes different tokens (device
counts that change under CUDA-graph replay: torchtitan pull 5541,
"Verification").  Each replay is checked against the oracle chain."""
import numpy as np
import pytest
import torch

import oracle
from activation_paging_gb300 import inputs
from gpu_util import bf16_to_host, combine_within, host, route_tolerance

pytestmark = pytest.mark.gpu

ap = pytest.importorskip("activation_paging_gb300")


@pytest.mark.parametrize("mode", ["separate", "fused", "route_fused"])
def test_graph_replay_with_changing_routing(mode):
    """mode: route, dispatch and push as three calls; route then the fused
    dispatch + push; or route, dispatch and push as one call."""
    T, H, E, k, P, chunks = 1024, 256, 32, 4, 16, 2
    rb = H * 2
    rows = T * k
    N = int(1.3 * chunks * rows / P)
    page_bytes = ap.page_bytes_for(P, (rb,))
    pool = ap.Pool(P, page_bytes, N, 1, 4, E, N)
    o = oracle.Pool(P, page_bytes, N, 1, 4, E, N, 0, keep_bytes=False)
    s = pool.stream
    dev = "cuda"
    bufs = []
    for c in range(chunks):
        b = {"logits": torch.empty((T, E), dtype=torch.float32, device=dev),
             "x": torch.empty((T, H), dtype=torch.bfloat16, device=dev),
             "y": torch.empty((rows, H), dtype=torch.bfloat16, device=dev),
             "idx": torch.empty((T, k), dtype=torch.int32, device=dev),
             "w": torch.empty((T, k), dtype=torch.float32, device=dev),
             "dst": torch.empty((rows, H), dtype=torch.bfloat16, device=dev),
             "out": torch.empty((T, H), dtype=torch.bfloat16, device=dev)}
        b["disp"] = {"xd": torch.empty((rows, H), dtype=torch.bfloat16, device=dev)}
        bufs.append(b)

    def load(rep):
        host_in = []
        for c, b in enumerate(bufs):
            seed = 10 * rep + c
            logits = inputs.router_logits(seed, T, E)
            x = inputs.normal_bf16(seed, inputs.X_STREAM, (T, H))
            y = inputs.normal_bf16(seed, inputs.Y_STREAM, (rows, H))
            with torch.cuda.stream(s):
                b["logits"].copy_(torch.from_numpy(logits))
                b["x"].copy_(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16))
                b["y"].copy_(torch.from_numpy(y.view(np.int16)).view(torch.bfloat16))
            host_in.append((logits, x, y))
        return host_in

    def step():
        for b in bufs:
            if mode == "route_fused":
                b["disp"] = pool.route_dispatch_stash(0, b["logits"], b["x"], k, E,
                                                      out=dict(b["disp"], idx=b["idx"], w=b["w"]))
                continue
            ap.route_topk(b["logits"], k, b["idx"], b["w"], stream=s)
            if mode == "fused":
                b["disp"] = pool.dispatch_stash(0, b["x"], b["idx"], E, out=b["disp"])
            else:
                b["disp"] = ap.dispatch_permute(b["x"], b["idx"], E, out=b["disp"], stream=s)
                pool.push(0, [b["disp"]["xd"]], b["disp"]["seg_off"], b["disp"]["live"])
        for b in bufs:
            pool.pop(0, [b["dst"]])
            ap.combine_unpermute(b["y"], b["disp"]["dest"], b["w"], out=b["out"], stream=s)

    def oracle_step(host_in):
        res = []
        for logits, x, y in host_in:
            idx, w = oracle.route_topk(logits, k)
            plan = oracle.dispatch(x, idx, E, 0, False)
            o.push_rb(0, (rb,), plan["rows"], plan["seg_off"], plan["live"])
            res.append((logits, idx, w, plan, y))
        for _ in host_in:
            o.pop(0, None, rows, nplanes=1)
        return res

    def check(res):
        torch.cuda.synchronize()
        assert pool.state() == o.state()
        rg, _ = pool.rings()
        ro, _ = o.rings()
        assert np.array_equal(rg, ro)
        for b, (logits, idx, w, plan, y) in zip(bufs, res):
            assert np.array_equal(host(b["idx"]), idx)
            assert np.all(np.abs(host(b["w"]).astype(np.float64) - w) <= route_tolerance(logits, idx, w))
            for key in ("counts", "live", "seg_off", "dest"):
                assert np.array_equal(host(b["disp"][key]), plan[key]), key
            assert np.array_equal(bf16_to_host(b["dst"]), plan["xd"])
            # the GPU combine used the GPU's weights, which differ from the
            # oracle's within the routing bound; the output bound follows
            exp, _ = oracle.combine(y, plan["dest"], w)
            assert combine_within(bf16_to_host(b["out"]), exp, y, plan["dest"], w, route_tolerance(logits, idx, w))

    # eager warm-up (allocates nothing inside the capture afterwards)
    res = oracle_step(load(0))
    with torch.cuda.stream(s):
        step()
    check(res)

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    counts_seen = []
    for rep in range(1, 5):
        res = oracle_step(load(rep))
        with torch.cuda.stream(s):
            graph.replay()
        check(res)
        counts_seen.append(tuple(host(bufs[0]["disp"]["counts"])))
    assert len(set(counts_seen)) == len(counts_seen)  # every replay routed differently
    assert pool.state()["head"] > N  # the free ring wrapped during the replays

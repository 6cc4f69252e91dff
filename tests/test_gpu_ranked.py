"""GPU parity of the split fused dispatch + push: count/rank (ap_count_rank,
optionally routing first and optionally with the expert scan) on a second
stream, then ap_dispatch_stash_ranked on the paging stream after an event.

Same results as the oracle's dispatch followed by its push (torchtitan pull
5541, "AI-Generated Details": the stash committed by the producer of the
rows): dispatch outputs, record, page table, pool bytes, rings, state and
flags, for records the copy kernel plans itself (one- and four-column count
reads) and records planned by the scan + plan kernel, compact and padded,
BF16 and E4M3, with overflowing pools."""
import numpy as np
import pytest
import torch

import oracle
from activation_paging_gb300 import inputs
from gpu_util import bf16_to_dev, bf16_to_host, host, to_dev

pytestmark = pytest.mark.gpu

ap = pytest.importorskip("activation_paging_gb300")
FILL = 0xA5


@pytest.mark.parametrize("scan", [False, True])
@pytest.mark.parametrize("T,H,E,k,C,padded,P,N,SP,fp8,route", [
    (4096, 256, 64, 6, 0, False, 32, 900, 0, False, False),     # planned in the copy kernel, one-column reads
    (8192, 256, 128, 8, 0, False, 64, 1200, 0, False, True),    # the headline's counts (128 x 128), routed
    (6000, 64, 48, 4, 560, True, 16, 1800, 0, False, False),    # padded, four-column reads, ragged row groups
    (17000, 64, 64, 4, 0, False, 64, 900, 200, False, True),    # scan + plan kernel (272 x 64 counts); spill
    (4096, 2056, 64, 6, 0, False, 128, 120, 0, True, False),    # E4M3, rows 8 bytes off; the pool overflows
    (4096, 2048, 64, 6, 0, False, 128, 260, 0, True, True),     # E4M3, aligned rows, routed; every page kept
    (3000, 1024, 32, 4, 300, True, 64, 200, 16, True, False),   # E4M3 padded with drops; spill
    (512, 128, 8, 2, 0, False, 16, 10, 4, False, True),         # spill exhausted: lost pages
])
def test_ranked_dispatch_stash_matches_oracle(T, H, E, k, C, padded, P, N, SP, fp8, route, scan):
    rb = (H, 4) if fp8 else (2 * H,)
    page_bytes = ap.page_bytes_for(P, rb)
    g = ap.Pool(P, page_bytes, N, 1, 4, E, N + SP + E, SP, fill=FILL)
    o = oracle.Pool(P, page_bytes, N, 1, 4, E, N + SP + E, SP, keep_bytes=True, fill=FILL)
    side = torch.cuda.Stream()
    for rep in range(2):
        logits = inputs.router_logits(700 + T + rep, T, E)
        x = inputs.normal_bf16(700 + T + rep, inputs.X_STREAM, (T, H))
        idx_o, w_o = oracle.route_topk(logits, k)
        plan = oracle.dispatch(x, idx_o, E, C, padded, fp8=fp8)
        planes = ([plan["xd"], plan["xd_scale"].view(np.uint8).reshape(-1, 4)] if fp8
                  else [plan["xd"].view(np.uint8).reshape(plan["rows"], rb[0])])
        rid_o = o.push(0, planes, plan["rows"], plan["seg_off"], plan["live"])
        xg = bf16_to_dev(x)
        out = {"xd": torch.full((plan["rows"], H), 0xA5, dtype=torch.uint8, device="cuda") if fp8 else
               torch.full((plan["rows"], H), 0xA5A5 - 0x10000, dtype=torch.int16, device="cuda").view(torch.bfloat16)}
        if fp8:
            out["xd_scale"] = torch.from_numpy(np.full(plan["rows"] * 4, 0xA5, np.uint8).view(np.float32)).cuda()
        torch.cuda.synchronize()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):  # count/rank beside the paging stream
            if route:
                r = ap.count_rank(E, logits=to_dev(logits), k=k, x=xg, stream=side, scan=scan, capacity=C,
                                  padded=padded)
            else:
                r = ap.count_rank(E, idx=to_dev(idx_o), x=xg, stream=side, scan=scan, capacity=C, padded=padded)
            ranked = torch.cuda.Event()
            ranked.record(side)
        g.stream.wait_event(ranked)
        out.update({key: r[key] for key in ("dest", "scratch", "counts", "live", "seg_off", "scanned") if key in r})
        with torch.cuda.stream(g.stream):
            d = g.dispatch_stash(0, xg, r["idx"], E, C, padded, fp8=fp8, out=out, ranked=True)
        torch.cuda.synchronize()
        if route:
            assert np.array_equal(host(r["idx"]), idx_o)
        assert d["record_id"] == rid_o
        for key in ("counts", "live", "seg_off", "dest"):
            assert np.array_equal(host(d[key]), plan[key]), key
        if fp8:
            assert np.array_equal(host(d["xd"]), plan["xd"])
            assert np.array_equal(host(d["xd_scale"]).view(np.uint32), plan["xd_scale"].view(np.uint32))
        else:
            assert np.array_equal(bf16_to_host(d["xd"]), plan["xd"])
        assert g.state() == o.state()
        a, b = g.record(0, rep), o.record(0, rep)
        for key in ("id", "npages", "ndev", "nspill", "nlost"):
            assert a[key] == b[key], key
        for key in ("page_table", "row0", "nrows"):
            assert np.array_equal(a[key], b[key]), key
    assert np.array_equal(host(g.pool), o.pool_bytes())
    if SP:
        assert np.array_equal(g.spill.numpy(), o.spill_bytes())
    rg, sg = g.rings()
    ro, so = o.rings()
    assert np.array_equal(rg, ro) and np.array_equal(sg, so)
    assert g.overflow() == o.state()["flags"]

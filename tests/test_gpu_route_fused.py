"""GPU parity: route + fused dispatch + push in one call.

``ap_route_dispatch_stash`` must leave exactly what ``ap_route_topk``
followed by ``ap_dispatch_stash`` leaves (ids, weights, dispatch outputs,
record, pool bytes, state), and match the oracle's route, dispatch and push."""
import numpy as np
import pytest
import torch

import oracle
from activation_paging_gb300 import inputs
from gpu_util import bf16_to_dev, bf16_to_host, host, route_tolerance, to_dev

pytestmark = pytest.mark.gpu

ap = pytest.importorskip("activation_paging_gb300")
FILL = 0xA5


def pools(P, rb, N, E, SP=0):
    page_bytes = ap.page_bytes_for(P, rb)
    mk = lambda: ap.Pool(P, page_bytes, N, 1, 4, E, N + SP + E, SP, fill=FILL)  # noqa: E731
    return mk(), mk(), page_bytes


@pytest.mark.parametrize("T,H,E,k,C,padded,fp8", [
    (8192, 256, 128, 8, 0, False, False),   # the benchmark's router shape, 128 count/rank blocks
    (1000, 64, 64, 6, 0, False, True),      # E4M3 records, ragged last block
    (777, 2056, 32, 5, 0, False, False),    # odd hidden size (8-byte rows)
    (300, 128, 256, 8, 40, True, False),    # padded with drops; 8 candidates per lane
    (129, 64, 1024, 32, 0, False, False),   # wide router: routed and ranked in two launches
    (65, 64, 1, 1, 0, False, False),        # one expert
    (0, 64, 8, 2, 0, False, False),         # no tokens
])
def test_route_dispatch_stash_equals_two_calls(T, H, E, k, C, padded, fp8):
    P = 16
    rb = (H, 4) if fp8 else (2 * H,)
    rows = E * C if padded else T * k
    N = rows // P + E + 8
    a, b, _ = pools(P, rb, N, E)
    logits = torch.from_numpy(inputs.router_logits(T + E, T, E)).cuda()
    x = bf16_to_dev(inputs.normal_bf16(T + E, inputs.X_STREAM, (T, H)))
    canary = lambda: torch.full((rows, H), 0x5A, dtype=torch.uint8, device="cuda") if fp8 else \
        torch.full((rows, H), 0x5A5A, dtype=torch.int16, device="cuda").view(torch.bfloat16)  # noqa: E731
    torch.cuda.synchronize()
    with torch.cuda.stream(a.stream):
        a.stream.wait_stream(torch.cuda.default_stream())
        idx, w = ap.route_topk(logits, k, stream=a.stream)
        da = a.dispatch_stash(0, x, idx, E, C, padded, fp8=fp8, out={"xd": canary()})
    with torch.cuda.stream(b.stream):
        b.stream.wait_stream(torch.cuda.default_stream())
        db = b.route_dispatch_stash(0, logits, x, k, E, C, padded, fp8=fp8, out={"xd": canary()})
    torch.cuda.synchronize()
    assert torch.equal(db["idx"], idx)
    assert torch.equal(db["w"].view(torch.int32), w.view(torch.int32))  # the same routing code: bit-identical
    keys = ["counts", "live", "seg_off", "dest", "src_tok"] + (["xd_scale"] if fp8 else [])
    for key in keys:
        assert torch.equal(da[key].view(torch.int32), db[key].view(torch.int32)), key
    assert torch.equal(da["xd"].view(torch.uint8), db["xd"].view(torch.uint8))
    assert a.state() == b.state()
    assert torch.equal(a.pool, b.pool)
    ra, rb_ = a.record(0), b.record(0)
    for key in ("page_table", "row0", "nrows"):
        assert np.array_equal(ra[key], rb_[key]), key


@pytest.mark.parametrize("T,H,E,k,P,N,SP", [
    (2049, 128, 64, 6, 32, 300, 200),   # ragged blocks; pool overflows into spill
    (512, 256, 16, 4, 8, 50, 0),        # lost pages
])
def test_route_dispatch_stash_matches_oracle(T, H, E, k, P, N, SP):
    rb = 2 * H
    page_bytes = ap.page_bytes_for(P, (rb,))
    g = ap.Pool(P, page_bytes, N, 1, 4, E, N + SP + E, SP, fill=FILL)
    o = oracle.Pool(P, page_bytes, N, 1, 4, E, N + SP + E, SP, keep_bytes=True, fill=FILL)
    logits = inputs.router_logits(T, T, E)
    x = inputs.normal_bf16(T, inputs.X_STREAM, (T, H))
    idx_o, w_o = oracle.route_topk(logits, k)
    plan = oracle.dispatch(x, idx_o, E, 0, False)
    o.push(0, [plan["xd"].view(np.uint8).reshape(plan["rows"], rb)], plan["rows"], plan["seg_off"], plan["live"])
    with torch.cuda.stream(g.stream):
        g.stream.wait_stream(torch.cuda.default_stream())
        d = g.route_dispatch_stash(0, to_dev(logits), bf16_to_dev(x), k, E)
    torch.cuda.synchronize()
    assert np.array_equal(host(d["idx"]), idx_o)
    assert np.all(np.abs(host(d["w"]).astype(np.float64) - w_o) <= route_tolerance(logits, idx_o, w_o))
    for key in ("counts", "live", "seg_off", "dest"):
        assert np.array_equal(host(d[key]), plan[key]), key
    assert np.array_equal(bf16_to_host(d["xd"]), plan["xd"])
    assert g.state() == o.state()
    assert np.array_equal(host(g.pool), o.pool_bytes())
    if SP:
        assert np.array_equal(g.spill.numpy(), o.spill_bytes())


def test_route_dispatch_stash_host_errors():
    g = ap.Pool(8, ap.page_bytes_for(8, (2 * 16,)), 64, 1, 1, 8)
    logits = torch.zeros((32, 8), dtype=torch.float32, device="cuda")
    x = torch.zeros((32, 16), dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(g.stream):
        with pytest.raises(ap.APError) as e:
            g.route_dispatch_stash(0, logits, x, 9, 8)  # k > E
        assert e.value.status == -1
    idx = torch.zeros((32, 2), dtype=torch.int32, device="cuda")
    w = torch.zeros((32, 2), dtype=torch.float32, device="cuda")
    rc = g.lib.ap_route_dispatch_stash(g.handle, 0, None, w.data_ptr(), x.data_ptr(), 32, 16, idx.data_ptr(), 2, 8, 0,
                                       0, 0, None, None, 64, None, None, None, None, None, None, 0, None, None,
                                       g.stream.cuda_stream)
    assert rc == -1  # no logits
    rc = g.lib.ap_route_dispatch_stash(g.handle, 0, logits.data_ptr(), w.data_ptr(), x.data_ptr(), 32, 16,
                                       idx.data_ptr(), 2, 8, 0, 0, 0, None, None, 64, None, None, None, None, None,
                                       None, 0, None, None, torch.cuda.Stream().cuda_stream)
    assert rc == -5  # not the paging stream


def test_route_dispatch_stash_headline_shape_matches_oracle():
    """Route + fused dispatch + push at the benchmark's chunk shape (T=8192,
    H=2048, E=128, top-8, dropless, 64-token pages, the benchmark's pool)
    against the oracle: ids exact, weights within the derived bound, every
    dispatch output, the record's page table and descriptors, the pool state,
    and every page's rows."""
    wl = inputs.WORKLOADS["qwen3_moe"]
    T, H, E, k, P = wl.T, wl.H, wl.E, wl.k, wl.page_tokens
    rb = 2 * H
    g = ap.Pool(P, wl.page_bytes, wl.num_pages, 1, 4, E, wl.num_pages, fill=FILL)
    o = oracle.Pool(P, wl.page_bytes, wl.num_pages, 1, 4, E, wl.num_pages, 0, keep_bytes=False)
    logits = inputs.router_logits(0, T, E)
    x = inputs.normal_bf16(0, inputs.X_STREAM, (T, H))
    idx_o, w_o = oracle.route_topk(logits, k)
    plan = oracle.dispatch(x, idx_o, E, 0, False)
    o.push_rb(0, (rb,), plan["rows"], plan["seg_off"], plan["live"])
    with torch.cuda.stream(g.stream):
        g.stream.wait_stream(torch.cuda.default_stream())
        d = g.route_dispatch_stash(0, to_dev(logits), bf16_to_dev(x), k, E)
    torch.cuda.synchronize()
    assert np.array_equal(host(d["idx"]), idx_o)
    assert np.all(np.abs(host(d["w"]).astype(np.float64) - w_o) <= route_tolerance(logits, idx_o, w_o))
    for key in ("counts", "live", "seg_off", "dest"):
        assert np.array_equal(host(d[key]), plan[key]), key
    assert np.array_equal(host(d["src_tok"])[:plan["rows"]], plan["src_tok"])
    assert np.array_equal(bf16_to_host(d["xd"]), plan["xd"])
    assert g.state() == o.state()
    a, b = g.record(0), o.record(0)
    for key in ("npages", "ndev", "nspill", "nlost"):
        assert a[key] == b[key], key
    for key in ("page_table", "row0", "nrows"):
        assert np.array_equal(a[key], b[key]), key
    # every page holds the dispatched rows it was given (the oracle's rows, checked above)
    xd_bytes = d["xd"].view(torch.uint8).reshape(plan["rows"], rb)
    for pid, r0, nr in zip(a["page_table"].tolist(), a["row0"].tolist(), a["nrows"].tolist()):
        assert 0 <= pid < g.N
        page = g.pool[pid * wl.page_bytes: pid * wl.page_bytes + nr * rb]
        assert torch.equal(page, xd_bytes[r0:r0 + nr].reshape(-1))

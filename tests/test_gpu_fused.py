"""GPU parity: the fused dispatch + push against the oracle's dispatch and push.

The fused call must leave exactly what a dispatch followed by a push leaves:
dispatch outputs, the record and its page table, rings, counters, flags and
every pool / spill byte (compared with the oracle's byte-exact pool), and the
pop of the record must give the dispatched rows back."""
import numpy as np
import pytest
import torch

import oracle
from activation_paging_gb300 import inputs
from gpu_util import bf16_to_dev, bf16_to_host, host, to_dev

pytestmark = pytest.mark.gpu

ap = pytest.importorskip("activation_paging_gb300")
FILL = 0xA5


@pytest.mark.parametrize("T,H,E,k,C,padded,P,N,SP", [
    (512, 128, 8, 2, 160, True, 16, 80, 0),       # padded, exactly enough pages
    (1000, 264, 16, 4, 0, False, 32, 150, 0),     # compact, 8-byte rows path, page tails
    (777, 2056, 32, 6, 0, False, 64, 40, 64),     # odd hidden size; pool overflows into spill
    (300, 64, 8, 2, 0, False, 8, 10, 5),          # spill exhausted: lost pages
    (600, 64, 1024, 16, 0, False, 8, 3000, 0),    # the most experts
    (131100, 64, 64, 8, 0, False, 64, 16000, 2000),  # a record of 1.05 M pairs; spills
    # records planned inside the copy kernel with more than sixteen count/rank
    # blocks per reading thread: four-column reads (128 x 128 counts, the
    # headline's; 94 x 48 with a ragged last row group), padded, and one-column
    # reads for E % 4 != 0
    (8192, 256, 128, 8, 0, False, 64, 2400, 0),
    (6000, 64, 48, 4, 0, False, 16, 1600, 0),
    (6000, 64, 48, 4, 560, True, 16, 1800, 0),
    (6000, 64, 50, 4, 0, False, 16, 1600, 0),
])
def test_fused_matches_oracle_dispatch_then_push(T, H, E, k, C, padded, P, N, SP):
    rb = H * 2
    page_bytes = ap.page_bytes_for(P, (rb,))
    g = ap.Pool(P, page_bytes, N, 2, 4, E, N + SP + E, SP, fill=FILL)
    o = oracle.Pool(P, page_bytes, N, 2, 4, E, N + SP + E, SP, keep_bytes=True, fill=FILL)
    for rep in range(2):
        logits = inputs.router_logits(T + rep, T, E)
        x = inputs.normal_bf16(T + rep, inputs.X_STREAM, (T, H))
        idx, _ = oracle.route_topk(logits, k)
        plan = oracle.dispatch(x, idx, E, C, padded)
        rid_o = o.push(rep, [plan["xd"].view(np.uint8).reshape(plan["rows"], rb)], plan["rows"], plan["seg_off"],
                       plan["live"])
        xd_dev = torch.full((plan["rows"], H), 0xA5A5 - 0x10000, dtype=torch.int16, device="cuda")
        torch.cuda.synchronize()
        with torch.cuda.stream(g.stream):
            d = g.dispatch_stash(rep, bf16_to_dev(x), to_dev(idx), E, C, padded,
                                 out={"xd": xd_dev.view(torch.bfloat16)})
        torch.cuda.synchronize()
        assert d["record_id"] == rid_o
        for key in ("counts", "live", "seg_off", "dest"):
            assert np.array_equal(host(d[key]), plan[key]), key
        assert np.array_equal(bf16_to_host(d["xd"]), plan["xd"])
        assert g.state() == o.state()
        a, b = g.record(rep, 0), o.record(rep, 0)
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
    # pops give the rows back (lost pages leave the canary)
    for rep in range(2):
        rec = o.record(rep, 0)
        rows = int(max(rec["row0"] + rec["nrows"])) + 1 if rec["npages"] else 1
        dst_np = [np.full((rows, rb), 0x3C, np.uint8)]
        dst = to_dev(dst_np[0])
        torch.cuda.synchronize()
        g.pop(rep, [dst])
        o.pop(rep, dst_np, rows)
        torch.cuda.synchronize()
        assert np.array_equal(host(dst), dst_np[0])
    assert g.state() == o.state()


def test_fused_equals_unfused_on_the_gpu():
    wl = inputs.WORKLOADS["qwen3_moe"]
    logits = torch.from_numpy(inputs.router_logits(5, wl.T, wl.E)).cuda()
    x = bf16_to_dev(inputs.normal_bf16(5, inputs.X_STREAM, (wl.T, wl.H)))
    idx, _ = ap.route_topk(logits, wl.k)
    a = ap.Pool(wl.page_tokens, wl.page_bytes, wl.num_pages, 1, 2, wl.E, fill=0)
    b = ap.Pool(wl.page_tokens, wl.page_bytes, wl.num_pages, 1, 2, wl.E, fill=0)
    d1 = ap.dispatch_permute(x, idx, wl.E)
    a.push(0, [d1["xd"]], d1["seg_off"], d1["live"])
    with torch.cuda.stream(b.stream):
        b.stream.wait_stream(torch.cuda.default_stream())
        d2 = b.dispatch_stash(0, x, idx, wl.E)
    torch.cuda.synchronize()
    for key in ("counts", "live", "seg_off", "dest", "xd"):
        assert torch.equal(d1[key].view(torch.int16) if key == "xd" else d1[key],
                           d2[key].view(torch.int16) if key == "xd" else d2[key]), key
    assert a.state() == b.state()
    ra, rb_ = a.record(0), b.record(0)
    assert np.array_equal(ra["page_table"], rb_["page_table"])
    assert torch.equal(a.pool, b.pool)


def test_fused_host_errors():
    g = ap.Pool(8, ap.page_bytes_for(8, (2 * 6,)), 16, 1, 1, 4)
    x = torch.zeros((16, 6), dtype=torch.bfloat16, device="cuda")  # 12-byte rows: not 8-byte aligned
    idx = torch.zeros((16, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(ap.APError) as e:
        with torch.cuda.stream(g.stream):
            g.dispatch_stash(0, x, idx, 4)
    assert e.value.status == -6
    rc = g.lib.ap_dispatch_stash(g.handle, 0, None, 0, 8, None, 2, 4, 0, 0, 0, None, None, 0, None, None, None, None,
                                 None, None, 0, None, None, torch.cuda.Stream().cuda_stream)
    assert rc == -5  # not the paging stream


# Two warps per token. A row of H values is H/8 16-byte vectors (8 bf16 each).
# When every row is 16-byte aligned (H % 16 == 0 and aligned buffers), warp 0
# takes the first ceil(H/16) vectors and warp 1 the rest, one per lane per
# round. Otherwise the row is cut into 16-code units of two vectors and, for
# odd H/8, one lone last vector; warp 0 takes the first ceil(units/2) units,
# warp 1 the rest and the lone vector, and rows that start 8 bytes off a
# 16-byte boundary get aligned 16-byte stores straddling two units. xd_off
# starts the dispatch buffer 8 bytes into its allocation.
@pytest.mark.parametrize("T,H,E,k,P,N,SP,xd_off", [
    (4096, 2048, 64, 6, 128, 120, 0, 0),    # the FP8 layer-stack shape: 128 / 128 vectors, 4 rounds
    (4096, 2056, 64, 6, 128, 120, 0, 0),    # its non-divisible variant: 64 / 64 units and the lone vector
    (999, 2056, 64, 6, 128, 40, 64, 0),     # the same rows with spill
    (300, 1024, 16, 4, 32, 20, 4, 0),       # 64 / 64 vectors, 2 rounds; lost pages
    (600, 4096, 32, 4, 32, 100, 16, 0),     # the widest rows: 256 / 256 vectors, 8 rounds; spill
    (500, 2304, 32, 4, 32, 100, 16, 0),     # 144 / 144 vectors: the 5-round instance; spill
    (700, 2312, 48, 5, 64, 70, 40, 0),      # 72 / 72 units and a lone vector: 3 rounds, ragged; spill
    (175000, 64, 64, 6, 128, 8300, 100, 0),  # a record of 1.05 M pairs, 4 / 4 vectors; spills
    (257, 8, 8, 2, 16, 64, 8, 0),           # a lone vector and no unit: warp 1 writes the whole row
    (300, 16, 8, 3, 16, 80, 8, 8),          # one unit, warp 1 idle; every dispatch row 8 bytes off
    (300, 24, 8, 3, 16, 80, 8, 0),          # one unit and the lone vector (warp 0's lookahead)
    (200, 40, 16, 4, 8, 120, 0, 0),         # 1 / 1 units and the lone vector
    (333, 1024, 16, 4, 32, 50, 8, 8),       # 32 / 32 units, dispatch rows 8 bytes off, page rows aligned
    (333, 1032, 16, 4, 32, 50, 8, 0),       # 32 / 32 units and the lone vector: the widest one-round rows
    (333, 1040, 16, 4, 32, 50, 8, 0),       # 33 / 32 units: one lane of warp 0 takes a second round
    (250, 3080, 16, 4, 32, 40, 8, 0),       # 96 / 96 units and the lone vector: the widest three-round rows
    (250, 4088, 16, 4, 32, 40, 8, 0),       # 128 / 127 units and the lone vector: four rounds
])
def test_fused_e4m3_matches_oracle(T, H, E, k, P, N, SP, xd_off):
    rb = (H, 4)
    page_bytes = ap.page_bytes_for(P, rb)
    g = ap.Pool(P, page_bytes, N, 1, 4, E, N + SP + E, SP, fill=FILL)
    o = oracle.Pool(P, page_bytes, N, 1, 4, E, N + SP + E, SP, keep_bytes=True, fill=FILL)
    logits = inputs.router_logits(H + T, T, E)
    x = inputs.normal_bf16(H + T, inputs.X_STREAM, (T, H))
    idx, _ = oracle.route_topk(logits, k)
    plan = oracle.dispatch(x, idx, E, 0, False, fp8=True)
    rid_o = o.push(0, [plan["xd"], plan["xd_scale"].view(np.uint8).reshape(-1, 4)], plan["rows"], plan["seg_off"],
                   plan["live"])
    xd = torch.full((plan["rows"] * H + xd_off,), 0xA5, dtype=torch.uint8, device="cuda")[xd_off:].view(plan["rows"], H)
    assert xd.data_ptr() % 16 == xd_off
    xs = torch.from_numpy(np.full(plan["rows"] * 4, 0xA5, np.uint8).view(np.float32)).cuda()
    torch.cuda.synchronize()
    with torch.cuda.stream(g.stream):
        d = g.dispatch_stash(0, bf16_to_dev(x), to_dev(idx), E, fp8=True, out={"xd": xd, "xd_scale": xs})
    torch.cuda.synchronize()
    assert d["record_id"] == rid_o
    for key in ("counts", "live", "seg_off", "dest"):
        assert np.array_equal(host(d[key]), plan[key]), key
    assert np.array_equal(host(d["xd"]), plan["xd"])
    assert np.array_equal(host(d["xd_scale"]).view(np.uint32), plan["xd_scale"].view(np.uint32))
    assert g.state() == o.state()
    a, b = g.record(0, 0), o.record(0, 0)
    for key in ("npages", "ndev", "nspill", "nlost"):
        assert a[key] == b[key], key
    assert np.array_equal(a["page_table"], b["page_table"])
    assert np.array_equal(host(g.pool), o.pool_bytes())
    if SP:
        assert np.array_equal(g.spill.numpy(), o.spill_bytes())
    dq = [np.full((plan["rows"], H), 0x3C, np.uint8), np.full((plan["rows"], 4), 0x3C, np.uint8)]
    dg = [to_dev(dq[0]), to_dev(dq[1])]
    torch.cuda.synchronize()
    g.pop(0, dg)
    o.pop(0, dq, plan["rows"])
    torch.cuda.synchronize()
    assert np.array_equal(host(dg[0]), dq[0]) and np.array_equal(host(dg[1]), dq[1])
    assert g.state() == o.state()


def test_launch_counter_counts_enqueued_kernels():
    """The library counts the kernels it enqueues: eager calls as they launch,
    graph capture once, replays not at all."""
    T, H, E, k = 256, 64, 8, 2
    logits = torch.from_numpy(inputs.router_logits(3, T, E)).cuda()
    x = bf16_to_dev(inputs.normal_bf16(3, inputs.X_STREAM, (T, H)))
    g = ap.Pool(16, ap.page_bytes_for(16, (2 * H,)), 64, 1, 2, E)
    n0 = ap.launch_count()
    idx, w = ap.route_topk(logits, k)
    assert ap.launch_count() - n0 == 1
    n1 = ap.launch_count()
    with torch.cuda.stream(g.stream):
        g.stream.wait_stream(torch.cuda.default_stream())
        d = g.dispatch_stash(0, x, idx, E)
        y = torch.empty_like(d["xd"])
        g.pop(0, [y])
    torch.cuda.synchronize()
    assert ap.launch_count() - n1 == 3  # a small record: count/rank, fused copy (which plans it), pop copy
    # a record with more block counts than the copy kernel plans itself (T/64 blocks x E > 16384):
    # count/rank, scan + plan, fused copy, pop copy
    T2, E2 = 4160, 256
    x2 = bf16_to_dev(inputs.normal_bf16(4, inputs.X_STREAM, (T2, H)))
    idx2 = torch.randint(0, E2, (T2, 2), dtype=torch.int32, device="cuda")
    g2 = ap.Pool(16, ap.page_bytes_for(16, (2 * H,)), T2 * 2 // 16 + E2, 1, 2, E2)
    n2 = ap.launch_count()
    with torch.cuda.stream(g2.stream):
        g2.stream.wait_stream(torch.cuda.default_stream())
        d2 = g2.dispatch_stash(0, x2, idx2, E2)
        g2.pop(0, [torch.empty_like(d2["xd"])])
    torch.cuda.synchronize()
    assert ap.launch_count() - n2 == 4
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ap.route_topk(logits, k, idx, w, stream=s)  # warm-up outside the capture
    torch.cuda.synchronize()
    n2 = ap.launch_count()
    with torch.cuda.graph(graph, stream=s):
        ap.route_topk(logits, k, idx, w, stream=s)
    assert ap.launch_count() - n2 == 1
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert ap.launch_count() - n2 == 1


def test_copy_kernel_timing_events():
    """ap_pool_time_copies: the library records the caller's events around
    the copy kernel; that span lies inside the whole call's span."""
    T, H, E, k = 4096, 512, 16, 4
    logits = torch.from_numpy(inputs.router_logits(9, T, E)).cuda()
    x = bf16_to_dev(inputs.normal_bf16(9, inputs.X_STREAM, (T, H)))
    g = ap.Pool(16, ap.page_bytes_for(16, (2 * H,)), T * k // 16 + E, 1, 2, E)
    idx, _ = ap.route_topk(logits, k)
    torch.cuda.synchronize()
    spans = []
    for call in ("dispatch_stash", "pop"):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ca, cb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g.time_copies(ca, cb)
        with torch.cuda.stream(g.stream):
            a.record(g.stream)
            if call == "dispatch_stash":
                d = g.dispatch_stash(0, x, idx, E)
            else:
                y = torch.empty_like(d["xd"])
                g.pop(0, [y])
            b.record(g.stream)
        g.time_copies(None, None)
        torch.cuda.synchronize()
        spans.append((a.elapsed_time(b), ca.elapsed_time(cb), a.elapsed_time(ca), cb.elapsed_time(b)))
    for whole, copy, lead, trail in spans:
        assert 0 < copy <= whole and lead >= 0 and trail >= 0
    assert torch.equal(y, d["xd"])


@pytest.mark.parametrize("padded", [False, True])
def test_fused_empty_record_matches_oracle(padded):
    """No tokens: the record is still planned (no pages), like a push of
    empty segments; then a normal record and both pops."""
    E, H, P, C = 16, 64, 8, 4
    rb = 2 * H
    page_bytes = ap.page_bytes_for(P, (rb,))
    g = ap.Pool(P, page_bytes, 40, 1, 4, E, 64, 0, fill=FILL)
    o = oracle.Pool(P, page_bytes, 40, 1, 4, E, 64, 0, keep_bytes=True, fill=FILL)
    x0 = torch.empty((0, H), dtype=torch.bfloat16, device="cuda")
    i0 = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    with torch.cuda.stream(g.stream):
        g.stream.wait_stream(torch.cuda.default_stream())
        d = g.dispatch_stash(0, x0, i0, E, C if padded else 0, padded)
    torch.cuda.synchronize()
    plan = oracle.dispatch(np.zeros((0, H), np.uint16), np.zeros((0, 2), np.int32), E, C if padded else 0, padded)
    rows = plan["rows"]
    o.push(0, [np.zeros((rows, rb), np.uint8)], rows, plan["seg_off"], plan["live"])
    for key in ("counts", "live", "seg_off"):
        assert np.array_equal(host(d[key]), plan[key]), key
    assert g.state() == o.state()
    assert g.record(0)["npages"] == o.record(0)["npages"] == 0
    T = 40
    x = inputs.normal_bf16(5, inputs.X_STREAM, (T, H))
    idx, _ = oracle.route_topk(inputs.router_logits(5, T, E), 2)
    plan = oracle.dispatch(x, idx, E, 0, False)
    o.push(0, [plan["xd"].view(np.uint8).reshape(plan["rows"], rb)], plan["rows"], plan["seg_off"], plan["live"])
    with torch.cuda.stream(g.stream):
        g.dispatch_stash(0, bf16_to_dev(x), to_dev(idx), E)
    torch.cuda.synchronize()
    assert g.state() == o.state()
    for _ in range(2):
        r = o.record(0)
        n = int(max(r["row0"] + r["nrows"])) if r["npages"] else 0
        dst_np = [np.full((max(n, 1), rb), 0x3C, np.uint8)]
        dst = to_dev(dst_np[0])
        torch.cuda.synchronize()
        g.pop(0, [dst])
        o.pop(0, dst_np, dst_np[0].shape[0])
        torch.cuda.synchronize()
        assert np.array_equal(host(dst), dst_np[0])
    assert g.state() == o.state()
    assert np.array_equal(host(g.pool), o.pool_bytes())


@pytest.mark.parametrize("T,E,fp8", [
    (512, 16, False),   # a small record: the copy kernel plans it
    (17000, 64, False),  # 266 count/rank blocks x 64 experts: the scan + plan kernel plans it
    (600, 32, True),    # E4M3 codes and scales, planned by the copy kernel
])
def test_fused_record_overflow_matches_oracle(T, E, fp8):
    """A record that needs more pages than its page table holds: the first
    max_pages_per_record pages are kept (device pages, then spill), the rest
    are dropped and AP_FLAG_RECORD_OVERFLOW is set, exactly as the oracle's
    push of the same dispatch; the pop brings back the kept pages' rows."""
    H, k, P, N, SP, maxp = 64, 4, 16, 12, 6, 15
    rb = (H, 4) if fp8 else (2 * H,)
    page_bytes = ap.page_bytes_for(P, rb)
    g = ap.Pool(P, page_bytes, N, 1, 2, E, maxp, SP, fill=FILL)
    o = oracle.Pool(P, page_bytes, N, 1, 2, E, maxp, SP, keep_bytes=True, fill=FILL)
    logits = inputs.router_logits(T + 7, T, E)
    x = inputs.normal_bf16(T + 7, inputs.X_STREAM, (T, H))
    idx, _ = oracle.route_topk(logits, k)
    plan = oracle.dispatch(x, idx, E, 0, False, fp8=fp8)
    if fp8:
        planes_o = [plan["xd"], plan["xd_scale"].view(np.uint8).reshape(-1, 4)]
    else:
        planes_o = [plan["xd"].view(np.uint8).reshape(plan["rows"], 2 * H)]
    o.push(0, planes_o, plan["rows"], plan["seg_off"], plan["live"])
    torch.cuda.synchronize()
    with torch.cuda.stream(g.stream):
        g.stream.wait_stream(torch.cuda.default_stream())
        d = g.dispatch_stash(0, bf16_to_dev(x), to_dev(idx), E, fp8=fp8)
    torch.cuda.synchronize()
    for key in ("counts", "live", "seg_off", "dest"):
        assert np.array_equal(host(d[key]), plan[key]), key
    st = g.state()
    assert st == o.state()
    assert st["flags"] & ap.FLAG_RECORD_OVERFLOW
    a, b = g.record(0), o.record(0)
    for key in ("npages", "ndev", "nspill", "nlost"):
        assert a[key] == b[key], key
    assert a["npages"] == maxp
    for key in ("page_table", "row0", "nrows"):
        assert np.array_equal(a[key], b[key]), key
    assert np.array_equal(host(g.pool), o.pool_bytes())
    assert np.array_equal(g.spill.numpy(), o.spill_bytes())
    dq = [np.full(p_.shape, 0x3C, np.uint8) for p_ in planes_o]
    dg = [to_dev(q_) for q_ in dq]
    torch.cuda.synchronize()
    g.pop(0, dg)
    o.pop(0, dq, plan["rows"])
    torch.cuda.synchronize()
    for a_, b_ in zip(dg, dq):
        assert np.array_equal(host(a_).reshape(b_.shape), b_)
    assert g.state() == o.state()

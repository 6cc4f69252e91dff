"""Full-size workloads through the whole path, against the oracle.

Each test runs one workload's schedule at its full size in the launch
configuration the benchmark times: route -> dispatch -> stash push(es) ->
pop(s) -> combine.  Integer metadata (indices, counts, offsets, destinations,
page tables, rings, counters, flags) is compared in full with the oracle,
whose page pool runs metadata-only at these sizes.  Dispatch payloads (BF16 rows,
E4M3 codes and scales) and combine outputs are compared in full; pool pages
are compared on samples, plus the size-independent property that popped rows
equal pushed rows.
"""
import numpy as np
import pytest
import torch

import oracle
from activation_paging_gb300 import inputs
from gpu_util import bf16_to_dev, bf16_to_host, host, route_tolerance, to_dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

ap = pytest.importorskip("activation_paging_gb300")


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def compare_pool(g: "ap.Pool", o: oracle.Pool, slots):
    assert g.state() == o.state()
    rg, sg = g.rings()
    ro, so = o.rings()
    assert np.array_equal(rg, ro) and np.array_equal(sg, so)
    for s in slots:
        assert g.queue_len(s) == o.queue_len(s)
        for q in range(o.queue_len(s)):
            a, b = g.record(s, q), o.record(s, q)
            for key in ("id", "npages", "ndev", "nspill", "nlost", "nseg"):
                assert a[key] == b[key], key
            for key in ("page_table", "row0", "nrows"):
                assert np.array_equal(a[key], b[key]), key


def check_pages(g: "ap.Pool", rec: dict, planes, page_bytes, plane_off, nsample=64, seed=0):
    """Sampled pages of a live record hold exactly the rows they were given;
    the bytes after the live rows of a first-use page keep the pool canary."""
    n = rec["npages"]
    pick = np.random.default_rng(seed).choice(n, min(n, nsample), replace=False)
    for ordn in pick:
        pid, r0, nr = int(rec["page_table"][ordn]), int(rec["row0"][ordn]), int(rec["nrows"][ordn])
        if pid < 0:
            continue
        if pid < g.N:
            page = g.pool[pid * page_bytes:(pid + 1) * page_bytes]
        else:
            page = g.spill[(pid - g.N) * page_bytes:(pid - g.N + 1) * page_bytes].to("cuda")
        for p, off in zip(planes, plane_off):
            rb = p.numel() // p.shape[0] * p.element_size()
            want = p.view(torch.uint8).reshape(p.shape[0], rb)[r0:r0 + nr].reshape(-1)
            assert torch.equal(page[off:off + nr * rb], want)


@pytest.mark.parametrize("fused", [False, True])
def test_qwen3_moe_two_chunks(fused):
    wl = inputs.WORKLOADS["qwen3_moe"]
    rb = wl.row_bytes
    g = ap.Pool(wl.page_tokens, wl.page_bytes, wl.num_pages, 1, 4, wl.E, wl.num_pages, fill=0xA5)
    o = oracle.Pool(wl.page_tokens, wl.page_bytes, wl.num_pages, 1, 4, wl.E, wl.num_pages, 0, keep_bytes=False)
    chunks = []
    for c in range(wl.chunks):
        logits = inputs.router_logits(c, wl.T, wl.E)
        x = inputs.normal_bf16(c, inputs.X_STREAM, (wl.T, wl.H))
        idx_o, w_o = oracle.route_topk(logits, wl.k)
        plan = oracle.dispatch(x, idx_o, wl.E, 0, False)
        idx, w = ap.route_topk(to_dev(logits), wl.k)
        if fused:
            g.stream.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(g.stream):
                d = g.dispatch_stash(0, bf16_to_dev(x), idx, wl.E)
            torch.cuda.synchronize()
        else:
            d = ap.dispatch_permute(bf16_to_dev(x), idx, wl.E)
        assert np.array_equal(host(idx), idx_o)
        assert np.all(np.abs(host(w).astype(np.float64) - w_o) <= route_tolerance(logits, idx_o, w_o))
        for key in ("counts", "live", "seg_off", "dest"):
            assert np.array_equal(host(d[key]), plan[key]), key
        assert np.array_equal(bf16_to_host(d["xd"]), plan["xd"])
        if not fused:
            g.stream.wait_stream(torch.cuda.current_stream())
            g.push(0, [d["xd"]], d["seg_off"], d["live"])
        o.push_rb(0, rb, plan["rows"], plan["seg_off"], plan["live"])
        chunks.append((d, w_o, plan))
    torch.cuda.synchronize()
    compare_pool(g, o, [0])
    assert g.overflow() == 0  # 10% headroom covers the page tails
    check_pages(g, g.record(0, 0), [chunks[0][0]["xd"]], wl.page_bytes, [0])
    for c, (d, w_o, plan) in enumerate(chunks):
        dst = torch.empty_like(d["xd"])
        g.pop(0, [dst])
        o.pop(0, None, plan["rows"], nplanes=1)
        torch.cuda.synchronize()
        assert torch.equal(dst, d["xd"])  # dropless compact: every row is live
        y = inputs.normal_bf16(c, inputs.Y_STREAM, (plan["rows"], wl.H))
        out = ap.combine_unpermute(bf16_to_dev(y), to_dev(plan["dest"]), to_dev(w_o))
        exp, _ = oracle.combine(y, plan["dest"], w_o)
        assert np.array_equal(bf16_to_host(out), exp)
    compare_pool(g, o, [0])


def test_skewed_padded_with_drops():
    wl = inputs.WORKLOADS["skewed"]
    C = wl.capacity
    logits = inputs.router_logits(0, wl.T, wl.E, wl.zipf_s, wl.zipf_beta)
    x = inputs.normal_bf16(0, inputs.X_STREAM, (wl.T, wl.H))
    idx_o, w_o = oracle.route_topk(logits, wl.k)
    plan = oracle.dispatch(x, idx_o, wl.E, C, True)
    assert plan["counts"].max() / (wl.T * wl.k / wl.E) > 7.5
    assert np.any(plan["live"] % wl.page_tokens != 0)  # tail masks exercised
    idx, w = ap.route_topk(to_dev(logits), wl.k)
    canary = torch.full((plan["rows"], wl.H), 0xA5A5 - 0x10000, dtype=torch.int16, device="cuda")
    d = ap.dispatch_permute(bf16_to_dev(x), idx, wl.E, C, True, out={"xd": canary.view(torch.bfloat16)})
    for key in ("counts", "live", "seg_off", "dest"):
        assert np.array_equal(host(d[key]), plan[key]), key
    xd_h = bf16_to_host(d["xd"])
    assert np.array_equal(xd_h, plan["xd"])
    g = ap.Pool(wl.page_tokens, wl.page_bytes, wl.num_pages, 1, 2, wl.E, wl.num_pages, fill=0xA5)
    o = oracle.Pool(wl.page_tokens, wl.page_bytes, wl.num_pages, 1, 2, wl.E, wl.num_pages, 0, keep_bytes=False)
    g.stream.wait_stream(torch.cuda.current_stream())
    g.push(0, [d["xd"]], d["seg_off"], d["live"])
    o.push_rb(0, wl.row_bytes, plan["rows"], plan["seg_off"], plan["live"])
    torch.cuda.synchronize()
    compare_pool(g, o, [0])
    check_pages(g, g.record(0, 0), [d["xd"]], wl.page_bytes, [0])
    dst = torch.full((plan["rows"], wl.H), 0x3C3C, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    g.pop(0, [dst])
    o.pop(0, None, plan["rows"], nplanes=1)
    torch.cuda.synchronize()
    compare_pool(g, o, [0])
    got = bf16_to_host(dst)
    live_rows = np.zeros(plan["rows"], bool)
    for e in range(wl.E):
        live_rows[plan["seg_off"][e]:plan["seg_off"][e] + plan["live"][e]] = True
    assert np.array_equal(got[live_rows], plan["xd"][live_rows])
    assert np.all(got[~live_rows] == 0x3C3C)  # rows past the live prefix are untouched
    # combine of the reloaded rows with identity experts (dropped pairs are
    # masked), every token compared
    out = bf16_to_host(ap.combine_unpermute(dst, to_dev(plan["dest"]), to_dev(w_o)))
    exp, _ = oracle.combine(plan["xd"], plan["dest"], w_o)
    assert np.array_equal(out, exp)


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("H", [2048, 2056])
def test_dsv2_lite_fp8_layer_stack(H, fused):
    """27 layers x 8 microbatches of E4M3 + scale records, pushed forward and
    popped with the layers reversed (per-slot FIFO across microbatches).
    Every record's codes and scales are compared with the oracle's FP8
    dispatch (the microbatch quantised once, permuted per layer).  With
    ``fused`` every push is the fused dispatch + push, as the benchmark runs
    the workload."""
    wl = inputs.WORKLOADS["dsv2_lite_fp8"].replace(H=H)
    rb = wl.row_bytes
    N = wl.num_pages
    g = ap.Pool(wl.page_tokens, wl.page_bytes, N, wl.layers, wl.microbatches, wl.E, 4096, fill=0xA5)
    o = oracle.Pool(wl.page_tokens, wl.page_bytes, N, wl.layers, wl.microbatches, wl.E, 4096, 0, keep_bytes=False)
    kept = {}
    checked = 0
    for mb in range(wl.microbatches):
        x = inputs.normal_bf16(100 + mb, inputs.X_STREAM, (wl.T, wl.H))
        x_dev = bf16_to_dev(x)
        q_o, s_o = oracle.quantize_rows_e4m3(x)
        for layer in range(wl.layers):
            logits = inputs.router_logits(1000 + mb * wl.layers + layer, wl.T, wl.E)
            idx_o, _ = oracle.route_topk(logits, wl.k)
            plan = oracle.dispatch_plan(idx_o, wl.E, 0, False)
            idx, _ = ap.route_topk(to_dev(logits), wl.k)
            g.stream.wait_stream(torch.cuda.current_stream())
            if fused:
                with torch.cuda.stream(g.stream):
                    d = g.dispatch_stash(layer, x_dev, idx, wl.E, fp8=True)
                torch.cuda.current_stream().wait_stream(g.stream)
            else:
                d = ap.dispatch_permute(x_dev, idx, wl.E, fp8=True)
            for key in ("counts", "live", "seg_off", "dest"):
                assert np.array_equal(host(d[key]), plan[key]), key
            xd = np.zeros((plan["rows"], wl.H), np.uint8)
            xs = np.zeros(plan["rows"], np.float32)
            oracle.permute_rows_fp8(q_o, s_o, plan["dest"], xd, xs)
            assert np.array_equal(host(d["xd"]), xd)
            assert np.array_equal(host(d["xd_scale"]).view(np.uint32), xs.view(np.uint32))
            checked += 1
            if not fused:
                g.stream.wait_stream(torch.cuda.current_stream())
                g.push(layer, [d["xd"], d["xd_scale"]], d["seg_off"], d["live"])
            o.push_rb(layer, rb, plan["rows"], plan["seg_off"], plan["live"])
            kept[(mb, layer)] = (d["xd"], d["xd_scale"])
    torch.cuda.synchronize()
    assert checked == wl.microbatches * wl.layers
    compare_pool(g, o, range(wl.layers))
    assert g.overflow() == 0
    rec = g.record(5, 3)
    plane1 = (wl.page_tokens * rb[0] + 15) // 16 * 16
    check_pages(g, rec, list(kept[(3, 5)]), wl.page_bytes, [0, plane1])
    for mb in range(wl.microbatches):
        for layer in reversed(range(wl.layers)):
            xd, xs = kept.pop((mb, layer))
            dq, ds = torch.empty_like(xd), torch.empty_like(xs)
            g.pop(layer, [dq, ds])
            o.pop(layer, None, xd.shape[0], nplanes=2)
            torch.cuda.synchronize()
            assert torch.equal(dq, xd) and torch.equal(ds.view(torch.int32), xs.view(torch.int32))
    compare_pool(g, o, range(wl.layers))


@pytest.mark.parametrize("fused", [False, True])
def test_spill_two_sources_interleaved(fused):
    """Pool at 60% of two live records: the second source spills to pinned host
    memory, the overflow flag stays set, reloads are byte-exact.  With
    ``fused`` every push is the fused dispatch + push call."""
    wl = inputs.WORKLOADS["spill"]
    rb = wl.row_bytes
    g = ap.Pool(wl.page_tokens, wl.page_bytes, wl.num_pages, 2, 2, wl.E, 8192, wl.spill_pages, fill=0xA5)
    o = oracle.Pool(wl.page_tokens, wl.page_bytes, wl.num_pages, 2, 2, wl.E, 8192, wl.spill_pages,
                    keep_bytes=False)
    data = {}

    def make(name, seed):
        logits = inputs.router_logits(seed, wl.T, wl.E, wl.zipf_s, wl.zipf_beta)
        x = inputs.normal_bf16(seed, inputs.X_STREAM, (wl.T, wl.H))
        idx_o, w_o = oracle.route_topk(logits, wl.k)
        plan = oracle.dispatch_plan(idx_o, wl.E, 0, False)
        idx, w = ap.route_topk(to_dev(logits), wl.k)
        d = ap.dispatch_permute(bf16_to_dev(x), idx, wl.E)
        for key in ("counts", "live", "seg_off", "dest"):
            assert np.array_equal(host(d[key]), plan[key]), key
        rows = np.random.default_rng(seed).choice(plan["rows"], 2048, replace=False)
        got = bf16_to_host(d["xd"][torch.from_numpy(rows).cuda()])
        assert np.array_equal(got, x[plan["src_tok"][rows]])
        d["x_dev"], d["idx_dev"] = bf16_to_dev(x), idx
        data[name] = (d, plan, x, w_o)

    def push(slot, name):
        d, plan, _, _ = data[name]
        g.stream.wait_stream(torch.cuda.current_stream())
        if fused:
            dest_before = d["dest"].clone()
            with torch.cuda.stream(g.stream):
                g.dispatch_stash(slot, d["x_dev"], d["idx_dev"], wl.E, out=d)
            torch.cuda.synchronize()
            assert torch.equal(d["dest"], dest_before)
        else:
            g.push(slot, [d["xd"]], d["seg_off"], d["live"])
        o.push_rb(slot, rb, plan["rows"], plan["seg_off"], plan["live"])

    def pop(slot, name):
        d, plan, x, w_o = data.pop(name)
        dst = torch.empty_like(d["xd"])
        g.pop(slot, [dst])
        o.pop(slot, None, plan["rows"], nplanes=1)
        torch.cuda.synchronize()
        assert torch.equal(dst, d["xd"])
        # identity experts: every kept row of token t holds x[t], so the
        # combine of the reloaded rows is the oracle's combine over x with
        # each pair pointing at its own token (the same products and sums, in
        # the same order); every token compared
        out = bf16_to_host(ap.combine_unpermute(dst, d["dest"], to_dev(w_o)))
        kept_pairs = plan["dest"] >= 0
        assert np.array_equal(plan["src_tok"][plan["dest"][kept_pairs]],
                              np.nonzero(kept_pairs)[0].astype(np.int32))
        own = np.where(kept_pairs, np.arange(wl.T, dtype=np.int32)[:, None], -1).astype(np.int32)
        exp, _ = oracle.combine(x, own, w_o)
        assert np.array_equal(out, exp)

    make("a0", 0)
    push(0, "a0")
    make("b0", 1)
    push(1, "b0")
    torch.cuda.synchronize()
    compare_pool(g, o, [0, 1])
    st = g.state()
    assert st["flags"] == ap.FLAG_POOL_OVERFLOW  # spilled, nothing lost
    rec_b = g.record(1, 0)
    assert rec_b["nspill"] > 0 and rec_b["nlost"] == 0
    check_pages(g, rec_b, [data["b0"][0]["xd"]], wl.page_bytes, [0], nsample=32)
    pop(0, "a0")
    make("a1", 2)
    push(0, "a1")
    pop(1, "b0")
    pop(0, "a1")
    torch.cuda.synchronize()
    compare_pool(g, o, [0, 1])
    st = g.state()
    assert st["flags"] == ap.FLAG_POOL_OVERFLOW  # sticky after every page came back
    assert st["tail"] - st["head"] == wl.num_pages

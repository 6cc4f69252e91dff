"""GPU parity: calibration and lazy pool sizing against the oracle.

torchtitan pull 5541, "AI-Generated Details": calibration parks live prefixes
before the paged buffers exist and reload restores the capacity shape.
Megatron-LM pull 7342, "Summary": the activation arena grows lazily.  A pool
starts with no device pages (its records go to pinned spill pages), the
library measures the pages the schedule holds at most, and the pool grows to
that many pages in place (an arena of reserved device addresses), with records
still queued.  After every step the device state, rings, page tables and byte
images must equal the oracle's."""
import numpy as np
import pytest
import torch

import oracle
from activation_paging_gb300 import inputs
from gpu_util import bf16_to_dev, host, to_dev
from test_gpu_stash import FILL, Twin, rows_np
from test_oracle_calibrate import held_by_hand, schedule

pytestmark = pytest.mark.gpu

ap = pytest.importorskip("activation_paging_gb300")


def test_arena_grows_in_place_and_keeps_its_bytes():
    a = ap.Arena(64 << 20)
    base0, mapped, reserved = a.info()
    assert mapped == 0 and reserved >= 64 << 20
    a.grow(1 << 20)
    v = a.view(1 << 20)
    v.fill_(0x5A)
    a.grow(24 << 20)
    base1, mapped, _ = a.info()
    assert base1 == base0 and mapped >= 24 << 20  # same addresses, more of them mapped
    w = a.view(24 << 20)
    w[1 << 20:].fill_(0x33)
    torch.cuda.synchronize()
    h = host(w)
    assert np.all(h[:1 << 20] == 0x5A) and np.all(h[1 << 20:] == 0x33)
    with pytest.raises(ap.APError):
        a.grow(reserved + 1)
    del v, w
    a.close()


@pytest.mark.parametrize("seed", [3, 4])
def test_calibrate_grow_and_rerun_match_the_oracle(seed):
    P, rb, rows, nseg = 4, (16,), 48, 6
    ops = schedule(seed)
    _, peak = held_by_hand(ops, P, 64)
    seg_off = (np.arange(nseg) * (rows // nseg)).astype(np.int32)
    # calibration: no device pages; every page parks in the spill pages
    t = Twin(P, rb, 0, S=3, R=4, segs=nseg, maxp=64, SP=peak, NMAX=peak + 8)
    pending = {s: [] for s in range(3)}
    for i, (op, s, live) in enumerate(ops):
        if op == "push":
            src = rows_np(1000 + i, rows, rb[0])
            t.push(s, [src], seg_off, live)
            pending[s].append((src, live))
        else:
            src, live = pending[s].pop(0)
            dst = t.pop(s, [(rows, rb[0])])[0]
            for o, l in zip(seg_off, live):
                assert np.array_equal(dst[o:o + l], src[o:o + l])  # the parked live rows come back
        t.check()
    st = t.g.state()
    assert st["held_high_water"] == peak and st["high_water"] == 0 and st["spill_high_water"] == peak
    assert t.g.calibrated_pages() == peak
    # grow to the measured demand, reset, run again: no overflow, every page used at the peak
    t.grow(peak)
    t.check(images=True)
    t.g.reset()
    t.o.reset()
    for i, (op, s, live) in enumerate(ops):
        if op == "push":
            t.push(s, [rows_np(2000 + i, rows, rb[0])], seg_off, live)
        else:
            t.pop(s, [(rows, rb[0])])
    t.check(images=True)
    st = t.g.state()
    assert st["flags"] == 0 and st["high_water"] == peak


def test_grow_with_records_queued_and_after_wraparound():
    P, rb = 4, (24, 4)
    t = Twin(P, rb, 10, S=2, R=8, segs=8, maxp=40, SP=12, NMAX=40)
    seg_off = np.array([0, 10, 20, 30], np.int32)
    for r in range(4):  # wrap the 10-page ring a few times
        t.push(0, [rows_np(r, 40, 24), rows_np(50 + r, 40, 4)], seg_off, [9, 10, 3, 0])
        t.pop(0, [(40, 24), (40, 4)])
    t.check(images=True)
    assert t.g.state()["head"] > 10
    t.push(0, [rows_np(7, 40, 24), rows_np(8, 40, 4)], seg_off, [10, 10, 10, 10])   # 12 pages: 10 device, 2 spill
    t.push(1, [rows_np(9, 40, 24), rows_np(10, 40, 4)], seg_off, [4, 0, 8, 1])      # 4 pages: all spill
    t.check(images=True)
    t.grow(17)
    t.check(images=True)
    t.push(1, [rows_np(11, 40, 24), rows_np(12, 40, 4)], seg_off, [10, 10, 7, 0])   # 8 pages: 7 new device, 1 spill
    t.check(images=True)
    t.grow(40)
    t.push(0, [rows_np(13, 40, 24), rows_np(14, 40, 4)], seg_off, [10, 10, 10, 10])
    t.check(images=True)
    for s in (0, 1, 1, 0):
        t.pop(s, [(40, 24), (40, 4)])
        t.check(images=True)
    assert t.g.state()["held"] == 0


def test_grow_rejects_bad_requests():
    pool = ap.Pool(4, ap.page_bytes_for(4, (16,)), 8, max_num_pages=16)
    with pytest.raises(ap.APError):
        pool.grow(4)   # cannot shrink
    with pytest.raises(ap.APError):
        pool.grow(17)  # past the growth limit
    fixed = ap.Pool(4, ap.page_bytes_for(4, (16,)), 8)
    with pytest.raises(ValueError):
        fixed.grow(9)  # created without room to grow
    rc = pool.lib.ap_pool_grow(pool.handle, 12, None, pool.stream.cuda_stream)
    assert rc == -1  # the pool memory must be given
    rc = pool.lib.ap_pool_grow(pool.handle, 12, pool.arena.info()[0], torch.cuda.Stream().cuda_stream)
    assert rc == -5  # not the paging stream


def test_fused_fp8_layer_stack_calibrated_then_grown():
    """E4M3 records of a small layer stack: calibrate with no device pages (the
    live prefixes park in pinned spill pages), grow to the measured demand,
    run again on the device: same pages, rows and bytes as the oracle, and no
    page spills the second time."""
    T, H, E, k, P, L, M = 1024, 256, 32, 4, 64, 4, 2
    rb = (H, 4)
    page_bytes = ap.page_bytes_for(P, rb)
    max_rec = T * k // P + E
    spill = L * M * max_rec
    g = ap.Pool(P, page_bytes, 0, L, M, E, max_rec, spill, fill=FILL, max_num_pages=spill)
    o = oracle.Pool(P, page_bytes, 0, L, M, E, max_rec, spill, keep_bytes=True, fill=FILL, max_num_pages=spill)
    order = [(m, l) for m in range(M) for l in range(L)] + [(m, l) for m in range(M) for l in reversed(range(L))]

    def run():
        outs = {}
        for n, (m, l) in enumerate(order):
            if n < L * M:  # forward: push
                seed = 10 * m + l
                logits = inputs.router_logits(seed, T, E)
                x = inputs.normal_bf16(seed, inputs.X_STREAM, (T, H))
                idx, _ = oracle.route_topk(logits, k)
                plan = oracle.dispatch(x, idx, E, 0, False, fp8=True)
                o.push(l, [plan["xd"], plan["xd_scale"].view(np.uint8).reshape(-1, 4)], plan["rows"],
                       plan["seg_off"], plan["live"])
                with torch.cuda.stream(g.stream):
                    g.stream.wait_stream(torch.cuda.default_stream())
                    g.dispatch_stash(l, bf16_to_dev(x), to_dev(idx), E, fp8=True)
                torch.cuda.synchronize()
                outs[(m, l)] = plan
            else:  # backward: pop, layers reversed
                plan = outs[(m, l)]
                dq = [np.full((plan["rows"], H), 0x3C, np.uint8), np.full((plan["rows"], 4), 0x3C, np.uint8)]
                dg = [to_dev(dq[0]), to_dev(dq[1])]
                torch.cuda.synchronize()
                g.pop(l, dg)
                o.pop(l, dq, plan["rows"])
                torch.cuda.synchronize()
                assert np.array_equal(host(dg[0]), dq[0]) and np.array_equal(host(dg[1]), dq[1])
                assert np.array_equal(dq[0], plan["xd"])  # dropless: every row was parked and restored
            assert g.state() == o.state()

    run()
    demand = g.calibrated_pages()
    st = g.state()
    assert st["high_water"] == 0 and st["spill_high_water"] == demand == o.state()["held_high_water"]
    g.grow(demand)
    o.grow(demand)
    g.reset()
    o.reset()
    run()  # the same routing: the measured demand is exactly enough
    st = g.state()
    assert st["flags"] == 0 and st["high_water"] == demand and st["spill_high_water"] == 0
    assert np.array_equal(host(g.pool), o.pool_bytes())

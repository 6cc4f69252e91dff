"""Pins of the oracle's calibration and lazy pool sizing.

torchtitan pull 5541, "AI-Generated Details": calibration parks the live
prefixes before the paged buffers exist, and reload restores the capacity
shape.  Megatron-LM pull 7342, "Summary": the activation arena's capacity
grows lazily.  The oracle starts a pool with no device pages (every page goes
to the spill pages, or is lost), measures the pages its queued records hold
at most, and grows the device pool by that many pages.  The pins below check
the measured demand against a count made here from the live counts alone, show
that the demand is both enough and the least that is enough, and check what a
grow must keep: queued records, their bytes, their page ids and conservation.
"""
import numpy as np
import pytest

import oracle
from activation_paging_gb300 import inputs
from test_oracle_pool import check_conservation, rand_rows

P_FILL = 0xA5


def schedule(seed, n_ops=40, S=3, nseg=6, rows=48):
    """A seeded mix of pushes and pops over S slots: (op, slot, live) tuples,
    never popping an empty slot nor overfilling one (depth 4)."""
    rng = np.random.default_rng(seed)
    depth = [0] * S
    ops = []
    for _ in range(n_ops):
        s = int(rng.integers(S))
        if depth[s] and (depth[s] == 4 or rng.random() < 0.4):
            ops.append(("pop", s, None))
            depth[s] -= 1
        else:
            live = rng.integers(0, rows // nseg + 1, nseg).astype(np.int32)
            ops.append(("push", s, live))
            depth[s] += 1
    return ops


def run(pool, ops, rb, rows, nseg, check=None):
    """Run a schedule on an oracle pool; every pop must give back the pushed
    live rows.  Returns the held-page count after every op."""
    seg_off = (np.arange(nseg) * (rows // nseg)).astype(np.int32)
    pending = {s: [] for s in range(pool.S)}
    for i, (op, s, live) in enumerate(ops):
        if op == "push":
            src = rand_rows(1000 + i, rows, rb)
            pool.push(s, [src], rows, seg_off, live)
            pending[s].append((src, live))
        else:
            src, live = pending[s].pop(0)
            dst = np.full((rows, rb), 0x3C, np.uint8)
            pool.pop(s, [dst], rows)
            if check is not None:
                check(src, live, dst, seg_off)
    return pending


def held_by_hand(ops, P, maxp):
    """Pages held by queued records after each op, and their maximum, from
    the live counts alone: a record holds sum over segments of ceil(live/P)
    pages (at most maxp)."""
    queues, held, peak, trace = {}, 0, 0, []
    for op, s, live in ops:
        q = queues.setdefault(s, [])
        if op == "push":
            n = min(int(sum((int(l) + P - 1) // P for l in live)), maxp)
            q.append(n)
            held += n
        else:
            held -= q.pop(0)
        peak = max(peak, held)
        trace.append(held)
    return trace, peak


def live_rows_back(src, live, dst, seg_off):
    for o, l in zip(seg_off, live):
        assert np.array_equal(dst[o:o + l], src[o:o + l])
        assert np.all(dst[o + l:o + (len(dst) // len(seg_off))] == 0x3C)  # rows past live untouched


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_held_pages_match_a_count_from_live_counts(seed):
    P, rb, rows, nseg = 4, 16, 48, 6
    ops = schedule(seed)
    trace, peak = held_by_hand(ops, P, 64)
    pool = oracle.Pool(P, P * rb, 64, 3, 4, nseg, 64, 0, keep_bytes=True, fill=P_FILL)
    seg_off = (np.arange(nseg) * (rows // nseg)).astype(np.int32)
    src = rand_rows(seed, rows, rb)
    for i, (op, s, live) in enumerate(ops):
        if op == "push":
            pool.push(s, [src], rows, seg_off, live)
        else:
            pool.pop(s, [np.zeros((rows, rb), np.uint8)], rows)
        assert pool.state()["held"] == trace[i]
    assert pool.state()["held_high_water"] == peak


def test_calibration_parks_live_prefixes_in_spill_and_reload_restores_them():
    P, rb, rows, nseg = 4, 16, 48, 6
    ops = schedule(7)
    _, peak = held_by_hand(ops, P, 64)
    cal = oracle.Pool(P, P * rb, 0, 3, 4, nseg, 64, peak, keep_bytes=True, fill=P_FILL, max_num_pages=peak)
    run(cal, ops, rb, rows, nseg, check=live_rows_back)
    st = cal.state()
    assert st["high_water"] == 0 and st["num_pages"] == 0  # no device page was used
    assert st["spill_high_water"] == peak == st["held_high_water"]
    assert st["flags"] == oracle.FLAG_POOL_OVERFLOW  # the (empty) device pool overflowed; nothing was lost


def test_calibration_without_spill_still_measures_the_demand():
    P, rb, rows, nseg = 4, 16, 48, 6
    ops = schedule(8)
    _, peak = held_by_hand(ops, P, 64)
    cal = oracle.Pool(P, P * rb, 0, 3, 4, nseg, 64, 0, keep_bytes=False, max_num_pages=1)
    seg_off = (np.arange(nseg) * (rows // nseg)).astype(np.int32)
    for op, s, live in ops:
        if op == "push":
            cal.push_rb(s, (rb,), rows, seg_off, live)
        else:
            cal.pop(s, None, rows)
    st = cal.state()
    assert st["held_high_water"] == peak
    assert st["flags"] == oracle.FLAG_POOL_OVERFLOW | oracle.FLAG_SPILL_OVERFLOW  # pages were lost


@pytest.mark.parametrize("seed", [3, 4, 5])
def test_grown_to_the_demand_is_enough_and_one_page_less_is_not(seed):
    P, rb, rows, nseg = 4, 16, 48, 6
    ops = schedule(seed)
    cal = oracle.Pool(P, P * rb, 0, 3, 4, nseg, 64, 0, keep_bytes=False, max_num_pages=1000)
    seg_off = (np.arange(nseg) * (rows // nseg)).astype(np.int32)
    for op, s, live in ops:
        if op == "push":
            cal.push_rb(s, (rb,), rows, seg_off, live)
        else:
            cal.pop(s, None, rows)
    demand = cal.state()["held_high_water"]
    assert demand == held_by_hand(ops, P, 64)[1]
    for n, ok in ((demand, True), (demand - 1, False)):
        pool = oracle.Pool(P, P * rb, 0, 3, 4, nseg, 64, 0, keep_bytes=True, fill=P_FILL, max_num_pages=demand)
        pool.grow(n)
        run(pool, ops, rb, rows, nseg, check=live_rows_back if ok else None)
        st = pool.state()
        if ok:
            assert st["flags"] == 0 and st["high_water"] == demand  # every page used at the peak, none short
        else:
            assert st["flags"] & oracle.FLAG_POOL_OVERFLOW


def test_grow_keeps_queued_records_their_bytes_and_page_ids():
    P, rb, rows, nseg = 4, 16, 48, 6
    seg_off = (np.arange(nseg) * 8).astype(np.int32)
    pool = oracle.Pool(P, P * rb, 10, 2, 4, nseg, 64, 20, keep_bytes=True, fill=P_FILL, max_num_pages=30)
    a = rand_rows(1, rows, rb)
    b = rand_rows(2, rows, rb)
    live_a = np.array([8, 5, 0, 8, 1, 4], np.int32)   # 2+2+0+2+1+1 = 8 pages
    live_b = np.array([8, 8, 8, 3, 0, 0], np.int32)   # 2+2+2+1 = 7 pages: 2 device, 5 spill
    pool.push(0, [a], rows, seg_off, live_a)
    pool.push(1, [b], rows, seg_off, live_b)
    ra, rb_ = pool.record(0), pool.record(1)
    assert (ra["ndev"], rb_["ndev"], rb_["nspill"]) == (8, 2, 5)
    assert all(30 <= i < 50 for i in rb_["page_table"][2:])  # spill ids start at the growth limit
    pool.pop(0, [np.zeros((rows, rb), np.uint8)], rows)        # a's 8 pages return to the ring
    st0 = pool.state()
    ring0, _ = pool.rings()
    free0 = [int(ring0[(st0["head"] + i) % 10]) for i in range(st0["tail"] - st0["head"])]
    pool.grow(25)
    st, (ring, _) = pool.state(), pool.rings()
    assert (st["head"], st["tail"], st["num_pages"]) == (0, len(free0) + 15, 25)
    assert list(ring[:len(free0)]) == free0 and list(ring[len(free0):st["tail"]]) == list(range(10, 25))
    assert np.array_equal(pool.record(1)["page_table"], rb_["page_table"])  # page ids unchanged
    check_conservation(pool)
    # a new record takes the old free pages first, then the new ones
    pool.push(0, [a], rows, seg_off, live_a)
    assert list(pool.record(0)["page_table"]) == (free0 + list(range(10, 25)))[:8]
    check_conservation(pool)
    dst = np.full((rows, rb), 0x3C, np.uint8)
    pool.pop(1, [dst], rows)  # b, pushed before the grow, comes back exactly
    live_rows_back(b, live_b, dst, seg_off)
    check_conservation(pool)


def test_grow_after_wraparound_and_errors():
    P, rb, nseg = 2, 8, 1
    pool = oracle.Pool(P, P * rb, 3, 1, 2, nseg, 8, 0, keep_bytes=True, fill=P_FILL, max_num_pages=6)
    x = rand_rows(3, 4, rb)
    for _ in range(5):  # 2 pages per record: the ring wraps
        pool.push(0, [x], 4, np.zeros(1, np.int32), np.array([4], np.int32))
        pool.pop(0, [np.zeros((4, rb), np.uint8)], 4)
    st = pool.state()
    assert st["head"] > 3
    ring, _ = pool.rings()
    order = [int(ring[(st["head"] + i) % 3]) for i in range(3)]
    pool.grow(6)
    assert list(pool.rings()[0]) == order + [3, 4, 5]
    with pytest.raises(oracle.OracleError):
        pool.grow(5)  # cannot shrink
    with pytest.raises(oracle.OracleError):
        pool.grow(7)  # past the growth limit
    with pytest.raises(oracle.OracleError):
        oracle.Pool(P, P * rb, 0, 1, 2, nseg, 8, 0)  # no device pages and no room to grow

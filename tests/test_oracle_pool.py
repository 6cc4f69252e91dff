"""Pins of the oracle's paged stash (pool, free lists, spill, FIFO, flags).

The stash has no closed form to compare with, so the pins are the invariants
the pages fix: per-slot FIFO order, payload bytes surviving push -> pop
exactly, wrapped allocation and recycling, host spill, a sticky overflow flag,
live-prefix and page-tail masks, plus page conservation and special cases.
"""
import numpy as np
import pytest

import oracle
from activation_paging_gb300 import inputs

P_FILL = 0xA5


def make_pool(P=4, rb=(16,), N=32, S=3, R=8, segs=8, maxp=64, SP=0):
    page_bytes = P * rb[0]
    if len(rb) == 2:
        page_bytes = (page_bytes + 15) // 16 * 16 + P * rb[1]
    return oracle.Pool(P, page_bytes, N, S, R, segs, maxp, SP, keep_bytes=True, fill=P_FILL), page_bytes


def rand_rows(seed, rows, rb):
    return inputs.payload_bytes(seed, (rows, rb))


def live_pages(pool):
    """Device and spill page ids held by every live record."""
    dev, sp = [], []
    for s in range(pool.S):
        for q in range(pool.queue_len(s)):
            r = pool.record(s, q)
            pt = r["page_table"]
            dev += [int(i) for i in pt if 0 <= i < pool.N]
            sp += [int(i) - pool.NMAX for i in pt if i >= pool.NMAX]
    return dev, sp


def check_conservation(pool):
    st = pool.state()
    ring, sring = pool.rings()
    free = [int(ring[(st["head"] + i) % pool.N]) for i in range(st["tail"] - st["head"])]
    dev, sp = live_pages(pool)
    assert len(set(dev)) == len(dev), "a device page is held by two records"
    assert sorted(free + dev) == list(range(pool.N))
    if pool.SP:
        sfree = [int(sring[(st["spill_head"] + i) % pool.SP]) for i in range(st["spill_tail"] - st["spill_head"])]
        assert sorted(sfree + sp) == list(range(pool.SP))


def test_fifo_and_exact_bytes_two_planes():
    pool, pb = make_pool(P=4, rb=(24, 4), N=40)
    rows = 30
    recs = []
    for i in range(3):
        a = rand_rows(10 + i, rows, 24)
        b = rand_rows(20 + i, rows, 4)
        a[0, :4] = [0xFF, 0xFF, 0xC0, 0x7F]  # NaN bit patterns survive an opaque copy
        seg_off = np.array([0, 9, 20], np.int32)
        live = np.array([7, 11, 10], np.int32)
        rid = pool.push(0, [a, b], rows, seg_off, live)
        recs.append((rid, a, b, seg_off, live))
    for rid, a, b, seg_off, live in recs:
        da = np.full_like(a, 0x11)
        db = np.full_like(b, 0x22)
        assert pool.pop(0, [da, db], rows) == rid  # FIFO
        mask = np.zeros(rows, bool)
        for o, l in zip(seg_off, live):
            mask[o:o + l] = True
        assert np.array_equal(da[mask], a[mask]) and np.array_equal(db[mask], b[mask])
        assert np.all(da[~mask] == 0x11) and np.all(db[~mask] == 0x22)  # live-prefix mask
    st = pool.state()
    assert st["flags"] == 0 and st["tail"] - st["head"] == pool.N


def test_page_contents_and_tail_canary():
    pool, pb = make_pool(P=4, rb=(8,), N=16)
    src = rand_rows(1, 20, 8)
    pool.push(1, [src], 20, np.array([0, 10], np.int32), np.array([6, 9], np.int32))
    rec = pool.record(1)
    assert rec["npages"] == 2 + 3
    img = pool.pool_bytes().reshape(pool.N, pb)
    for n in range(rec["npages"]):
        pid, r0, nr = rec["page_table"][n], rec["row0"][n], rec["nrows"][n]
        assert np.array_equal(img[pid, :nr * 8], src[r0:r0 + nr].ravel())
        assert np.all(img[pid, nr * 8:] == P_FILL)  # page-tail mask
    assert rec["nrows"].tolist() == [4, 2, 4, 4, 1]
    assert rec["row0"].tolist() == [0, 4, 10, 14, 18]


def test_single_token_pages_follow_ring_order():
    pool, _ = make_pool(P=1, rb=(4,), N=12)
    src = rand_rows(2, 10, 4)
    pool.push(0, [src], 10, np.array([0], np.int32), np.array([10], np.int32))
    assert pool.record(0)["page_table"].tolist() == list(range(10))


def test_wrap_around_and_recycling_random():
    rng = np.random.default_rng(5)
    pool, pb = make_pool(P=4, rb=(8,), N=24, S=3, R=4, segs=4)
    held = {s: [] for s in range(3)}
    total_alloc = 0
    for step in range(400):
        s = int(rng.integers(0, 3))
        if held[s] and (rng.random() < 0.5 or len(held[s]) == 4):
            rid, src, seg, live = held[s].pop(0)
            dst = np.zeros_like(src)
            assert pool.pop(s, [dst], src.shape[0]) == rid
            for o, l in zip(seg, live):
                assert np.array_equal(dst[o:o + l], src[o:o + l])
        else:
            live = rng.integers(0, 9, size=4).astype(np.int32)
            seg = (np.arange(4) * 9).astype(np.int32)
            src = rand_rows(step, 36, 8)
            st = pool.state()
            need = int(np.sum((live + 3) // 4))
            if need > st["tail"] - st["head"]:
                continue
            rid = pool.push(s, [src], 36, seg, live)
            total_alloc += need
            held[s].append((rid, src, seg, live))
        check_conservation(pool)
    assert total_alloc > 3 * pool.N  # allocation wrapped the ring several times
    assert pool.state()["flags"] == 0


def test_exactly_full_is_not_overflow():
    wl = inputs.WORKLOADS["tiny"]
    pool = oracle.Pool(wl.page_tokens, wl.page_bytes, wl.num_pages, wl.num_slots, 2, wl.E, 64, 0)
    x = inputs.normal_bf16(0, 0, (wl.T, wl.H))
    for s in range(wl.num_slots):
        pool.push(s, [x], wl.T, np.array([0], np.int32), np.array([wl.T], np.int32))
    st = pool.state()
    assert st["flags"] == 0 and st["tail"] == st["head"] and st["high_water"] == wl.num_pages
    for s in range(wl.num_slots):
        d = np.zeros_like(x)
        pool.pop(s, [d], wl.T)
        assert np.array_equal(d, x)
    check_conservation(pool)


def test_overflow_spills_and_is_sticky():
    pool, pb = make_pool(P=4, rb=(8,), N=6, S=2, SP=8)
    a = rand_rows(1, 32, 8)
    b = rand_rows(2, 32, 8)
    pool.push(0, [a], 32, np.array([0], np.int32), np.array([16], np.int32))  # 4 pages
    pool.push(1, [b], 32, np.array([0], np.int32), np.array([22], np.int32))  # 6 pages: 2 device, 4 spill
    st = pool.state()
    assert st["flags"] == oracle.FLAG_POOL_OVERFLOW
    r = pool.record(1)
    assert (r["ndev"], r["nspill"], r["nlost"]) == (2, 4, 0)
    assert all(pid >= pool.N for pid in r["page_table"][2:])
    check_conservation(pool)
    for s, src, live in ((1, b, 22), (0, a, 16)):
        d = np.zeros_like(src)
        pool.pop(s, [d], 32)
        assert np.array_equal(d[:live], src[:live])
    st = pool.state()
    assert st["flags"] == oracle.FLAG_POOL_OVERFLOW  # sticky
    assert st["spill_high_water"] == 4
    check_conservation(pool)
    pool.reset()
    assert pool.state()["flags"] == 0


def test_spill_exhausted_loses_pages():
    pool, pb = make_pool(P=4, rb=(8,), N=2, S=1, SP=1)
    a = rand_rows(3, 20, 8)
    pool.push(0, [a], 20, np.array([0], np.int32), np.array([20], np.int32))  # 5 pages: 2 dev, 1 spill, 2 lost
    st = pool.state()
    assert st["flags"] == oracle.FLAG_POOL_OVERFLOW | oracle.FLAG_SPILL_OVERFLOW
    r = pool.record(0)
    assert (r["ndev"], r["nspill"], r["nlost"]) == (2, 1, 2)
    assert r["page_table"].tolist()[3:] == [-1, -1]
    d = np.full_like(a, 0x33)
    pool.pop(0, [d], 20)
    assert np.array_equal(d[:12], a[:12])
    assert np.all(d[12:] == 0x33)  # lost pages leave their rows untouched
    check_conservation(pool)


def test_enough_pages_sets_no_flag():
    pool, _ = make_pool(P=8, rb=(4,), N=100, S=2)
    src = rand_rows(4, 64, 4)
    for s in range(2):
        for _ in range(3):
            pool.push(s, [src], 64, np.array([0, 30], np.int32), np.array([29, 34], np.int32))
    assert pool.state()["flags"] == 0


def test_bad_counts_and_record_capacity():
    pool, _ = make_pool(P=4, rb=(8,), N=16, maxp=3)
    src = rand_rows(5, 10, 8)
    pool.push(0, [src], 10, np.array([8, 0], np.int32), np.array([5, 4], np.int32))
    assert pool.state()["flags"] == oracle.FLAG_BAD_COUNT
    assert pool.record(0)["npages"] == 1  # the out-of-range segment is not paged
    pool.reset()
    big = rand_rows(6, 20, 8)
    pool.push(0, [big], 20, np.array([0], np.int32), np.array([20], np.int32))  # 5 pages > 3
    st = pool.state()
    assert st["flags"] == oracle.FLAG_RECORD_OVERFLOW
    assert pool.record(0)["npages"] == 3


def test_host_errors():
    pool, _ = make_pool(P=4, rb=(8,), N=16, S=1, R=2)
    src = rand_rows(7, 8, 8)
    seg, live = np.array([0], np.int32), np.array([8], np.int32)
    with pytest.raises(oracle.OracleError) as e:
        pool.pop(0, [np.zeros_like(src)], 8)
    assert e.value.rc == oracle.EEMPTY
    pool.push(0, [src], 8, seg, live)
    pool.push(0, [src], 8, seg, live)
    with pytest.raises(oracle.OracleError) as e:
        pool.push(0, [src], 8, seg, live)
    assert e.value.rc == oracle.EQFULL
    with pytest.raises(oracle.OracleError) as e:
        pool.push(1, [src], 8, seg, live)
    assert e.value.rc == oracle.EINVAL
    wide = rand_rows(8, 8, 16)  # 4 rows x 16 B > 32-byte page
    pool.pop(0, [np.zeros_like(src)], 8)
    with pytest.raises(oracle.OracleError) as e:
        pool.push(0, [wide], 8, seg, live)
    assert e.value.rc == oracle.EINVAL

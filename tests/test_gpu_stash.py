"""GPU parity: the paged stash against the oracle's byte-exact simulation.

After every push and pop the device state (ring counters, flags, high-water
marks), both free rings, every live record's page table and page rows, and
at the end the whole pool and spill byte images must equal the oracle's.
Popped destination bytes are compared as well, canaries included."""
import numpy as np
import pytest
import torch

import oracle
from activation_paging_gb300 import inputs
from gpu_util import host, to_dev

pytestmark = pytest.mark.gpu

ap = pytest.importorskip("activation_paging_gb300")
FILL = 0xA5


class Twin:
    """One GPU pool and one oracle pool driven with the same operations."""

    def __init__(self, P, rb, N, S=2, R=8, segs=64, maxp=None, SP=0, max_ctas=0, keep_bytes=True, NMAX=0):
        self.page_bytes = ap.page_bytes_for(P, rb)
        maxp = maxp or (max(N, NMAX) + SP)
        self.g = ap.Pool(P, self.page_bytes, N, S, R, segs, maxp, SP, max_ctas=max_ctas, fill=FILL,
                         max_num_pages=NMAX)
        self.o = oracle.Pool(P, self.page_bytes, N, S, R, segs, maxp, SP, keep_bytes=keep_bytes, fill=FILL,
                             max_num_pages=NMAX)
        self.S = S
        self.rb = rb

    def grow(self, n):
        self.g.grow(n)
        self.o.grow(n)
        torch.cuda.synchronize()

    def push(self, slot, planes_np, seg_off, live):
        dev = [to_dev(p) for p in planes_np]
        rid_g = self.g.push(slot, dev, to_dev(np.asarray(seg_off, np.int32)), to_dev(np.asarray(live, np.int32)))
        if self.o.keep_bytes:
            rid_o = self.o.push(slot, planes_np, planes_np[0].shape[0], seg_off, live)
        else:
            rid_o = self.o.push_rb(slot, [p.nbytes // max(p.shape[0], 1) for p in planes_np], planes_np[0].shape[0],
                                   seg_off, live)
        assert rid_g == rid_o
        torch.cuda.synchronize()
        return dev

    def pop(self, slot, shapes, fill=0x3C):
        dst_np = [np.full(s, fill, np.uint8) for s in shapes]
        dst = [to_dev(d) for d in dst_np]
        rid_g = self.g.pop(slot, dst)
        rid_o = self.o.pop(slot, dst_np, shapes[0][0])
        assert rid_g == rid_o
        torch.cuda.synchronize()
        for a, b in zip(dst, dst_np):
            assert np.array_equal(host(a), b)
        return dst_np

    def check(self, images=False):
        sg, so = self.g.state(), self.o.state()
        assert sg == so, (sg, so)
        # occupancy read-out: the oracle's ring counters, and the pages its queued records hold
        held_dev = sum(self.o.record(s, q)["ndev"] for s in range(self.S) for q in range(self.o.queue_len(s)))
        held_sp = sum(self.o.record(s, q)["nspill"] for s in range(self.S) for q in range(self.o.queue_len(s)))
        want = dict(pages_in_use=so["num_pages"] - (so["tail"] - so["head"]), high_water=so["high_water"],
                    spill_in_use=self.o.SP - (so["spill_tail"] - so["spill_head"]))
        assert want["pages_in_use"] == held_dev and want["spill_in_use"] == held_sp
        assert self.g.stats() == want
        assert self.g.stats(wait=False) == want  # the same figures, without touching the GPU
        rg, sgr = self.g.rings()
        ro, sro = self.o.rings()
        assert np.array_equal(rg, ro)
        assert np.array_equal(sgr, sro)
        for s in range(self.S):
            assert self.g.queue_len(s) == self.o.queue_len(s)
            for q in range(self.o.queue_len(s)):
                a, b = self.g.record(s, q), self.o.record(s, q)
                for key in ("id", "npages", "ndev", "nspill", "nlost", "nseg"):
                    assert a[key] == b[key], key
                for key in ("page_table", "row0", "nrows"):
                    assert np.array_equal(a[key], b[key]), key
        if images:
            assert np.array_equal(host(self.g.pool), self.o.pool_bytes()[:self.g.N * self.page_bytes])
            if self.g.spill is not None:
                assert np.array_equal(self.g.spill.numpy(), self.o.spill_bytes())


def rows_np(seed, rows, rb):
    return inputs.payload_bytes(seed, (rows, rb))


def test_tiny_workload_schedule():
    """Four slots each push x [256, 128] bf16 (16 pages each): the 64-page pool
    is exactly full, no overflow; then the padded dispatch output round trip."""
    wl = inputs.WORKLOADS["tiny"]
    t = Twin(wl.page_tokens, wl.row_bytes, wl.num_pages, S=wl.num_slots, R=2, segs=wl.E)
    x = inputs.normal_bf16(0, 0, (wl.T, wl.H)).view(np.uint8).reshape(wl.T, wl.H * 2)
    for s in range(wl.num_slots):
        t.push(s, [x], [0], [wl.T])
        t.check()
    st = t.g.state()
    assert st["flags"] == 0 and st["tail"] == st["head"] and st["high_water"] == wl.num_pages
    t.check(images=True)
    for s in range(wl.num_slots):
        d = t.pop(s, [x.shape])
        assert np.array_equal(d[0], x)
        t.check()
    # (ii) padded dispatch output, nseg = E, live prefixes with tails
    logits = inputs.router_logits(0, wl.T, wl.E)
    idx, _ = oracle.route_topk(logits, wl.k)
    plan = oracle.dispatch(inputs.normal_bf16(0, 0, (wl.T, wl.H)), idx, wl.E, wl.capacity, True)
    xd = plan["xd"].view(np.uint8).reshape(plan["rows"], wl.H * 2)
    t.push(0, [xd], plan["seg_off"], plan["live"])
    t.check(images=True)
    d = t.pop(0, [xd.shape])
    t.check(images=True)
    assert t.g.overflow() == 0


@pytest.mark.parametrize("max_ctas", [1, 7, 0])
def test_random_sequences_with_spill_and_overflow(max_ctas):
    """Random pushes/pops over 3 slots on a small pool with a small spill:
    wrap-around, recycling, spill, lost pages, sticky flags."""
    rng = np.random.default_rng(max_ctas + 1)
    P, rb = 8, (40,)
    t = Twin(P, rb, N=40, S=3, R=4, segs=6, SP=12, max_ctas=max_ctas)
    held = {s: [] for s in range(3)}
    for step in range(120):
        s = int(rng.integers(0, 3))
        if held[s] and (rng.random() < 0.45 or len(held[s]) == 4):
            shape = held[s].pop(0)
            t.pop(s, [shape])
        else:
            nseg = int(rng.integers(0, 7))
            cap = int(rng.integers(1, 40))
            live = rng.integers(0, cap + 1, size=nseg).astype(np.int32)
            seg_off = (np.arange(nseg) * cap).astype(np.int32)
            rows = max(nseg * cap, 1)
            src = rows_np(step, rows, rb[0])
            t.push(s, [src], seg_off, live)
            held[s].append(src.shape)
        t.check()
    t.check(images=True)
    assert t.g.state()["flags"] & ap.FLAG_POOL_OVERFLOW  # the pool was too small at some point


def test_two_planes_fp8_layout_odd_rows():
    """E4M3 rows of 2056 bytes (8-byte aligned at odd rows) + FP32 scales."""
    P, H = 128, 2056
    t = Twin(P, (H, 4), N=30, S=2, R=4, segs=8)
    rng = np.random.default_rng(3)
    held = {0: [], 1: []}
    for rep in range(3):
        live = rng.integers(0, 400, size=8).astype(np.int32)
        seg_off = (np.concatenate([[0], np.cumsum(live)[:-1]]) + 1).astype(np.int32)  # odd offsets
        rows = int(seg_off[-1] + live[-1] + 3)
        t.push(rep % 2, [rows_np(10 + rep, rows, H), rows_np(20 + rep, rows, 4)], seg_off, live)
        held[rep % 2].append(rows)
        t.check()
    t.check(images=True)
    for s in (0, 1):
        for rows in held[s]:
            t.pop(s, [(rows, H), (rows, 4)])
            t.check()


def test_spill_exhausted_lost_pages_and_reset():
    t = Twin(4, (16,), N=3, S=1, R=4, segs=2, SP=2, maxp=16)
    src = rows_np(1, 40, 16)
    t.push(0, [src], [0, 20], [13, 11])  # 4 + 3 pages: 3 device, 2 spill, 2 lost
    t.check(images=True)
    assert t.g.overflow() == ap.FLAG_POOL_OVERFLOW | ap.FLAG_SPILL_OVERFLOW
    t.pop(0, [src.shape])
    t.check(images=True)
    t.g.reset()
    t.o.reset()
    t.check()
    assert t.g.overflow() == 0


def test_bad_counts_and_record_capacity():
    t = Twin(4, (8,), N=16, S=1, R=4, segs=4, maxp=3)
    src = rows_np(2, 10, 8)
    t.push(0, [src], [8, 0, -1], [5, 8, 2])  # out-of-range and negative segments: BAD_COUNT
    t.check()
    assert t.g.overflow() & ap.FLAG_BAD_COUNT
    big = rows_np(3, 20, 8)
    t.push(0, [big], [0], [20])  # 5 pages > 3: RECORD_OVERFLOW, first 3 kept
    t.check()
    # pop into a destination of 6 rows: the page holding rows 4..7 is skipped, still recycled
    t.pop(0, [(6, 8)])
    t.check()
    t.pop(0, [(20, 8)])
    t.check(images=True)


def test_host_errors():
    pool = ap.Pool(4, 64, 8, num_slots=1, max_records_per_slot=1, max_segments=2)
    src = torch.zeros((8, 16), dtype=torch.uint8, device="cuda")
    so = torch.zeros(1, dtype=torch.int32, device="cuda")
    lv = torch.full((1,), 8, dtype=torch.int32, device="cuda")
    with pytest.raises(ap.APError) as e:
        pool.pop(0, [src])
    assert e.value.status == -2
    pool.push(0, [src], so, lv)
    with pytest.raises(ap.APError) as e:
        pool.push(0, [src], so, lv)
    assert e.value.status == -3
    pool.pop(0, [src])
    with pytest.raises(ap.APError) as e:  # 4 rows of 32 bytes do not fit a 64-byte page
        pool.push(0, [torch.zeros((8, 32), dtype=torch.uint8, device="cuda")], so, lv)
    assert e.value.status == -1
    other = torch.cuda.Stream()
    rc = pool.lib.ap_stash_push(pool.handle, 0, 1, None, None, 0, 0, None, None, None, other.cuda_stream)
    assert rc == -5  # not the paging stream


def test_max_ctas_environment(monkeypatch):
    monkeypatch.setenv("AP_STASH_MAX_CTAS", "37")
    pool = ap.Pool(4, 64, 8)
    assert pool.max_ctas == 37
    monkeypatch.delenv("AP_STASH_MAX_CTAS")
    assert ap.Pool(4, 64, 8).max_ctas == 2048
    p5 = ap.Pool(4, 64, 8, max_ctas=5)
    assert p5.max_ctas == 5
    p5.max_ctas = 64
    assert p5.max_ctas == 64
    p5.max_ctas = 0
    assert p5.max_ctas == 2048


def test_flags_device_pointer_is_the_sticky_word():
    t = Twin(4, (16,), N=2, S=1, R=2, segs=1, SP=1, maxp=8)
    t.push(0, [rows_np(1, 16, 16)], [0], [16])  # 4 pages: 2 device, 1 spill, 1 lost
    ptr = t.g.flags_device_ptr()
    assert ptr == t.g.meta.data_ptr() + 32
    word = t.g.meta[32:36].view(torch.int32)
    assert int(host(word)[0]) == t.o.state()["flags"] == ap.FLAG_POOL_OVERFLOW | ap.FLAG_SPILL_OVERFLOW


def test_many_segments_plan_in_global_memory():
    """More segments than the plan keeps in shared memory (2048): the plan
    searches its tables in global memory; same results as the oracle."""
    rng = np.random.default_rng(11)
    nseg = 3000
    live = rng.integers(0, 6, size=nseg).astype(np.int32)
    seg_off = np.concatenate([[0], np.cumsum(live)[:-1]]).astype(np.int32)
    rows = int(live.sum()) + 1
    t = Twin(4, (16,), N=1200, S=1, R=2, segs=4096, maxp=4096)
    src = rows_np(12, rows, 16)
    t.push(0, [src], seg_off, live)
    t.check(images=True)
    t.pop(0, [(rows, 16)])
    t.check(images=True)


@pytest.mark.parametrize("P,rb,N,SP", [(1, (24,), 30, 6), (512, (8,), 4, 2), (3, (20, 4), 25, 5)])
def test_page_size_extremes(P, rb, N, SP):
    """One-row pages (the page table is the ring order, row by row), pages far
    larger than any segment (every segment's tail page is mostly empty), and
    an odd page size with two planes, through wrap-around and spill."""
    rng = np.random.default_rng(P)
    t = Twin(P, rb, N=N, S=2, R=4, segs=4, SP=SP)
    held = {s: [] for s in range(2)}
    for step in range(40):
        s = int(rng.integers(0, 2))
        if held[s] and (rng.random() < 0.5 or len(held[s]) == 4):
            shapes = held[s].pop(0)
            t.pop(s, shapes)
        else:
            nseg = int(rng.integers(1, 5))
            cap = int(rng.integers(1, 9))
            live = rng.integers(0, cap + 1, size=nseg).astype(np.int32)
            seg_off = (np.arange(nseg) * cap).astype(np.int32)
            rows = nseg * cap
            planes = [rows_np(100 * step + i, rows, b) for i, b in enumerate(rb)]
            t.push(s, planes, seg_off, live)
            held[s].append([p.shape for p in planes])
            if P == 1:
                rec = t.o.record(s, len(held[s]) - 1)
                assert int(rec["npages"]) == int(live.sum())  # one page per live row
        t.check()
    t.check(images=True)


def test_pool_stats_wait_and_cached_readouts():
    """ap_pool_stats: zeros before any read-out; wait = 0 returns the last
    synchronising read-out (it does not see later pushes); wait = 1 reads the
    current occupancy, which matches the oracle."""
    P, rb = 4, (32,)
    t = Twin(P, rb, N=10, S=1, R=4, segs=4, SP=6)
    assert t.g.stats(wait=False) == dict(pages_in_use=0, high_water=0, spill_in_use=0)
    src = rows_np(5, 48, rb[0])
    t.push(0, [src], [0, 16, 32], [16, 9, 16])  # 4 + 3 + 4 = 11 pages: 10 device, 1 spill
    t.check()
    first = t.g.stats(wait=False)
    assert first == dict(pages_in_use=10, high_water=10, spill_in_use=1)
    t.pop(0, [src.shape])
    assert t.g.stats(wait=False) == first  # no read-out since the pop
    assert t.g.stats() == dict(pages_in_use=0, high_water=10, spill_in_use=0)
    t.g.reset()
    t.o.reset()
    assert t.g.stats() == dict(pages_in_use=0, high_water=0, spill_in_use=0)

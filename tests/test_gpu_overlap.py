"""GPU parity of the overlapped schedule: reloads prefetched early on the
high-priority paging stream and waited on late by the compute stream.

torchtitan pull 5541 ("AI-Generated Details": one high-priority paging stream,
reloads launched early and waited on late) and pull 5542 (early launch and
late wait across the combined graphs).  While bf16 GEMMs run on a
normal-priority compute stream, the records are popped on the paging stream;
the compute stream waits for the pops only after its own work, then consumes
the reloaded rows (a combine).  After the join every popped byte, both rings,
the state and the flags must equal the oracle's, and the consumer must have
seen the reloaded rows, not stale ones."""
import numpy as np
import pytest
import torch

import oracle
from activation_paging_gb300 import inputs
from gpu_util import bf16_to_dev, bf16_to_host, host, to_dev

pytestmark = pytest.mark.gpu

ap = pytest.importorskip("activation_paging_gb300")
FILL = 0xA5


def gemm_work(stream, n=4096, reps=6):
    """A few milliseconds of bf16 GEMMs on `stream` (the compute the reloads hide under)."""
    g = torch.Generator(device="cuda").manual_seed(1)
    a = torch.randn((n, n), device="cuda", dtype=torch.bfloat16, generator=g)
    b = torch.randn((n, n), device="cuda", dtype=torch.bfloat16, generator=g)
    c = torch.empty((n, n), device="cuda", dtype=torch.bfloat16)
    torch.cuda.synchronize()

    def run():
        with torch.cuda.stream(stream):
            for _ in range(reps):
                torch.matmul(a, b, out=c)
    return run, c


@pytest.mark.parametrize("max_ctas", [64, 0])
def test_reloads_overlapped_with_compute_match_oracle(max_ctas):
    overlapped_schedule(max_ctas, None, torch.cuda.Stream(priority=0))


@pytest.fixture
def green_streams():
    """Two disjoint SM partitions (green contexts, made by the bench-only
    libap_bench.so) and a stream in each: (small, rest, SMs of each)."""
    import ctypes
    from activation_paging_gb300 import build as cuda_build
    lib = ctypes.CDLL(cuda_build.BENCH_LIB)
    vp, ip = ctypes.c_void_p, ctypes.c_int
    lib.apb_green_split.restype = ip
    lib.apb_green_split.argtypes = [ip, ip] + [ctypes.POINTER(vp)] * 2 + [ctypes.POINTER(ip)] * 2 + \
        [ctypes.POINTER(vp)] * 2
    lib.apb_green_destroy.restype = ip
    lib.apb_green_destroy.argtypes = [vp] * 4
    s1, s2, c1, c2 = vp(), vp(), vp(), vp()
    n1, n2 = ip(), ip()
    rc = lib.apb_green_split(torch.cuda.current_device(), 16, ctypes.byref(s1), ctypes.byref(s2), ctypes.byref(n1),
                             ctypes.byref(n2), ctypes.byref(c1), ctypes.byref(c2))
    if rc < 0:
        pytest.skip(f"the driver lacks green-context entry point {-rc} of apb_green_split")
    assert rc == 0, f"green context split failed: CUDA driver error {rc}"
    yield (torch.cuda.ExternalStream(s1.value), torch.cuda.ExternalStream(s2.value), n1.value, n2.value)
    torch.cuda.synchronize()
    assert lib.apb_green_destroy(s1, s2, c1, c2) == 0


def test_reloads_on_an_sm_partition_match_oracle(green_streams):
    """The same schedule with the paging stream in a green context of at least
    16 SMs and the GEMMs in one of the other SMs: the pool runs on whatever
    stream it is given, and the bytes, rings and state still equal the
    oracle's."""
    small, rest, n_small, n_rest = green_streams
    assert n_small >= 16 and n_rest >= 1
    assert n_small + n_rest <= torch.cuda.get_device_properties(0).multi_processor_count
    overlapped_schedule(0, small, rest)


def overlapped_schedule(max_ctas, paging, compute):
    T, H, E, k, P = 2048, 1024, 64, 8, 32
    rb = 2 * H
    page_bytes = ap.page_bytes_for(P, (rb,))
    nrec = 3
    N = (T * k // P + E) * nrec
    g = ap.Pool(P, page_bytes, N, 1, 4, E, N, max_ctas=max_ctas, fill=FILL, stream=paging)
    o = oracle.Pool(P, page_bytes, N, 1, 4, E, N, 0, keep_bytes=True, fill=FILL)
    recs = []
    for r in range(nrec):
        logits = inputs.router_logits(300 + r, T, E)
        x = inputs.normal_bf16(300 + r, inputs.X_STREAM, (T, H))
        idx_o, w_o = oracle.route_topk(logits, k)
        plan = oracle.dispatch(x, idx_o, E, 0, False)
        o.push(0, [plan["xd"].view(np.uint8).reshape(plan["rows"], rb)], plan["rows"], plan["seg_off"],
               plan["live"])
        with torch.cuda.stream(g.stream):
            g.stream.wait_stream(torch.cuda.default_stream())
            g.dispatch_stash(0, bf16_to_dev(x), to_dev(idx_o), E)
        recs.append((plan, w_o))
    torch.cuda.synchronize()
    assert g.state() == o.state()

    assert g.stream.priority < compute.priority  # the paging stream has the higher priority
    run_gemm, c = gemm_work(compute)
    dst = [torch.full((plan["rows"], H), 0x3C3C, dtype=torch.int16, device="cuda").view(torch.bfloat16)
           for plan, _ in recs]
    outs = [torch.empty((T, H), dtype=torch.bfloat16, device="cuda") for _ in recs]
    start = torch.cuda.Event()
    start.record(compute)
    g.stream.wait_event(start)
    with torch.cuda.stream(g.stream):
        for d in dst:            # early launch of every reload
            g.pop(0, [d])
        done = torch.cuda.Event()
        done.record(g.stream)
    run_gemm()                   # compute that does not need the reloads
    compute.wait_event(done)     # late wait
    with torch.cuda.stream(compute):
        for (plan, w_o), d, out in zip(recs, dst, outs):
            ap.combine_unpermute(d, to_dev(plan["dest"]), to_dev(w_o), out=out, stream=compute)
    torch.cuda.synchronize()

    for (plan, w_o), d, out in zip(recs, dst, outs):
        want = np.full((plan["rows"], rb), 0x3C, np.uint8)
        o.pop(0, [want], plan["rows"])
        assert np.array_equal(bf16_to_host(d).view(np.uint8).reshape(plan["rows"], rb), want)
        exp, _ = oracle.combine(want.view(np.uint16).reshape(plan["rows"], H), plan["dest"], w_o)
        assert np.array_equal(bf16_to_host(out), exp)  # the consumer saw the reloaded rows
    assert g.state() == o.state()
    rg, sg = g.rings()
    ro, so = o.rings()
    assert np.array_equal(rg, ro) and np.array_equal(sg, so)
    assert g.overflow() == 0
    assert torch.isfinite(c.float()).all()  # the GEMMs ran to completion beside the reloads


def test_restash_during_compute_then_reload_matches_oracle():
    """The push side of the same schedule: records are stashed on the paging
    stream while the compute stream runs, the source buffers are overwritten
    on the compute stream only after it waits for the push, and the reloads
    still return the original rows."""
    T, H, E, k, P = 1536, 512, 32, 6, 16
    rb = 2 * H
    page_bytes = ap.page_bytes_for(P, (rb,))
    N = T * k // P + E
    g = ap.Pool(P, page_bytes, N, 1, 2, E, N, fill=FILL)
    o = oracle.Pool(P, page_bytes, N, 1, 2, E, N, 0, keep_bytes=True, fill=FILL)
    logits = inputs.router_logits(400, T, E)
    x = inputs.normal_bf16(400, inputs.X_STREAM, (T, H))
    idx_o, _ = oracle.route_topk(logits, k)
    plan = oracle.dispatch(x, idx_o, E, 0, False)
    d = ap.dispatch_permute(bf16_to_dev(x), to_dev(idx_o), E)
    torch.cuda.synchronize()
    compute = torch.cuda.Stream(priority=0)
    run_gemm, _ = gemm_work(compute, reps=4)
    ready = torch.cuda.Event()
    ready.record(compute)
    g.stream.wait_event(ready)
    with torch.cuda.stream(g.stream):
        g.push(0, [d["xd"]], d["seg_off"], d["live"])
        pushed = torch.cuda.Event()
        pushed.record(g.stream)
    o.push(0, [plan["xd"].view(np.uint8).reshape(plan["rows"], rb)], plan["rows"], plan["seg_off"], plan["live"])
    run_gemm()
    compute.wait_event(pushed)
    with torch.cuda.stream(compute):
        d["xd"].fill_(0)  # the dispatch buffer is reused once the stash holds the rows
    g.stream.wait_stream(compute)
    back = torch.empty_like(d["xd"])
    with torch.cuda.stream(g.stream):
        g.pop(0, [back])
    want = np.zeros((plan["rows"], rb), np.uint8)
    o.pop(0, [want], plan["rows"])
    torch.cuda.synchronize()
    assert np.array_equal(host(back.view(torch.uint8)).reshape(plan["rows"], rb), want)
    assert np.array_equal(bf16_to_host(back), plan["xd"])
    assert g.state() == o.state()

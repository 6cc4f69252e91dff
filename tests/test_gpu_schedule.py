"""The benchmark's two-stream schedules compute what the serial schedules do.

`bench.py` times the other workloads (skewed, FP8 layer stack, spill) as one
CUDA graph in which each routing runs on a second stream ahead of its fused
dispatch + push and each combine runs there after its pop, while every pool
call stays on the paging stream in schedule order.  Here two identical
schedules on reduced shapes are run side by side: one as two serial eager
passes, the other as one eager pass and one replay of its captured
two-stream graph.  Their pool states, free rings, last reloaded rows and last
combine outputs must be identical (the serial path itself is checked against
the oracle by the other tests)."""
import pytest
import torch

import bench
from activation_paging_gb300 import inputs

pytestmark = pytest.mark.gpu

ap = pytest.importorskip("activation_paging_gb300")


def reduced(name):
    if name == "dsv2_lite_fp8":
        T, layers, mbs, E = 512, 4, 3, 64
        return inputs.WORKLOADS[name].replace(T=T, layers=layers, microbatches=mbs, num_slots=layers,
                                              num_pages=layers * mbs * (T * 6 // 128 + E))
    if name == "spill":  # the pool holds 60% of two live records, the spill half of them
        T, H = 1024, 256
        return inputs.WORKLOADS[name].replace(T=T, H=H, num_pages=-(-6 * 2 * T * 8 // (10 * 64)),
                                              spill_pages=2 * T * 8 // (2 * 64))
    T = 2048  # skewed, padded with drops; capacity follows T
    wl = inputs.WORKLOADS[name].replace(T=T)
    return wl.replace(num_pages=wl.E * -(-wl.capacity // wl.page_tokens))


@pytest.mark.parametrize("name", ["dsv2_lite_fp8", "spill", "skewed"])
def test_two_stream_graph_equals_serial_schedule(name):
    wl = reduced(name)
    dev = torch.device("cuda", 0)
    serial = bench.ScheduleStep(wl, dev)
    graphed = bench.ScheduleStep(wl, dev)
    for _ in range(2):
        serial.run()
    graphed.run()
    torch.cuda.synchronize()
    for t in graphed.dst:  # the replay must write them again
        t.zero_()
    graphed.out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=graphed.stream):
        graphed.run_concurrent()
    with torch.cuda.stream(graphed.stream):
        g.replay()
    torch.cuda.synchronize()
    assert serial.pool.state() == graphed.pool.state()
    ra, sa = serial.pool.rings()
    rb, sb = graphed.pool.rings()
    assert (ra == rb).all() and (sa == sb).all()
    for a, b in zip(serial.dst, graphed.dst):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert torch.equal(serial.out.view(torch.int16), graphed.out.view(torch.int16))
    if name == "spill":
        assert serial.pool.state()["flags"] & ap.FLAG_POOL_OVERFLOW  # the reduced pool still spills
    del g

"""CPU checks of the benchmark's measurement arithmetic (no GPU).

The rates `bench.py` reports are algorithmic bytes over event time against a
measured peak; the spill workload's bound adds the host-link time of its
spilled pages to the HBM time of the rest.  These tests feed the functions
fixed event times, byte counts and link rates and compare with the numbers
worked out by hand."""
import types

import pytest

import bench


class FakeEvent:
    """Stands in for a CUDA event: elapsed_time(other) in milliseconds."""

    def __init__(self, t_ms):
        self.t = t_ms

    def elapsed_time(self, other):
        return other.t - self.t


def pair(ms):
    return FakeEvent(0.0), FakeEvent(ms)


def test_ops_table_rates_and_copy_kernel_columns():
    op_bytes = {"dispatch_stash": 600_000_000, "route_dispatch_stash": 605_000_000, "pop": 500_000_000,
                "combine": 300_000_000}
    events = {
        "route_dispatch_stash": [pair(0.11), pair(0.09)],        # mean 0.10 ms
        "route_dispatch_stash:copy": [pair(0.09), pair(0.09)],   # the copy kernel alone
        "pop": [pair(0.1)],
        "pop:copy": [pair(0.08)],
        "combine": [pair(0.05)],
    }
    ops = bench.ops_table(events, op_bytes, peak=6000.0)
    r = ops["route_dispatch_stash"]
    assert r["ms"] == pytest.approx(0.10)
    assert r["gbs"] == pytest.approx(605_000_000 / 0.10e-3 / 1e9, rel=1e-3)    # 6050 GB/s
    assert r["frac"] == pytest.approx(6050 / 6000, rel=1e-3)
    # the routing call's copy kernel moves the dispatch + push bytes, not the router's
    assert r["copy_gbs"] == pytest.approx(600_000_000 / 0.09e-3 / 1e9, rel=1e-3)
    assert ops["pop"]["copy_frac"] == pytest.approx(500_000_000 / 0.08e-3 / 1e9 / 6000, rel=1e-3)
    assert "copy_ms" not in ops["combine"]
    assert "route_dispatch_stash:copy" not in ops


def test_link_bound_adds_link_time_of_spilled_bytes(monkeypatch):
    monkeypatch.setattr(bench, "link_rates", lambda device: {"h2d": 200.0, "d2h": 100.0})
    G = 10 ** 9
    st = types.SimpleNamespace(
        bytes={"route": 1 * G, "dispatch_stash": 40 * G, "pop": 30 * G, "combine": 9 * G},
        sched=[("push", "a"), ("push", "b"), ("pop", "a"), ("pop", "b")])
    link = 20 * G                       # spilled bytes, both directions together
    bound = bench.link_bound(st, link, peak=1000.0, pass_s=0.5, device=None)
    per_pass = 2 * (1 + 40) * G + 2 * (30 + 9) * G
    assert bound["hbm_bytes"] == per_pass - link
    assert bound["link_bytes"] == {"d2h": 10 * G, "h2d": 10 * G}
    # 140 GB of HBM at 1000 GB/s, 10 GB out at 100 GB/s and 10 GB in at 200 GB/s
    expect_s = 140 / 1000 + 10 / 100 + 10 / 200
    assert bound["bound_ms"] == pytest.approx(expect_s * 1e3, rel=1e-6)
    assert bound["frac"] == pytest.approx(expect_s / 0.5, rel=1e-3)

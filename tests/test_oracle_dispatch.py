"""Pins of the oracle's dispatch (counts, capacity, stable rank, permute)."""
import json
import os

import numpy as np
import pytest

import oracle
from activation_paging_gb300 import inputs

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_examples.json")))


def brute_force_plan(idx, E, C, padded):
    """O(n^2) restatement: a pair's rank counts every earlier pair (t', j')
    routed to the same expert; kept iff dropless or rank < C."""
    T, k = idx.shape
    pairs = [(t, j) for t in range(T) for j in range(k)]
    rank = {}
    for n, (t, j) in enumerate(pairs):
        e = idx[t, j]
        rank[(t, j)] = sum(1 for (t2, j2) in pairs[:n] if idx[t2, j2] == e)
    counts = [sum(1 for (t, j) in pairs if idx[t, j] == e) for e in range(E)]
    live = [c if C <= 0 else min(c, C) for c in counts]
    if padded:
        seg = [e * C for e in range(E)]
    else:
        seg = [sum(live[:e]) for e in range(E)]
    dest = np.full((T, k), -1, np.int32)
    for (t, j), r in rank.items():
        if C <= 0 or r < C:
            dest[t, j] = seg[idx[t, j]] + r
    return np.array(counts), np.array(live), np.array(seg), dest


@pytest.mark.parametrize("C,padded", [(6, True), (6, False), (0, False), (40, True)])
def test_brute_force_tiny(C, padded):
    T, E, k = 37, 5, 2
    idx, _ = oracle.route_topk(inputs.router_logits(7, T, E), k)
    plan = oracle.dispatch_plan(idx, E, C, padded)
    counts, live, seg, dest = brute_force_plan(idx, E, C, padded)
    assert np.array_equal(plan["counts"], counts)
    assert np.array_equal(plan["live"], live)
    assert np.array_equal(plan["seg_off"], seg)
    assert np.array_equal(plan["dest"], dest)


@pytest.mark.parametrize("wl_name", ["tiny", "qwen3_moe", "skewed"])
def test_invariants(wl_name):
    wl = inputs.WORKLOADS[wl_name]
    T = min(wl.T, 4096)
    wl = wl.replace(T=T)
    idx, _ = oracle.route_topk(inputs.router_logits(0, T, wl.E, wl.zipf_s, wl.zipf_beta), wl.k)
    C = wl.capacity
    plan = oracle.dispatch_plan(idx, wl.E, C, wl.padded)
    counts, live, dest, src = plan["counts"], plan["live"], plan["dest"], plan["src_tok"]
    assert counts.sum() == T * wl.k
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=wl.E))
    kept = dest >= 0
    assert live.sum() + (~kept).sum() == T * wl.k
    assert np.array_equal(live, np.minimum(counts, C) if C > 0 else counts)
    # every token lands in k distinct experts
    assert all(len(set(r)) == wl.k for r in idx.tolist())
    # dest and src_tok are inverse on kept pairs
    t_of = np.repeat(np.arange(T), wl.k).reshape(T, wl.k)
    assert np.array_equal(src[dest[kept]], t_of[kept])
    assert len(np.unique(dest[kept])) == kept.sum()
    # rows inside each segment: token ids strictly ascending, segment inside its range
    for e in range(wl.E):
        rows = np.arange(plan["seg_off"][e], plan["seg_off"][e] + live[e])
        toks = src[rows]
        assert np.all(np.diff(toks) > 0)
        assert np.all((idx[toks] == e).any(1))
    # a dropped pair is exactly one whose arrival rank reaches the capacity
    if C > 0:
        for e in range(wl.E):
            assert (kept & (idx == e)).sum() == live[e]


def test_capacity_formula_golden():
    for key in ("tiny_capacity", "skewed_capacity"):
        g = GOLDEN[key]
        assert oracle.capacity_rows(g["capacity_factor"], g["T"], g["k"], g["E"]) == g["capacity"]
    assert inputs.WORKLOADS["tiny"].capacity == GOLDEN["tiny_capacity"]["capacity"]
    assert inputs.WORKLOADS["skewed"].capacity == GOLDEN["skewed_capacity"]["capacity"]


def test_bad_expert_index_is_skipped():
    idx = np.array([[0, 9], [1, -1], [0, 1]], np.int32)
    plan = oracle.dispatch_plan(idx, 2, 0, False)
    assert plan["status"] & oracle.FLAG_BAD_INDEX
    assert plan["dest"].tolist() == [[0, -1], [2, -1], [1, 3]]
    assert plan["counts"].tolist() == [2, 2]


def test_permute_copies_rows_and_keeps_canary():
    T, H, E, k, C = 50, 24, 4, 2, 20
    idx, _ = oracle.route_topk(inputs.router_logits(1, T, E), k)
    x = inputs.normal_bf16(1, 0, (T, H))
    plan = oracle.dispatch(x, idx, E, C, True)
    xd, dest = plan["xd"], plan["dest"]
    written = np.zeros(E * C, bool)
    for t in range(T):
        for j in range(k):
            if dest[t, j] >= 0:
                assert np.array_equal(xd[dest[t, j]], x[t])
                written[dest[t, j]] = True
    assert np.all(xd[~written].view(np.uint8) == 0xA5)


def test_empty_input():
    idx = np.zeros((0, 2), np.int32)
    plan = oracle.dispatch_plan(idx, 4, 0, False)
    assert plan["counts"].tolist() == [0] * 4
    assert plan["seg_off"].tolist() == [0] * 4

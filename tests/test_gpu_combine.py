"""GPU parity: combine / un-permute against the CPU oracle, through the C ABI.

The gate is |gpu - oracle| <= 1 BF16 ulp of the oracle value; both sides use
separately rounded single-precision multiply and add in the same order, so
the tests also record that the outputs are in fact bit-identical."""
import numpy as np
import pytest
import torch

import oracle
from activation_paging_gb300 import inputs
from gpu_util import bf16_to_dev, bf16_to_host, host, to_dev

pytestmark = pytest.mark.gpu

ap = pytest.importorskip("activation_paging_gb300")


def within_one_ulp(got: np.ndarray, exp: np.ndarray) -> bool:
    g = inputs.bf16_bits_to_f32(got).astype(np.float64)
    e = inputs.bf16_bits_to_f32(exp).astype(np.float64)
    ulp = np.where(e == 0, 2.0 ** -133, 2.0 ** (np.frexp(np.abs(e))[1] - 8))
    return bool(np.all(np.abs(g - e) <= ulp))


def combine_both(T, H, E, k, C, padded, seed=0, y_rows=None, zipf_s=0.0, beta=0.0):
    logits = inputs.router_logits(seed, T, E, zipf_s, beta)
    idx, w = oracle.route_topk(logits, k)
    plan = oracle.dispatch_plan(idx, E, C, padded)
    rows = y_rows or plan["rows"]
    y = inputs.normal_bf16(seed, inputs.Y_STREAM, (rows, H))
    exp, st_o = oracle.combine(y, plan["dest"], w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ap.combine_unpermute(bf16_to_dev(y), to_dev(plan["dest"]), to_dev(w), status=status)
    return bf16_to_host(out), exp, int(host(status)[0]), st_o


@pytest.mark.parametrize("T,H,E,k,C,padded", [
    (256, 128, 8, 2, 80, True),       # tiny workload
    (1000, 2048, 128, 8, 0, False),   # Qwen3-like shape, fewer tokens
    (1537, 264, 32, 8, 300, True),    # drops; H not a multiple of 256
    (600, 2056, 64, 6, 0, False),     # odd hidden size
    (100, 10, 8, 2, 0, False),        # H % 8 != 0: 4-byte vectors
    (100, 6, 8, 2, 0, False),         # 2 columns per lane step
    (50, 7, 8, 2, 0, False),          # odd H: scalar path
    (9, 7168, 256, 8, 0, False),      # wide rows
])
def test_combine_matches_oracle(T, H, E, k, C, padded):
    got, exp, st, st_o = combine_both(T, H, E, k, C, padded, seed=H + T)
    assert st == st_o == 0
    assert within_one_ulp(got, exp)
    assert np.array_equal(got, exp)  # same operation order: bit-identical


def test_combine_full_size_qwen3_chunk():
    wl = inputs.WORKLOADS["qwen3_moe"]
    got, exp, st, _ = combine_both(wl.T, wl.H, wl.E, wl.k, 0, False, seed=3)
    assert within_one_ulp(got, exp) and np.array_equal(got, exp)


def test_combine_full_size_spill_sampled():
    """T=32768, H=7168, top-8: oracle on a sample of 512 tokens."""
    wl = inputs.WORKLOADS["spill"]
    logits = inputs.router_logits(0, wl.T, wl.E, wl.zipf_s, wl.zipf_beta)
    idx, w = oracle.route_topk(logits, wl.k)
    plan = oracle.dispatch_plan(idx, wl.E, 0, False)
    y = inputs.normal_bf16(0, inputs.Y_STREAM, (plan["rows"], wl.H))
    out = bf16_to_host(ap.combine_unpermute(bf16_to_dev(y), to_dev(plan["dest"]), to_dev(w)))
    sample = np.random.default_rng(1).choice(wl.T, 512, replace=False)
    sample.sort()
    dest_s = plan["dest"][sample]
    rows = np.unique(dest_s[dest_s >= 0])
    y_rows = y[rows]
    remap = np.full(plan["rows"], -1, np.int64)
    remap[rows] = np.arange(rows.size)
    dest_local = np.where(dest_s >= 0, remap[np.maximum(dest_s, 0)], -1).astype(np.int32)
    exp, _ = oracle.combine(y_rows, dest_local, w[sample])
    assert np.array_equal(out[sample], exp)


def test_combine_edge_cases():
    y = inputs.normal_bf16(1, 2, (6, 64))
    dest = np.array([[-1, -1], [0, 1], [-1, 3], [5, 9]], np.int32)  # all dropped; partial; out-of-range row
    w = np.full((4, 2), 0.5, np.float32)
    exp, st_o = oracle.combine(y, dest, w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = bf16_to_host(ap.combine_unpermute(bf16_to_dev(y), to_dev(dest), to_dev(w), status=status))
    assert np.array_equal(got, exp)
    assert np.all(got[0] == 0)
    assert host(status)[0] & ap.FLAG_BAD_INDEX and st_o & oracle.FLAG_BAD_INDEX
    # k = 1, unit weights: a pure gather
    d1 = np.random.default_rng(0).permutation(6).astype(np.int32).reshape(6, 1)
    g1 = bf16_to_host(ap.combine_unpermute(bf16_to_dev(y), to_dev(d1), to_dev(np.ones((6, 1), np.float32))))
    assert np.array_equal(g1, y[d1[:, 0]])
    # no token
    e = ap.combine_unpermute(bf16_to_dev(y), torch.empty((0, 2), dtype=torch.int32, device="cuda"),
                             torch.empty((0, 2), dtype=torch.float32, device="cuda"))
    assert e.shape == (0, 64)


def test_identity_experts_return_x():
    T, H, E, k = 2048, 512, 32, 4
    logits = inputs.router_logits(4, T, E)
    x = inputs.normal_bf16(4, 0, (T, H))
    idx, w = ap.route_topk(to_dev(logits), k)
    d = ap.dispatch_permute(bf16_to_dev(x), idx, E)
    out = bf16_to_host(ap.combine_unpermute(d["xd"], d["dest"], w))
    xf, of = inputs.bf16_bits_to_f32(x).astype(np.float64), inputs.bf16_bits_to_f32(out).astype(np.float64)
    ulp = np.where(xf == 0, 2.0 ** -133, 2.0 ** (np.frexp(np.abs(xf))[1] - 8))
    assert np.all(np.abs(of - xf) <= ulp)

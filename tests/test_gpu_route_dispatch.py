"""GPU parity: router and dispatch against the CPU oracle, through the C ABI.

Indices, counts, offsets, destinations, source tokens and payload bytes are
compared bit for bit; router weights within the single-precision bound
derived in ``gpu_util.route_tolerance``."""
import numpy as np
import pytest
import torch

import oracle
from activation_paging_gb300 import inputs
from gpu_util import bf16_to_dev, bf16_to_host, host, route_tolerance, to_dev

pytestmark = pytest.mark.gpu

ap = pytest.importorskip("activation_paging_gb300")


def route_both(T, E, k, seed=0, zipf_s=0.0, beta=0.0):
    logits = inputs.router_logits(seed, T, E, zipf_s, beta)
    idx_o, w_o = oracle.route_topk(logits, k)
    idx_g, w_g = ap.route_topk(to_dev(logits), k)
    torch.cuda.synchronize()
    return logits, idx_o, w_o, host(idx_g), host(w_g)


@pytest.mark.parametrize("T,E,k", [(256, 8, 2), (1000, 64, 6), (777, 128, 8), (300, 256, 8), (129, 1024, 32),
                                   (64, 33, 5), (5, 1, 1), (3, 32, 32)])
def test_route_matches_oracle(T, E, k):
    logits, idx_o, w_o, idx_g, w_g = route_both(T, E, k, seed=T + E)
    assert np.array_equal(idx_g, idx_o)
    tol = route_tolerance(logits, idx_o, w_o)
    assert np.all(np.abs(w_g.astype(np.float64) - w_o) <= tol)


def test_route_ties_and_full_size():
    l = np.zeros((64, 128), np.float32)
    l[::2, 5] = 1.0
    idx_o, w_o = oracle.route_topk(l, 8)
    idx_g, w_g = ap.route_topk(to_dev(l), 8)
    assert np.array_equal(host(idx_g), idx_o)
    for name in ("qwen3_moe", "skewed", "spill"):
        wl = inputs.WORKLOADS[name]
        logits, idx_o, w_o, idx_g, w_g = route_both(wl.T, wl.E, wl.k, 0, wl.zipf_s, wl.zipf_beta)
        assert np.array_equal(idx_g, idx_o), name
        assert np.all(np.abs(w_g.astype(np.float64) - w_o) <= route_tolerance(logits, idx_o, w_o)), name


def dispatch_both(T, H, E, k, capacity, padded, fp8=False, seed=0, zipf_s=0.0, beta=0.0):
    logits = inputs.router_logits(seed, T, E, zipf_s, beta)
    idx, _ = oracle.route_topk(logits, k)
    x = inputs.normal_bf16(seed, inputs.X_STREAM, (T, H))
    plan = oracle.dispatch(x, idx, E, capacity, padded, fp8=fp8, fill=0xA5)
    rows = plan["rows"]
    dev = {}
    if fp8:
        dev["xd"] = torch.full((rows, H), 0xA5, dtype=torch.uint8, device="cuda")
        dev["xd_scale"] = torch.from_numpy(np.full(rows * 4, 0xA5, np.uint8).view(np.float32)).cuda()
    else:
        dev["xd"] = torch.full((rows, H), 0xA5A5 - 0x10000, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ap.dispatch_permute(bf16_to_dev(x), to_dev(idx), E, capacity, padded, fp8=fp8, out=dev, status=status)
    torch.cuda.synchronize()
    return plan, out, int(host(status)[0])


def check_plan(plan, out):
    for name in ("counts", "live", "seg_off", "dest"):
        assert np.array_equal(host(out[name]), plan[name]), name
    src_g = host(out["src_tok"])
    kept = plan["src_tok"] >= 0
    assert np.array_equal(src_g[kept], plan["src_tok"][kept])
    assert np.all(src_g[~kept] == -1)


@pytest.mark.parametrize("T,H,E,k,C,padded", [
    (256, 128, 8, 2, 80, True),        # tiny workload
    (1000, 136, 16, 4, 0, False),      # compact dropless, H not a multiple of 16 elements
    (1537, 256, 32, 8, 300, True),     # padded with drops, several rank blocks, ragged tail
    (2049, 64, 64, 6, 150, False),     # compact with a capacity
    (513, 2056, 64, 6, 0, False),      # odd hidden size
    (7, 40, 4, 3, 2, True),            # fewer tokens than a warp
    (300, 12, 8, 2, 0, False),         # rows of 24 bytes: 8-byte vectors
    (100, 7, 8, 2, 0, False),          # rows of 14 bytes: 2-byte vectors
    (3000, 32, 1024, 32, 0, False),    # the most experts and choices
    (131073, 64, 64, 8, 0, False),     # a record of 2^20 + 8 pairs (2049 rank blocks)
    (140000, 32, 128, 8, 9000, True),  # large padded record with drops
])
def test_dispatch_bf16_matches_oracle(T, H, E, k, C, padded):
    plan, out, st = dispatch_both(T, H, E, k, C, padded, seed=T)
    assert st == 0
    check_plan(plan, out)
    assert np.array_equal(bf16_to_host(out["xd"]), plan["xd"])  # every row, canary included


@pytest.mark.parametrize("T,H,E,k", [(4096, 2048, 64, 6), (4096, 2056, 64, 6), (333, 100, 8, 3), (65, 30, 4, 2),
                                     (50, 9, 4, 2), (175000, 64, 64, 6)])  # the last: a record of 1.05 M pairs
def test_dispatch_e4m3_matches_oracle(T, H, E, k):
    plan, out, st = dispatch_both(T, H, E, k, 0, False, fp8=True, seed=H)
    assert st == 0
    check_plan(plan, out)
    assert np.array_equal(host(out["xd"]), plan["xd"])
    assert np.array_equal(host(out["xd_scale"]).view(np.uint32), plan["xd_scale"].view(np.uint32))


@pytest.mark.parametrize("H", [2048, 64, 20])  # register path (8 vectors per lane, a partial vector); generic path
def test_dispatch_e4m3_special_values(H):
    """Rows with NaN (either sign), infinities, -0, BF16 denormals, all
    zeros and all NaN: the row amax ignores NaN, as the oracle's float max
    does, and every code and scale matches the oracle bit for bit."""
    T, E, k = 12, 4, 2
    x = inputs.normal_bf16(H, inputs.X_STREAM, (T, H))
    x[0, 5] = 0x7FC0                       # NaN
    x[1, 3] = 0xFFC1                       # negative NaN, other payload
    x[2, 7] = 0x7F80                       # +inf: amax inf, scale inf, codes of finite values 0
    x[3, 1] = 0xFF80                       # -inf
    x[4, :] = 0x8000                       # all -0: amax 0, scale 1
    x[5, :] = 0x0001                       # all smallest denormals
    x[6, :] = 0x7FC0                       # all NaN: amax 0
    x[7, ::3] = 0x0003                     # denormals among normal values
    x[8, :] = 0x0000
    x[9, H - 1] = 0x4F80                   # a large value (2^32) at the end of the row
    logits = inputs.router_logits(H, T, E)
    idx, _ = oracle.route_topk(logits, k)
    plan = oracle.dispatch(x, idx, E, 0, False, fp8=True, fill=0xA5)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ap.dispatch_permute(bf16_to_dev(x), to_dev(idx), E, 0, False, fp8=True, status=status)
    torch.cuda.synchronize()
    assert np.array_equal(host(out["xd"]), plan["xd"])
    assert np.array_equal(host(out["xd_scale"]).view(np.uint32), plan["xd_scale"].view(np.uint32))


def test_dispatch_full_size_skewed():
    wl = inputs.WORKLOADS["skewed"]
    plan, out, st = dispatch_both(wl.T, wl.H, wl.E, wl.k, wl.capacity, True, seed=0, zipf_s=wl.zipf_s,
                                  beta=wl.zipf_beta)
    check_plan(plan, out)
    assert (plan["dest"] < 0).sum() > 0  # the skew drops pairs
    xd = bf16_to_host(out["xd"])
    assert np.array_equal(xd, plan["xd"])


def test_dispatch_full_size_qwen3_chunk():
    wl = inputs.WORKLOADS["qwen3_moe"]
    plan, out, st = dispatch_both(wl.T, wl.H, wl.E, wl.k, 0, False, seed=1)
    check_plan(plan, out)
    assert np.array_equal(bf16_to_host(out["xd"]), plan["xd"])


def test_dispatch_bad_expert_ids_are_flagged():
    idx = np.array([[0, 9], [1, -1], [0, 1]], np.int32)
    x = inputs.normal_bf16(0, 0, (3, 16))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ap.dispatch_permute(bf16_to_dev(x), to_dev(idx), 2, 0, False, status=status)
    plan = oracle.dispatch_plan(idx, 2, 0, False)
    assert np.array_equal(host(out["dest"]), plan["dest"])
    assert host(status)[0] & ap.FLAG_BAD_INDEX


def test_dispatch_empty_input():
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    out = ap.dispatch_permute(x, idx, 8, 0, False)
    assert host(out["counts"]).tolist() == [0] * 8
    assert host(out["seg_off"]).tolist() == [0] * 8


def test_cast_e4m3_matches_oracle_encoder():
    vals = [0.0, -0.0, 448.0, -448.0, 464.0, 480.0, 1e30, -1e30, 2 ** -9, 2 ** -10, 3 * 2 ** -10, 2 ** -11,
            1e-30, 1.0, 0.0625]
    # every midpoint between neighbouring codes and its two neighbours
    mags = [oracle.e4m3_decode_one(c) for c in range(0x7F)]
    for a, b in zip(mags[:-1], mags[1:]):
        m = np.float32((a + b) / 2)
        vals += [m, np.nextafter(m, np.float32(0)), np.nextafter(m, np.float32(1e9))]
    vals = np.array(vals + [-v for v in vals], np.float32)
    rnd = np.random.default_rng(0)
    bits = rnd.integers(0, 2 ** 32, size=10_000_000, dtype=np.uint64).astype(np.uint32)
    r = bits.view(np.float32)
    r = r[np.isfinite(r)]
    scaled = (rnd.standard_normal(2_000_000) * 100).astype(np.float32)
    allv = np.concatenate([vals, r, scaled])
    got = host(ap.cast_e4m3(to_dev(allv)))
    exp = oracle.e4m3_encode(allv)
    assert np.array_equal(got, exp)


def test_cast_e4m3_matches_oracle_encoder_1e8():
    """The E4M3 conversion the FP8 dispatch uses against the oracle's own
    encoder on about 10^8 floats, in chunks: random signs, exponents and
    mantissas across and beyond the format's range (2^-14 .. 2^10), scaled
    normals, values next to every rounding midpoint, and arbitrary finite bit
    patterns."""
    rnd = np.random.default_rng(7)
    mags = [oracle.e4m3_decode_one(c) for c in range(0x7F)]
    mids = np.array([(a + b) / 2 for a, b in zip(mags[:-1], mags[1:])], np.float32)
    chunk = 1 << 24
    total = 0
    for i in range(6):
        if i < 2:  # uniform exponent over the format's range and a little beyond
            sign = rnd.integers(0, 2, chunk, dtype=np.uint32) << 31
            expo = (rnd.integers(-14, 11, chunk) + 127).astype(np.uint32) << 23
            mant = rnd.integers(0, 1 << 23, chunk, dtype=np.uint32)
            v = (sign | expo | mant).view(np.float32)
        elif i < 4:  # normals over six decades
            v = (rnd.standard_normal(chunk) * 10.0 ** rnd.uniform(-3, 3, chunk)).astype(np.float32)
        elif i == 4:  # a few float ulps around every midpoint
            m = mids[rnd.integers(0, mids.size, chunk)]
            v = (m.view(np.int32) + rnd.integers(-3, 4, chunk).astype(np.int32)).view(np.float32)
            v = np.where(rnd.integers(0, 2, chunk) == 1, -v, v).astype(np.float32)
        else:  # any finite bit pattern
            v = rnd.integers(0, 2 ** 32, chunk, dtype=np.uint64).astype(np.uint32).view(np.float32)
            v = v[np.isfinite(v)]
        got = host(ap.cast_e4m3(to_dev(v)))
        exp = oracle.e4m3_encode(v)
        assert np.array_equal(got, exp), i
        total += v.size
    assert total > 10 ** 8 * 0.99

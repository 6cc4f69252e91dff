"""GPU parity: backward of combine and of dispatch against the oracle.

dy and dx are compared bit for bit (same single roundings, same order); dw is
a float32 dot product whose summation order differs from the oracle's
(double), so it is held to the float32 summation bound
(H/32 + 6) * 2^-24 * sum_h |dout_h * y_h| plus the oracle's own rounding."""
import numpy as np
import pytest
import torch

import oracle
from activation_paging_gb300 import inputs
from gpu_util import bf16_to_dev, bf16_to_host, host, to_dev

pytestmark = pytest.mark.gpu

ap = pytest.importorskip("activation_paging_gb300")


def dw_bound(dout, y, dest):
    g = inputs.bf16_bits_to_f32(dout).astype(np.float64)
    yf = inputs.bf16_bits_to_f32(y).astype(np.float64)
    T, k = dest.shape
    H = y.shape[1]
    mag = np.zeros((T, k))
    for j in range(k):
        r = dest[:, j]
        ok = r >= 0
        mag[ok, j] = np.abs(g[ok] * yf[r[ok]]).sum(1)
    return (H / 32 + 6) * 2.0 ** -24 * mag


@pytest.mark.parametrize("T,H,E,k,C,padded", [
    (256, 128, 8, 2, 80, True),
    (1000, 2048, 128, 8, 0, False),
    (777, 264, 32, 6, 100, True),    # drops, H % 256 != 0
    (300, 30, 8, 2, 0, False),       # scalar path
    (200, 4104, 16, 4, 0, False),    # rows wider than a lane's register batch: the one-vector loop
])
def test_combine_backward_matches_oracle(T, H, E, k, C, padded):
    idx, w = oracle.route_topk(inputs.router_logits(T, T, E), k)
    plan = oracle.dispatch_plan(idx, E, C, padded)
    y = inputs.normal_bf16(T, inputs.Y_STREAM, (plan["rows"], H))
    dout = inputs.normal_bf16(T + 1, inputs.X_STREAM, (T, H))
    dy_o, dw_o, st_o = oracle.combine_backward(dout, y, plan["dest"], w, dy_fill=0xA5)
    dy_g = torch.full((plan["rows"], H), 0xA5A5 - 0x10000, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dy_g, dw_g = ap.combine_backward(bf16_to_dev(dout), bf16_to_dev(y), to_dev(plan["dest"]), to_dev(w), dy=dy_g,
                                     status=status)
    assert int(host(status)[0]) == st_o == 0
    assert np.array_equal(bf16_to_host(dy_g), dy_o)
    err = np.abs(host(dw_g).astype(np.float64) - dw_o)
    assert np.all(err <= dw_bound(dout, y, plan["dest"]) + 2.0 ** -24 * np.abs(dw_o))
    assert np.all(host(dw_g)[plan["dest"] < 0] == 0)


@pytest.mark.parametrize("T,H,E,k,C,padded", [
    (256, 128, 8, 2, 80, True),
    (1000, 2048, 128, 8, 0, False),
    (777, 264, 32, 6, 100, True),
    (300, 30, 8, 2, 0, False),
])
def test_dispatch_backward_matches_oracle(T, H, E, k, C, padded):
    idx, _ = oracle.route_topk(inputs.router_logits(T + 5, T, E), k)
    plan = oracle.dispatch_plan(idx, E, C, padded)
    dxd = inputs.normal_bf16(T, inputs.Y_STREAM, (plan["rows"], H))
    dx_o, st_o = oracle.dispatch_backward(dxd, plan["dest"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dx_g = ap.dispatch_backward(bf16_to_dev(dxd), to_dev(plan["dest"]), status=status)
    assert int(host(status)[0]) == st_o == 0
    assert np.array_equal(bf16_to_host(dx_g), dx_o)


def test_backward_through_the_stash():
    """Forward stashes the dispatched rows; the backward reloads them and
    computes the combine-weight gradient against the reloaded rows."""
    T, H, E, k, P = 2048, 512, 32, 4, 32
    logits = inputs.router_logits(9, T, E)
    x = inputs.normal_bf16(9, inputs.X_STREAM, (T, H))
    dout = inputs.normal_bf16(10, inputs.X_STREAM, (T, H))
    idx, w = ap.route_topk(to_dev(logits), k)
    d = ap.dispatch_permute(bf16_to_dev(x), idx, E)
    pool = ap.Pool(P, ap.page_bytes_for(P, (H * 2,)), int(1.2 * T * k / P) + E, 1, 2, E)
    pool.push(0, [d["xd"]], d["seg_off"], d["live"])
    back = torch.empty_like(d["xd"])
    pool.pop(0, [back])
    torch.cuda.current_stream().wait_stream(pool.stream)
    dy, dw = ap.combine_backward(bf16_to_dev(dout), back, d["dest"], w)
    dx = ap.dispatch_backward(dy, d["dest"])
    torch.cuda.synchronize()
    idx_o, w_o = oracle.route_topk(logits, k)
    plan = oracle.dispatch(x, idx_o, E, 0, False)
    dy_o, dw_o, _ = oracle.combine_backward(dout, plan["xd"], plan["dest"], host(w))
    dx_o, _ = oracle.dispatch_backward(dy_o, plan["dest"])
    assert np.array_equal(bf16_to_host(dy), dy_o)
    assert np.array_equal(bf16_to_host(dx), dx_o)
    err = np.abs(host(dw).astype(np.float64) - dw_o)
    assert np.all(err <= dw_bound(dout, plan["xd"], plan["dest"]) + 2.0 ** -24 * np.abs(dw_o))

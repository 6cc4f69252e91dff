"""Pins of the oracle's backward of combine and dispatch.

They check the oracle against the derivative of the forward definitions
(closed forms, a finite-difference-free exact gradient in rationals, unit
weights, identities), not against a restatement of the same code."""
from fractions import Fraction

import numpy as np

import oracle
from activation_paging_gb300 import inputs


def setup(T=24, H=12, E=5, k=2, C=7, padded=True, seed=0):
    idx, w = oracle.route_topk(inputs.router_logits(seed, T, E), k)
    plan = oracle.dispatch_plan(idx, E, C, padded)
    y = inputs.normal_bf16(seed, inputs.Y_STREAM, (plan["rows"], H))
    dout = inputs.normal_bf16(seed + 1, inputs.X_STREAM, (T, H))
    return plan, w, y, dout


def test_dw_is_the_exact_gradient_of_the_combined_sum():
    """f(w) = sum_t,h dout[t,h] * out_exact[t,h] is linear in w with
    df/dw[t,j] = <dout[t], y[dest(t,j)]>: compare with exact rationals."""
    plan, w, y, dout = setup()
    dy, dw, st = oracle.combine_backward(dout, y, plan["dest"], w)
    assert st == 0
    yf, gf = inputs.bf16_bits_to_f32(y), inputs.bf16_bits_to_f32(dout)
    T, k = plan["dest"].shape
    for t in range(T):
        for j in range(k):
            r = plan["dest"][t, j]
            if r < 0:
                assert dw[t, j] == 0.0
                continue
            exact = sum(Fraction(float(gf[t, h])) * Fraction(float(yf[r, h])) for h in range(y.shape[1]))
            assert dw[t, j] == np.float32(float(exact)) or abs(float(dw[t, j]) - float(exact)) <= 2 ** -24 * abs(
                float(exact))


def test_dy_rows_are_weighted_gradients():
    plan, w, y, dout = setup(padded=True)
    dy, dw, _ = oracle.combine_backward(dout, y, plan["dest"], w)
    gf = inputs.bf16_bits_to_f32(dout)
    written = np.zeros(plan["rows"], bool)
    for t, row in enumerate(plan["dest"]):
        for j, r in enumerate(row):
            if r >= 0:
                exp = inputs.f32_to_bf16_bits(np.float32(w[t, j]) * gf[t])
                assert np.array_equal(dy[r], exp)
                written[r] = True
    assert np.all(dy[~written] == 0xA5A5)  # rows no pair maps to are untouched


def test_unit_weight_gradient_is_the_output_gradient():
    T, H = 16, 20
    dout = inputs.normal_bf16(3, 0, (T, H))
    y = inputs.normal_bf16(3, 2, (T, H))
    dest = np.arange(T, dtype=np.int32).reshape(T, 1)
    dy, dw, _ = oracle.combine_backward(dout, y, dest, np.ones((T, 1), np.float32))
    assert np.array_equal(dy, dout)
    # y = dout: dw = |dout|^2
    _, dw2, _ = oracle.combine_backward(dout, dout, dest, np.ones((T, 1), np.float32))
    g = inputs.bf16_bits_to_f32(dout).astype(np.float64)
    np.testing.assert_allclose(dw2[:, 0], (g * g).sum(1), rtol=2 ** -23)


def test_dispatch_backward_adds_the_k_copies():
    """dispatch then its backward on the dispatched rows gives k * x (exact for k = 2, 4, 8)."""
    for k in (2, 4, 8):
        T, H, E = 64, 32, 16
        idx, _ = oracle.route_topk(inputs.router_logits(k, T, E), k)
        x = inputs.normal_bf16(k, 0, (T, H))
        plan = oracle.dispatch(x, idx, E, 0, False)
        dx, st = oracle.dispatch_backward(plan["xd"], plan["dest"])
        assert st == 0
        assert np.array_equal(dx, inputs.f32_to_bf16_bits(inputs.bf16_bits_to_f32(x) * np.float32(k)))


def test_dispatch_backward_skips_dropped_and_flags_bad_rows():
    dxd = inputs.normal_bf16(1, 0, (4, 8))
    dest = np.array([[-1, -1], [0, -1], [1, 2], [3, 9]], np.int32)
    dx, st = oracle.dispatch_backward(dxd, dest)
    assert st & oracle.FLAG_BAD_INDEX
    assert np.all(dx[0] == 0)
    assert np.array_equal(dx[1], dxd[0])
    assert np.array_equal(dx[3], dxd[3])
    f = inputs.bf16_bits_to_f32(dxd)
    assert np.array_equal(dx[2], inputs.f32_to_bf16_bits(f[1] + f[2]))

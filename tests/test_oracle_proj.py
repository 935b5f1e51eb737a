"""Pins of the oracle's projections around the layer (oracle.project /
oracle.forward_x): head layout, key normalisation, the gate forms, the
output projection and the bf16 rounding step, each against a construction
that reaches the same value by another route."""

import numpy as np

import gen
import oracle


def _ident_inputs(B=1, H=2, L=128, d=8, seed=3):
    rng = np.random.default_rng(seed)
    hidden = 3 * H * d
    x = gen.round_to_bf16(rng.standard_normal((B, L, hidden)).astype(np.float32))
    return x, np.eye(hidden), hidden


def test_bf16_rounding_ties_to_even():
    one = 1.0
    ulp = 2.0 ** -7  # bf16 spacing in [1, 2)
    vals = np.array([one + ulp / 2, one + 3 * ulp / 2, one + ulp / 4, one + 3 * ulp / 4, -(one + ulp / 2)])
    want = np.array([one, one + 2 * ulp, one, one + ulp, -one])
    np.testing.assert_array_equal(oracle._bf16(vals), want)


def test_identity_projection_splits_heads():
    B, H, L, d = 1, 2, 128, 8
    x, w, hidden = _ident_inputs(B, H, L, d)
    q, k, v, g, beta = oracle.project(x, w, np.zeros((hidden, 2 * H)), H)
    for h in range(H):
        np.testing.assert_array_equal(q[0, h], x[0, :, h * d:(h + 1) * d])
        np.testing.assert_array_equal(v[0, h], x[0, :, 2 * H * d + h * d:2 * H * d + (h + 1) * d])
        kr = x[0, :, H * d + h * d:H * d + (h + 1) * d].astype(np.float64)
        for t in range(L):  # one row at a time: a different route to the norm
            n = np.sqrt(sum(float(e) * float(e) for e in kr[t]))
            np.testing.assert_allclose(k[0, h, t], oracle._bf16(kr[t] / n), rtol=0, atol=0)


def test_zero_key_stays_zero():
    B, H, L, d = 1, 1, 64, 4
    x = np.zeros((B, L, 3 * d), np.float32)
    x[:, :, :d] = 1.0
    q, k, v, g, beta = oracle.project(x, np.eye(3 * d), np.zeros((3 * d, 2)), H)
    assert np.all(k == 0) and np.all(q == 1)


def test_gate_closed_forms():
    B, H, L, d = 1, 3, 64, 4
    x, w, hidden = _ident_inputs(B, H, L, d)
    b_a = np.array([0.0, 1.0, -2.0])
    a_scale = np.array([0.1, 0.5, 2.0])
    b_b = np.array([0.0, 3.0, -1.0])
    _, _, _, g, beta = oracle.project(x, w, np.zeros((hidden, 2 * H)), H, b_a=b_a, a_scale=a_scale, b_b=b_b)
    np.testing.assert_allclose(g[0, 0], -0.1 * np.log(2.0), rtol=1e-14)
    np.testing.assert_allclose(g[0, 1], -0.5 * np.log(1.0 + np.e), rtol=1e-14)
    np.testing.assert_allclose(g[0, 2], -2.0 * np.log(1.0 + np.exp(-2.0)), rtol=1e-14)
    np.testing.assert_allclose(beta[0, 0], 0.5, rtol=1e-15)
    np.testing.assert_allclose(beta[0, 1], 1.0 / (1.0 + np.exp(-3.0)), rtol=1e-14)
    # the a / b columns of W_ab reach the right heads: a one-hot column moves one gate
    w_ab = np.zeros((hidden, 2 * H))
    w_ab[0, 1] = 1.0  # a of head 1 reads x[..., 0]
    _, _, _, g2, beta2 = oracle.project(x, w, w_ab, H)
    np.testing.assert_allclose(g2[0, 1], -np.log1p(np.exp(x[0, :, 0].astype(np.float64))), rtol=1e-12)
    np.testing.assert_allclose(g2[0, 0], -np.log(2.0), rtol=1e-14)
    np.testing.assert_allclose(beta2, 0.5, rtol=1e-15)


def test_forward_x_matches_layer_on_projected_inputs():
    inp = gen.x_config_inputs("x_tiny")
    H, d = inp.H, inp.d
    r = oracle.forward_x(inp.x, inp.w_qkv, inp.w_ab, inp.w_s, inp.b_s, inp.w_g, inp.b_g, inp.w_o, H,
                         b_a=inp.b_a, a_scale=inp.a_scale, b_b=inp.b_b)
    lay = oracle.forward(r["q"], r["k"], r["v"], r["g"], r["beta"], inp.w_s, inp.b_s, inp.w_g, inp.b_g,
                         outputs=("out", "sel"))
    np.testing.assert_array_equal(r["sel"].reshape(-1), lay["sel"].reshape(-1))
    o = oracle._bf16(lay["out"]).reshape(inp.B, H, inp.L, d)
    # y[b, t] = sum over heads of o[b, h, t] W_o[h d .. h d + d)
    y = np.zeros((inp.B, inp.L, inp.hidden))
    for h in range(H):
        y += o[:, h] @ inp.w_o[h * d:(h + 1) * d].astype(np.float64)
    np.testing.assert_allclose(r["y"], oracle._bf16(y), rtol=0, atol=1e-12)


def test_output_projection_identity_keeps_head_order():
    inp = gen.x_config_inputs("x_tiny")
    H, d = inp.H, inp.d
    w_o = np.eye(H * d)
    r = oracle.forward_x(inp.x, inp.w_qkv, inp.w_ab, inp.w_s, inp.b_s, inp.w_g, inp.b_g, w_o, H,
                         b_a=inp.b_a, a_scale=inp.a_scale, b_b=inp.b_b)
    for h in range(H):
        np.testing.assert_array_equal(r["y"][:, :, h * d:(h + 1) * d], r["o"][:, h])

"""Pins of the oracle's per-branch RMSNorm and query-gated merge.

Neural Attention Search Linear, technical summary, "Kernmechanismen" item 4
(readings CONV-8, CONV-9).
"""

import numpy as np

import gen
import oracle


def _inp(seed=5):
    return gen.make_inputs(1, 2, 256, 32, dtype="f32", seed=seed, pattern="random", frac=0.5)


def _rms(x):
    return np.sqrt((x ** 2).mean(-1))


def test_saturated_gate_selects_one_branch():
    inp = _inp()
    eps = 1e-6
    inp.b_g[:] = -1e4
    lin = oracle.forward_inputs(inp, eps=eps, outputs=("o_l", "out"))
    inp.b_g[:] = 1e4
    soft = oracle.forward_inputs(inp, eps=eps, outputs=("o_s", "out"))
    for r, key in ((lin, "o_l"), (soft, "o_s")):
        x, y = r[key], r["out"]
        ms = (x ** 2).mean(-1)
        # same direction as the branch output ...
        cos = (x * y).sum(-1) / (np.linalg.norm(x, axis=-1) * np.linalg.norm(y, axis=-1))
        np.testing.assert_allclose(cos, 1.0, rtol=1e-12)
        # ... with RMS sqrt(ms / (ms + eps))
        np.testing.assert_allclose(_rms(y), np.sqrt(ms / (ms + eps)), rtol=1e-12)


def test_merge_is_gate_weighted_combination():
    inp = _inp(6)
    b_g = inp.b_g.copy()
    inp.b_g[:] = -1e4
    n_lin = oracle.forward_inputs(inp, outputs=("out",))["out"]
    inp.b_g[:] = 1e4
    n_soft = oracle.forward_inputs(inp, outputs=("out",))["out"]
    inp.b_g[:] = b_g
    out = oracle.forward_inputs(inp, outputs=("out",))["out"]
    z = np.einsum("hld,hd->hl", inp.q[0].astype(np.float64), inp.w_g.astype(np.float64)) + b_g[:, None]
    w = 1.0 / (1.0 + np.exp(-z))
    np.testing.assert_allclose(out, w[..., None] * n_soft + (1 - w[..., None]) * n_lin,
                               rtol=1e-12, atol=1e-13)
    assert 0.3 < w.min() and w.max() < 0.7  # the gate is genuinely mixing here


def test_scale_invariance_of_the_norm():
    inp = _inp(7)
    ref = oracle.forward_inputs(inp, eps=0.0, outputs=("out",))["out"]
    inp.v *= 8.0
    big = oracle.forward_inputs(inp, eps=0.0, outputs=("out",))["out"]
    np.testing.assert_allclose(big, ref, rtol=1e-12, atol=1e-12)


def test_norm_weights_scale_each_branch():
    inp = _inp(8)
    inp.b_g[:] = 1e4
    one = oracle.forward_inputs(inp, outputs=("out",))["out"]
    w = np.linspace(0.5, 2.0, 32).astype(np.float32)
    two = oracle.forward_inputs(inp, norm_w_soft=w, norm_w_lin=np.zeros(32, np.float32),
                                outputs=("out",))["out"]
    np.testing.assert_allclose(two, one * w, rtol=1e-14)

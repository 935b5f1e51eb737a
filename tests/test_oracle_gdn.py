"""Pins of the oracle's Gated DeltaNet branch with pseudo-update and rollback.

Neural Attention Search Linear, technical summary, "Kernmechanismen" item 3:
both hidden states are pseudo-updated for every chunk; for the operation not
selected the state returns to the chunk start (readings CONV-1, CONV-5).
"""

import math

import numpy as np
import pytest

import gen
import oracle
from derivations import gdn_chunkwise, gdn_product_form


def _run(inp, sel, scale=0.0, outputs=("o_l", "state")):
    return oracle.forward_inputs(inp, sel_in=sel, scale=scale, outputs=outputs)


@pytest.mark.parametrize("C,L,d,seed", [(4, 16, 4, 0), (3, 13, 3, 1), (5, 20, 6, 2)])
def test_product_form(C, L, d, seed):
    inp = gen.make_inputs(1, 2, L, d, dtype="f32", seed=seed, chunk=C, pattern="scored")
    rng = np.random.default_rng(seed)
    sel = rng.integers(0, 2, size=(1, 2, inp.n_chunks)).astype(np.uint8)
    r = _run(inp, sel)
    for h in range(2):
        o, S = gdn_product_form(inp.q[0, h], inp.k[0, h], inp.v[0, h], inp.g[0, h],
                                inp.beta[0, h], sel[0, h], C, 1 / math.sqrt(d))
        np.testing.assert_allclose(r["o_l"][h], o, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(r["state"][h], S, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("pattern", ["random", "all", "none", "alternating"])
def test_chunkwise_closed_form(pattern):
    inp = gen.make_inputs(1, 2, 256, 32, dtype="f32", seed=3, pattern=pattern, frac=0.5)
    sel, _ = oracle.select_inputs(inp)
    r = _run(inp, sel)
    for h in range(2):
        o, S = gdn_chunkwise(inp.q[0, h], inp.k[0, h], inp.v[0, h], inp.g[0, h],
                             inp.beta[0, h], sel[0, h], 64, 1 / math.sqrt(32))
        np.testing.assert_allclose(r["o_l"][h], o, rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(r["state"][h], S, rtol=1e-9, atol=1e-11)


def test_zero_write_strength_keeps_state_empty():
    inp = gen.make_inputs(1, 2, 128, 16, dtype="f32", seed=1, pattern="none")
    inp.beta[:] = 0.0
    r = oracle.forward_inputs(inp, outputs=("o_l", "state", "out", "o_s"))
    assert np.all(r["o_l"] == 0) and np.all(r["state"] == 0)
    # RMSNorm(0) = 0, so the merged output is the gated softmax part alone
    assert np.isfinite(r["out"]).all()


def test_delta_rule_exact_retrieval():
    # a = 1, beta = 1, orthonormal keys inside a chunk: writing v_t under key
    # k_t overwrites that slot, so S_t k_t = v_t; with q_t = k_t the readout
    # is scale * v_t.  (Delta rule without gate: DeltaNet, the a = 1 case.)
    C, d = 8, 8
    inp = gen.make_inputs(1, 1, 32, d, dtype="f32", seed=2, chunk=C, pattern="scored")
    eye = np.eye(d, dtype=np.float32)
    inp.k[0, 0] = eye[np.arange(32) % d]
    inp.q[0, 0] = inp.k[0, 0]
    inp.g[:] = 0.0
    inp.beta[:] = 1.0
    r = _run(inp, np.ones((1, 1, 4), np.uint8), scale=0.5)
    np.testing.assert_allclose(r["o_l"][0], 0.5 * inp.v[0, 0], rtol=1e-14, atol=1e-14)


def test_scalar_closed_form():
    # d = 1, k = 1, constant a, beta, v = 1, all chunks linear:
    # S_t = r S_{t-1} + beta with r = a (1 - beta) -> S_t = beta (1 - r^t) / (1 - r).
    C, L = 4, 16
    inp = gen.make_inputs(1, 1, L, 1, dtype="f32", seed=0, chunk=C, pattern="scored")
    inp.k[:] = 1.0
    inp.q[:] = 1.0
    inp.v[:] = 1.0
    a, beta = 0.9, 0.25
    inp.g[:] = np.float32(math.log(a))
    inp.beta[:] = beta
    a32 = float(np.float32(math.exp(np.float32(math.log(a)))))  # decay as the oracle sees it
    a64 = math.exp(float(np.float32(math.log(a))))
    r = _run(inp, np.ones((1, 1, 4), np.uint8), scale=1.0)
    rr = a64 * (1 - beta)
    t = np.arange(1, L + 1)
    np.testing.assert_allclose(r["o_l"][0, :, 0], beta * (1 - rr ** t) / (1 - rr), rtol=1e-13)
    del a32


def test_rollback_metamorphic():
    C = 64
    inp = gen.make_inputs(1, 1, 512, 16, dtype="f32", seed=8, pattern="scored")
    sel = np.array([[[1, 0, 1, 0, 0, 1, 1, 0]]], np.uint8)
    base = oracle.forward_inputs(inp, sel_in=sel, outputs=("o_s", "o_l", "state"))
    # perturb V inside softmax chunk 3: Gated DeltaNet output moves only inside chunk 3
    inp2 = gen.make_inputs(1, 1, 512, 16, dtype="f32", seed=8, pattern="scored")
    inp2.v[0, 0, 3 * C:4 * C] += 1.0
    p = oracle.forward_inputs(inp2, sel_in=sel, outputs=("o_s", "o_l", "state"))
    diff = np.abs(p["o_l"] - base["o_l"]).max(axis=-1)[0]
    assert diff[3 * C:4 * C].max() > 1e-3
    assert diff[: 3 * C].max() == 0 and diff[4 * C:].max() == 0
    np.testing.assert_array_equal(p["state"], base["state"])
    # ... while the softmax output of every later token sees the change
    ds = np.abs(p["o_s"] - base["o_s"]).max(axis=-1)[0]
    assert ds[4 * C:].min() > 0 and ds[: 3 * C].max() == 0
    # perturb V inside linear chunk 2: softmax output moves only inside chunk 2
    inp3 = gen.make_inputs(1, 1, 512, 16, dtype="f32", seed=8, pattern="scored")
    inp3.v[0, 0, 2 * C:3 * C] += 1.0
    p3 = oracle.forward_inputs(inp3, sel_in=sel, outputs=("o_s", "o_l"))
    ds = np.abs(p3["o_s"] - base["o_s"]).max(axis=-1)[0]
    assert ds[2 * C:3 * C].max() > 1e-3
    assert ds[: 2 * C].max() == 0 and ds[3 * C:].max() == 0


def test_last_chunk_rollback_in_final_state():
    inp = gen.make_inputs(1, 1, 192, 8, dtype="f32", seed=4, pattern="scored")
    sel_a = np.array([[[1, 1, 0]]], np.uint8)
    sel_b = np.array([[[1, 1, 1]]], np.uint8)
    two = gen.make_inputs(1, 1, 128, 8, dtype="f32", seed=4, pattern="scored")
    ra = _run(inp, sel_a)
    rb = _run(inp, sel_b)
    r2 = _run(two, np.array([[[1, 1]]], np.uint8))
    np.testing.assert_array_equal(ra["state"], r2["state"])
    assert np.abs(rb["state"] - ra["state"]).max() > 1e-3

"""Pins of the oracle's softmax branch.

Neural Attention Search Linear, technical summary, "Kernmechanismen" item 3:
the retained KV set keeps a chunk's tokens only when that chunk chose softmax;
inside a chunk both correlations are computed (reading CONV-4).
"""

import math

import numpy as np
import pytest
import torch

import gen
import oracle
from derivations import dense_masked_attention


def _run(inp, sel, scale=0.0, **kw):
    return oracle.forward_inputs(inp, sel_in=sel, scale=scale, outputs=("o_s",), **kw)["o_s"]


def _rand_sel(rng, B, H, N):
    return rng.integers(0, 2, size=(B, H, N)).astype(np.uint8)


@pytest.mark.parametrize("C,L,d", [(4, 24, 8), (64, 320, 16), (8, 37, 5)])
def test_dense_masked_attention(C, L, d):
    inp = gen.make_inputs(2, 2, L, d, dtype="f32", seed=7, chunk=C, pattern="scored")
    rng = np.random.default_rng(1)
    N = inp.n_chunks
    sel = _rand_sel(rng, 2, 2, N)
    o = _run(inp, sel)
    scale = 1 / math.sqrt(d)
    for f in range(4):
        b, h = divmod(f, 2)
        ref = dense_masked_attention(inp.q[b, h], inp.k[b, h], inp.v[b, h], sel[b, h], C, scale)
        np.testing.assert_allclose(o[f], ref, rtol=1e-12, atol=1e-12)


def test_all_softmax_is_causal_attention():
    inp = gen.make_inputs(1, 3, 256, 32, dtype="f32", seed=2, pattern="scored")
    sel = np.zeros((1, 3, 4), np.uint8)
    o = _run(inp, sel)
    q, k, v = (torch.from_numpy(x.astype(np.float64)) for x in (inp.q, inp.k, inp.v))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    np.testing.assert_allclose(o.reshape(1, 3, 256, 32), ref.numpy(), rtol=1e-10, atol=1e-12)


def test_all_linear_is_blockwise_causal_attention():
    C = 64
    inp = gen.make_inputs(1, 2, 256, 16, dtype="f32", seed=4, pattern="scored")
    sel = np.ones((1, 2, 4), np.uint8)
    o = _run(inp, sel).reshape(1, 2, 256, 16)
    for c in range(4):
        sl = slice(c * C, (c + 1) * C)
        q, k, v = (torch.from_numpy(x[:, :, sl].astype(np.float64)) for x in (inp.q, inp.k, inp.v))
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
        np.testing.assert_allclose(o[:, :, sl], ref.numpy(), rtol=1e-10, atol=1e-12)


def test_zero_query_averages_the_kv_set():
    C = 4
    inp = gen.make_inputs(1, 1, 16, 6, dtype="f32", seed=9, chunk=C, pattern="scored")
    inp.q[:] = 0.0
    sel = np.array([[[0, 1, 0, 1]]], np.uint8)
    o = _run(inp, sel)[0]
    v = inp.v[0, 0].astype(np.float64)
    # chunk 2, token 9: earlier softmax chunk 0 (tokens 0-3) plus tokens 8, 9
    np.testing.assert_allclose(o[9], v[[0, 1, 2, 3, 8, 9]].mean(0), rtol=1e-13)
    # chunk 3, token 15: chunks 0 and 2 retained, chunk 1 and 3's own prefix
    np.testing.assert_allclose(o[15], v[[0, 1, 2, 3, 8, 9, 10, 11, 12, 13, 14, 15]].mean(0), rtol=1e-13)
    # chunk 1, token 6: chunk 0 plus 4, 5, 6
    np.testing.assert_allclose(o[6], v[[0, 1, 2, 3, 4, 5, 6]].mean(0), rtol=1e-13)


def test_first_token_returns_its_value():
    inp = gen.make_inputs(1, 2, 128, 8, dtype="f32", seed=1, pattern="scored")
    o = _run(inp, np.zeros((1, 2, 2), np.uint8))
    np.testing.assert_allclose(o[:, 0], inp.v[0, :, 0], rtol=0, atol=0)


def test_rows_subset_matches_full():
    inp = gen.make_inputs(1, 2, 256, 16, dtype="f32", seed=6, pattern="random", frac=0.5)
    full = oracle.forward_inputs(inp, outputs=("o_s", "out"))
    rows = np.zeros(256, bool)
    rows[[0, 63, 64, 200, 255]] = True
    part = oracle.forward_inputs(inp, rows=rows, outputs=("o_s", "out"))
    for key in ("o_s", "out"):
        np.testing.assert_array_equal(part[key][:, rows], full[key][:, rows])
        assert np.isnan(part[key][:, ~rows]).all()

"""Pins of the decode-mode oracle (oracle.Decoder): stepped over a whole
sequence from an empty state it must reproduce the prefill oracle
(oracle.forward, itself pinned by the other test files) token by token --
selection, both branch outputs, the merged output and the final state --
including the all-softmax and all-linear extremes and a mid-chunk stop."""

import numpy as np
import pytest

import gen
import oracle


def _decode_all(inp, steps=None):
    dec = oracle.Decoder(inp.B, inp.H, inp.d, inp.d, inp.w_s, inp.b_s, inp.w_g, inp.b_g, chunk=inp.chunk)
    L = inp.L if steps is None else steps
    outs = {n: np.zeros((inp.B, inp.H, L, inp.d)) for n in ("out", "o_s", "o_l")}
    for t in range(L):
        o, s, l = dec.step(inp.q[:, :, t], inp.k[:, :, t], inp.v[:, :, t], inp.g[:, :, t], inp.beta[:, :, t])
        outs["out"][:, :, t], outs["o_s"][:, :, t], outs["o_l"][:, :, t] = o, s, l
    return dec, outs


@pytest.mark.parametrize("pattern,frac", [("random", 0.5), ("all", 1.0), ("none", 0.0)])
def test_decode_reproduces_prefill(pattern, frac):
    inp = gen.make_inputs(1, 2, 256, 16, dtype="f32", seed=21, pattern=pattern, frac=frac)
    dec, outs = _decode_all(inp)
    ref = oracle.forward_inputs(inp)
    assert np.array_equal(np.array(dec.sel, np.uint8).reshape(ref["sel"].shape), ref["sel"])
    for n in ("o_s", "o_l", "out"):
        np.testing.assert_allclose(outs[n].reshape(ref[n].shape), ref[n], rtol=0, atol=1e-10)
    np.testing.assert_allclose(dec.S.reshape(ref["state"].shape), ref["state"], rtol=0, atol=1e-10)


def test_retained_keys_are_the_softmax_chunks():
    inp = gen.make_inputs(1, 1, 320, 8, dtype="f32", seed=22, pattern="random", frac=0.5)
    dec, _ = _decode_all(inp)
    sel = np.array(dec.sel[0][0])
    want = np.concatenate([inp.k[0, 0, 64 * c:64 * (c + 1)] for c in np.flatnonzero(sel == 0)] or [np.zeros((0, 8))])
    np.testing.assert_array_equal(dec.kv_k[0][0], want)


def test_mid_chunk_prefix_matches_prefill_prefix():
    # the first 100 tokens: outputs equal the prefill of the whole sequence there
    # (the prefill is causal and selections of chunks 0 and 1 do not depend on later tokens)
    inp = gen.make_inputs(1, 2, 192, 16, dtype="f32", seed=23, pattern="random", frac=0.5)
    dec, outs = _decode_all(inp, steps=100)
    ref = oracle.forward_inputs(inp)
    for n in ("o_s", "o_l", "out"):
        np.testing.assert_allclose(outs[n].reshape(1 * 2, 100, 16), ref[n][:, :100], rtol=0, atol=1e-10)
    assert len(dec.sel[0][0]) == 1  # only chunk 0 is complete

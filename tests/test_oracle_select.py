"""Pins of the oracle's chunk selection (Attention Score Layer + argmax).

Neural Attention Search Linear, technical summary, "Kernmechanismen" item 1:
mean pooling per chunk, one linear score per operation, highest score wins.
"""

import numpy as np
import pytest

import gen
import oracle


def _empty(B, H, L, d):
    z = np.zeros((B, H, L, d), np.float32)
    return z.copy(), z.copy()


def test_hand_built_means_and_one_hot_rows():
    # Two chunks of 64 tokens; q[:, 1] and k[:, 2] vary around known means.
    B, H, L, d, C = 1, 1, 128, 4, 64
    q, k = _empty(B, H, L, d)
    wiggle = 0.01 * (np.arange(64) - 31.5)  # sums to zero over a chunk
    q[0, 0, :64, 1] = 0.3 + wiggle
    k[0, 0, :64, 2] = 0.5 - wiggle
    q[0, 0, 64:, 1] = 0.7 + wiggle
    k[0, 0, 64:, 2] = 0.2 + wiggle
    w_s = np.zeros((H, 2, 2 * d), np.float32)
    w_s[0, 0, 1] = 1.0  # softmax score reads mean q[1]
    w_s[0, 1, d + 2] = 1.0  # linear score reads mean k[2]
    sel, scores = oracle.select(q, k, w_s, None, chunk=C)
    np.testing.assert_allclose(scores[0, 0], [[0.3, 0.5], [0.7, 0.2]], atol=1e-6)
    assert sel[0, 0].tolist() == [1, 0]


def test_bias_and_tie():
    q, k = _empty(1, 2, 192, 8)
    w_s = np.zeros((2, 2, 16), np.float32)
    b_s = np.array([[0.0, 0.0], [-1.0, 0.0]], np.float32)
    sel, _ = oracle.select(q, k, w_s, b_s, chunk=64)
    assert sel[0, 0].tolist() == [0, 0, 0]  # exact tie -> softmax (row 0)
    assert sel[0, 1].tolist() == [1, 1, 1]


@pytest.mark.parametrize("pattern", ["all", "none"])
def test_forced_patterns(pattern):
    inp = gen.make_inputs(2, 3, 256, 32, seed=5, pattern=pattern)
    sel, _ = oracle.select_inputs(inp)
    assert np.all(sel == (0 if pattern == "all" else 1))


@pytest.mark.parametrize("pattern", ["random", "alternating", "first", "last", "bursts"])
def test_planted_chunks_are_recovered(pattern):
    # The generator plants a direction into the queries of chosen chunks; the
    # score layer must select exactly those, with a wide margin.
    kw = dict(frac=0.3)
    if pattern == "bursts":
        kw = dict(bursts=(2, 5, 4))
    inp = gen.make_inputs(2, 3, 64 * 40, 64, seed=11, pattern=pattern, **kw)
    sel, scores = oracle.select_inputs(inp)
    assert np.array_equal(sel == 0, inp.planted)
    assert np.abs(scores[..., 0] - scores[..., 1]).min() > 0.1


def test_permutation_inside_chunk_is_invisible():
    inp = gen.make_inputs(1, 2, 256, 32, seed=3, pattern="scored")
    sel, scores = oracle.select_inputs(inp)
    rng = np.random.default_rng(0)
    perm = np.concatenate([c * 64 + rng.permutation(64) for c in range(4)])
    sel2, scores2 = oracle.select(inp.q[:, :, perm], inp.k[:, :, perm], inp.w_s, inp.b_s)
    assert np.array_equal(sel, sel2)
    np.testing.assert_allclose(scores, scores2, rtol=0, atol=1e-12)


def test_partial_last_chunk_pools_its_own_tokens():
    # L = 80: the second chunk has 16 tokens, all with q[0] = 2 -> mean 2.
    q, k = _empty(1, 1, 80, 4)
    q[0, 0, 64:, 0] = 2.0
    w_s = np.zeros((1, 2, 8), np.float32)
    w_s[0, 0, 0] = 1.0
    sel, scores = oracle.select(q, k, w_s, np.array([[0.0, 1.0]], np.float32))
    np.testing.assert_allclose(scores[0, 0, :, 0], [0.0, 2.0])
    assert sel[0, 0].tolist() == [1, 0]


def test_workload_margins():
    # Every workload keeps score margins >= 1e-3 (so fp32 and fp64 argmax agree).
    for name in ("tiny", "small"):
        inp = gen.config_inputs(name)
        sel, scores = oracle.select_inputs(inp)
        assert np.abs(scores[..., 0] - scores[..., 1]).min() >= 1e-3, name
        if inp.planted is not None:
            assert np.array_equal(sel == 0, inp.planted)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["l8192", "sweep0", "sweep12", "sweep50", "sweep100", "long", "l128k"])
def test_large_workload_margins(name):
    """The full-size workloads too: every argmax margin >= 1e-3 on the rounded
    inputs (fp64 scores), and the score layer recovers the planted chunks
    exactly (or the forced all / none pattern)."""
    inp = gen.config_inputs(name)
    sel, scores = oracle.select_inputs(inp)
    margin = np.abs(scores[..., 0] - scores[..., 1]).min()
    assert margin >= 1e-3, (name, margin)
    if inp.planted is not None:
        assert np.array_equal(sel == 0, inp.planted), name
    if name == "sweep0":
        assert (sel == 1).all()
    if name == "sweep100":
        assert (sel == 0).all()

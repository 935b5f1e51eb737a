"""Pins of the NHA oracle (oracle/nha.py, reading CONV-16).

"Native Hybrid Attention for Efficient Sequence Modeling", section
"2. Methodologie", "Kernprincipes": the window size w is the layer's only
knob; w = 0 gives a pure linear RNN (the Gated Slot Attention slots alone)
and w = sequence length gives full attention.  Each pin computes the expected
values another way than the oracle's token loop: a library routine, the
closed (unrolled) form of the slot recurrence, or a closed form of a special
gate value.
"""

import numpy as np
import pytest
import torch

import gen
from oracle import nha


def _inputs(B=1, H=2, L=96, d=8, m=5, window=16, seed=0):
    return gen.make_nha_inputs(B, H, L, d, m, window, dtype="f32", seed=seed)


def _unrolled_slots(k, v, la):
    """K~_t, V~_t after the write of token t, for every t, from the closed form
    K~_t[s] = sum_{j <= t} (1 - alpha_j[s]) prod_{j < i <= t} alpha_i[s] k_j
    (dense [L, L, m] weights; no recurrence)."""
    k, v, la = (np.asarray(x, np.float64) for x in (k, v, la))
    L = k.shape[0]
    cum = np.cumsum(la, axis=0)  # [L, m], inclusive
    dec = np.exp(cum[:, None, :] - cum[None, :, :])  # [t, j, m] = prod_{j < i <= t} alpha_i
    w = (1.0 - np.exp(la))[None, :, :] * dec * np.tril(np.ones((L, L)))[:, :, None]
    return np.einsum("tjs,jd->tsd", w, k), np.einsum("tjs,jd->tsd", w, v)


def _dense(q, k, v, la, window, scale=None):
    """Every query's full score row [slots (if any were written); window keys],
    built from the unrolled slot memory and a dense window mask."""
    q = np.asarray(q, np.float64)
    L, d = q.shape
    sc = scale or 1.0 / np.sqrt(d)
    Ks, Vs = _unrolled_slots(k, v, la)
    o = np.zeros((L, d))
    for t in range(L):
        keep = np.array([t - window < j <= t for j in range(L)])
        z = [sc * (np.asarray(k, np.float64)[keep] @ q[t])]
        vals = [np.asarray(v, np.float64)[keep]]
        if t - window >= 0:
            z.insert(0, sc * (Ks[t - window] @ q[t]))
            vals.insert(0, Vs[t - window])
        z = np.concatenate(z)
        p = np.exp(z - z.max())
        o[t] = (p / p.sum()) @ np.concatenate(vals, 0)
    return o


def test_full_window_is_causal_attention():
    inp = _inputs(L=80, d=16, window=80)
    o = nha.forward_inputs(inp)
    for w in (80, 81, 1 << 20):  # any w >= L
        np.testing.assert_allclose(nha.forward_inputs(inp, window=w), o, rtol=0, atol=0)
    q, k, v = (torch.from_numpy(x.astype(np.float64)) for x in (inp.q, inp.k, inp.v))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_window_zero_is_gated_slot_attention():
    """w = 0: o_t = V~_t^T softmax(scale K~_t q_t) with the slots after token t's
    own write (Gated Slot Attention), from the unrolled slot memory."""
    inp = _inputs(L=64, d=8, m=6, window=0, seed=3)
    o = nha.forward_inputs(inp)
    for b in range(inp.B):
        for h in range(inp.H):
            Ks, Vs = _unrolled_slots(inp.k[b, h], inp.v[b, h], inp.log_alpha[b, h])
            q = inp.q[b, h].astype(np.float64)
            z = np.einsum("tsd,td->ts", Ks, q) / np.sqrt(inp.d)
            p = np.exp(z - z.max(1, keepdims=True))
            p /= p.sum(1, keepdims=True)
            ref = np.einsum("ts,tsd->td", p, Vs)
            np.testing.assert_allclose(o[b, h], ref, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("window", [1, 7, 16, 63])
def test_hybrid_windows_match_dense_scores(window):
    inp = _inputs(L=72, d=8, m=4, window=window, seed=window)
    o = nha.forward_inputs(inp)
    for b in range(inp.B):
        for h in range(inp.H):
            ref = _dense(inp.q[b, h], inp.k[b, h], inp.v[b, h], inp.log_alpha[b, h], window)
            np.testing.assert_allclose(o[b, h], ref, rtol=1e-10, atol=1e-12)


def test_gates_at_one_keep_the_slots_empty():
    """alpha = 1 writes nothing: the slots stay zero but, once the first token
    has left the window, take part with logit 0 and value 0 (m entries):
    o_t = sum_win e^{z_j} v_j / (sum_win e^{z_j} + m) for t >= w."""
    inp = _inputs(L=48, d=8, m=5, window=10, seed=5)
    inp.log_alpha[:] = 0.0
    o = nha.forward_inputs(inp)
    sc = 1 / np.sqrt(inp.d)
    q, k, v = (x[0, 0].astype(np.float64) for x in (inp.q, inp.k, inp.v))
    for t in range(inp.L):
        lo = max(0, t - 10 + 1)
        e = np.exp(sc * (k[lo:t + 1] @ q[t]))
        den = e.sum() + (inp.m if t >= 10 else 0)
        np.testing.assert_allclose(o[0, 0, t], (e @ v[lo:t + 1]) / den, rtol=1e-12, atol=1e-14)


def test_gates_at_zero_hold_the_token_that_left_the_window():
    """alpha -> 0: every slot holds exactly the token that just left the
    window (t - w), an m-fold copy of it next to the window."""
    inp = _inputs(L=40, d=8, m=3, window=6, seed=6)
    inp.log_alpha[:] = -80.0  # alpha = e^-80: 1 - alpha == 1 in float64
    o = nha.forward_inputs(inp)
    sc = 1 / np.sqrt(inp.d)
    q, k, v = (x[0, 1].astype(np.float64) for x in (inp.q, inp.k, inp.v))
    for t in range(inp.L):
        idx = list(range(max(0, t - 6 + 1), t + 1))
        wts = np.ones(len(idx))
        if t - 6 >= 0:
            idx = [t - 6] + idx
            wts = np.concatenate([[inp.m], wts])
        z = sc * (k[idx] @ q[t])
        p = wts * np.exp(z - z.max())
        np.testing.assert_allclose(o[0, 1, t], (p / p.sum()) @ v[idx], rtol=1e-11, atol=1e-13)

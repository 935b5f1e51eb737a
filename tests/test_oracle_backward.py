"""Pins of the backward oracle (oracle/backward.py), on the CPU.

Its forward is a second, independent write-out of "Neural Attention Search
Linear (NAtS-L)", technical summary, "Kernmechanismen" items 1, 3 and 4
(dense masked attention instead of the retained-list loop), so it is first
checked against the pinned C++ oracle; its gradients are then checked against
central finite differences of that forward in float64, input by input, and
against closed forms of the merge, the saturated gate and the all-softmax
case (causal attention, a library routine).
"""

import numpy as np
import pytest
import torch

import gen
import oracle
from oracle import backward as ob


def _case(seed, L=192, d=16, H=2, sel=None, norm=True):
    inp = gen.make_inputs(1, H, L, d, dtype="f32", seed=seed, pattern="random", frac=0.5)
    rng = np.random.default_rng(seed + 1000)
    N = L // 64
    if sel is None:
        sel = rng.integers(0, 2, size=(1, H, N)).astype(np.uint8)
        sel[0, 0, :3] = [0, 1, 0][:N]  # a retained chunk, a rolled-forward one, a rollback
    nws = (1 + 0.2 * rng.standard_normal(d)) if norm else None
    nwl = (1 + 0.2 * rng.standard_normal(d)) if norm else None
    b_g = 0.3 * rng.standard_normal(H)
    dout = rng.standard_normal((1, H, L, d))
    return inp, np.asarray(sel, np.uint8), nws, nwl, b_g, dout


def _args(inp, nws, nwl, b_g):
    return dict(q=inp.q, k=inp.k, v=inp.v, g=inp.g, beta=inp.beta, w_g=inp.w_g, b_g=b_g,
                norm_w_soft=nws, norm_w_lin=nwl)


def test_forward_matches_the_cpp_oracle():
    inp, sel, nws, nwl, b_g, dout = _case(301)
    ref = oracle.forward(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.w_s, inp.b_s, inp.w_g,
                         b_g.astype(np.float32), norm_w_soft=None if nws is None else nws.astype(np.float32),
                         norm_w_lin=None if nwl is None else nwl.astype(np.float32), sel_in=sel,
                         outputs=("o_s", "o_l", "out"))
    # the same values in float64 (the weights as the C++ side reads them: float32)
    x = ob.inputs64(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.w_g, b_g.astype(np.float32),
                    nws.astype(np.float32), nwl.astype(np.float32))
    with torch.no_grad():
        out, o_s, o_l = ob.forward_torch(x, sel)
    for name, mine in (("o_s", o_s), ("o_l", o_l), ("out", out)):
        np.testing.assert_allclose(mine.numpy().reshape(ref[name].shape), ref[name], rtol=1e-9, atol=1e-11,
                                   err_msg=name)


@pytest.mark.parametrize("name", ob.NAMES)
def test_gradient_matches_finite_differences(name):
    inp, sel, nws, nwl, b_g, dout = _case(302)
    args = _args(inp, nws, nwl, b_g)
    grads = ob.backward(sel=sel, dout=dout, **args)
    x = ob.inputs64(**args)
    rng = np.random.default_rng(7 + ob.NAMES.index(name))
    direction = torch.tensor(rng.standard_normal(tuple(x[name].shape)))
    R = torch.tensor(dout)

    def f(step):
        y = {n: t.detach().clone() for n, t in x.items()}
        y[name] = y[name] + step * direction
        with torch.no_grad():
            return float((ob.forward_torch(y, sel)[0] * R).sum())

    h = 1e-5
    fd = (f(h) - f(-h)) / (2 * h)
    an = float((torch.tensor(grads["d" + name]) * direction).sum())
    assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_gate_bias_gradient_closed_form():
    # d<R, out>/d b_g[h] = sum_t w (1 - w) <R_t, N_s,t - N_l,t>
    inp, sel, nws, nwl, b_g, dout = _case(303)
    res = ob.backward(sel=sel, dout=dout, **_args(inp, nws, nwl, b_g))
    eps = 1e-6
    rms = lambda o: o / np.sqrt((o * o).mean(-1, keepdims=True) + eps)
    ns, nl = rms(res["o_s"]) * nws, rms(res["o_l"]) * nwl
    z = np.einsum("bhld,hd->bhl", inp.q.astype(np.float64), inp.w_g.astype(np.float64)) + b_g[None, :, None]
    w = 1 / (1 + np.exp(-z))
    expect = (w * (1 - w) * (dout * (ns - nl)).sum(-1)).sum(axis=(0, 2))
    np.testing.assert_allclose(res["db_g"], expect, rtol=1e-10)
    # and the RMSNorm weights: sum_t (w R_t) * o_s,t / rms(o_s,t)
    np.testing.assert_allclose(res["dnorm_w_soft"], (w[..., None] * dout * rms(res["o_s"])).sum(axis=(0, 1, 2)),
                               rtol=1e-10)


def test_saturated_gate_cuts_the_other_branch():
    inp, sel, nws, nwl, b_g, dout = _case(304)
    soft = ob.backward(sel=sel, dout=dout, **_args(inp, nws, nwl, np.full(2, 1e4)))
    for n in ("dg", "dbeta", "dnorm_w_lin"):  # only the Gated DeltaNet side reads these
        assert np.all(soft[n] == 0.0), n
    lin = ob.backward(sel=sel, dout=dout, **_args(inp, nws, nwl, np.full(2, -1e4)))
    assert np.all(lin["dnorm_w_soft"] == 0.0)


def test_all_softmax_is_causal_attention_through_the_norm():
    # every chunk softmax and w = 1: out = RMSNorm(causal SDPA(q, k, v)) * w_soft
    inp, _, nws, nwl, _, dout = _case(305)
    sel = np.zeros((1, 2, 3), np.uint8)
    res = ob.backward(sel=sel, dout=dout, **_args(inp, nws, nwl, np.full(2, 1e4)))
    q, k, v = (torch.tensor(a.astype(np.float64), requires_grad=True) for a in (inp.q, inp.k, inp.v))
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    y = o * torch.rsqrt((o * o).mean(-1, keepdim=True) + 1e-6) * torch.tensor(nws)
    gq, gk, gv = torch.autograd.grad(y, [q, k, v], torch.tensor(dout))
    for name, ref in (("dq", gq), ("dk", gk), ("dv", gv)):
        np.testing.assert_allclose(res[name], ref.numpy(), rtol=1e-9, atol=1e-11, err_msg=name)


def test_last_chunk_from_its_prefix_and_state():
    # the gradients of the last chunk's tokens (dq, dk, dv, dg, dbeta) depend on
    # the earlier tokens only through the retained keys / values before it and
    # the Gated DeltaNet state at its start: the backward of the last chunk
    # alone, given those as constants, equals the whole sequence's there
    inp, sel, nws, nwl, b_g, dout = _case(306, L=256, d=16)
    whole = ob.backward(sel=sel, dout=dout, **_args(inp, nws, nwl, b_g))
    L0, d = 192, 16
    state0 = oracle.forward(inp.q[:, :, :L0], inp.k[:, :, :L0], inp.v[:, :, :L0], inp.g[:, :, :L0],
                            inp.beta[:, :, :L0], inp.w_s, inp.b_s, inp.w_g, b_g.astype(np.float32),
                            sel_in=sel[:, :, :3], outputs=("state",))["state"].reshape(1, 2, d, d)
    sl = slice(L0, 256)
    n_prefix = set()
    for h in range(2):
        keep = np.flatnonzero(np.repeat(sel[0, h, :3] == 0, 64))  # retained tokens before the last chunk
        n_prefix.add(len(keep))
        one = lambda a: a[:, h:h + 1, sl]
        local = ob.backward(one(inp.q), one(inp.k), one(inp.v), one(inp.g), one(inp.beta), inp.w_g[h:h + 1],
                            b_g[h:h + 1], sel[:, h:h + 1, 3:], one(dout), norm_w_soft=nws, norm_w_lin=nwl,
                            prefix_k=inp.k[:, h:h + 1, keep], prefix_v=inp.v[:, h:h + 1, keep],
                            state0=state0[:, h:h + 1])
        for n in ("dq", "dk", "dv", "dg", "dbeta"):
            np.testing.assert_allclose(local[n], whole[n][:, h:h + 1, sl], rtol=1e-9, atol=1e-11, err_msg=n)
    assert len(n_prefix) == 2  # the heads retain different prefixes


# ---- BWD-2: the straight-through surrogate of the score layer (opt-in) ----

def _st_case(seed, L=192, d=16, H=2):
    inp, sel, nws, nwl, b_g, dout = _case(seed, L=L, d=d, H=H)
    rng = np.random.default_rng(seed + 2000)
    w_s = 0.5 * rng.standard_normal((H, 2, 2 * d))
    b_s = 0.3 * rng.standard_normal((H, 2))
    return inp, sel, nws, nwl, b_g, dout, w_s, b_s


def _pooled(inp, chunk=64):
    q, k = inp.q.astype(np.float64), inp.k.astype(np.float64)
    B, H, L, d = q.shape
    N = L // chunk
    return np.concatenate([q.reshape(B, H, N, chunk, d).mean(3), k.reshape(B, H, N, chunk, d).mean(3)], axis=-1)


def test_st_surrogate_keeps_the_value_and_the_other_gradients():
    inp, sel, nws, nwl, b_g, dout, w_s, b_s = _st_case(311)
    args = _args(inp, nws, nwl, b_g)
    plain = ob.backward(sel=sel, dout=dout, **args)
    st = ob.backward(sel=sel, dout=dout, w_s=w_s, b_s=b_s, **args)
    np.testing.assert_array_equal(st["out"], plain["out"])  # the factor is exactly one
    for n in ("dv", "dg", "dbeta", "dw_g", "db_g", "dnorm_w_soft", "dnorm_w_lin"):
        np.testing.assert_allclose(st[n], plain[n], rtol=1e-12, atol=1e-14, err_msg=n)


def test_st_surrogate_closed_form():
    # ds_c = G_c (e_sel - pi_c), G_c = sum over the chunk's tokens of <dout_t, out_t>;
    # dW_s[h] = sum ds_c p_c^T, db_s[h] = sum ds_c; the chunk's tokens gain
    # W_s[h]^T ds_c / 64 in (dq, dk) (the q half of p, then the k half)
    inp, sel, nws, nwl, b_g, dout, w_s, b_s = _st_case(312)
    args = _args(inp, nws, nwl, b_g)
    plain = ob.backward(sel=sel, dout=dout, **args)
    st = ob.backward(sel=sel, dout=dout, w_s=w_s, b_s=b_s, **args)
    B, H, L, d = inp.q.shape
    N = L // 64
    p = _pooled(inp)                                                   # [B, H, N, 2d]
    s = np.einsum("bhnf,hof->bhno", p, w_s) + b_s[None, :, None, :]
    pi = np.exp(s - s.max(-1, keepdims=True))
    pi /= pi.sum(-1, keepdims=True)
    G = (dout * plain["out"]).reshape(B, H, N, 64, d).sum(axis=(3, 4))  # [B, H, N]
    ds = G[..., None] * (np.eye(2)[sel.astype(np.int64)] - pi)          # [B, H, N, 2]
    np.testing.assert_allclose(st["db_s"], ds.sum(axis=(0, 2)), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(st["dw_s"], np.einsum("bhno,bhnf->hof", ds, p), rtol=1e-10, atol=1e-12)
    extra = np.einsum("bhno,hof->bhnf", ds, w_s) / 64                   # [B, H, N, 2d]
    np.testing.assert_allclose(st["dq"] - plain["dq"], np.repeat(extra[..., :d], 64, axis=2), rtol=1e-8,
                               atol=1e-10)
    np.testing.assert_allclose(st["dk"] - plain["dk"], np.repeat(extra[..., d:], 64, axis=2), rtol=1e-8,
                               atol=1e-10)


@pytest.mark.parametrize("name", ("w_s", "b_s", "q", "k"))
def test_st_gradient_matches_finite_differences(name):
    # the surrogate's gradient is the derivative of its relaxed forward: out
    # scaled per chunk by pi_sel(theta) / pi_sel(theta_0), the selection fixed
    inp, sel, nws, nwl, b_g, dout, w_s, b_s = _st_case(313)
    args = _args(inp, nws, nwl, b_g)
    st = ob.backward(sel=sel, dout=dout, w_s=w_s, b_s=b_s, **args)
    x = ob.inputs64(**args)
    x["w_s"], x["b_s"] = torch.tensor(w_s), torch.tensor(b_s)
    with torch.no_grad():
        pi0 = ob.score_probs(x).gather(-1, torch.as_tensor(sel.astype(np.int64))[..., None])[..., 0].numpy()
    rng = np.random.default_rng(17)
    direction = torch.tensor(rng.standard_normal(tuple(x[name].shape)))
    R = torch.tensor(dout)

    def f(step):
        y = {n: t.detach().clone() for n, t in x.items()}
        y[name] = y[name] + step * direction
        with torch.no_grad():
            return float((ob.forward_st(y, sel, pi_bar=pi0)[0] * R).sum())

    h = 1e-5
    fd = (f(h) - f(-h)) / (2 * h)
    an = float((torch.tensor(st["d" + name]) * direction).sum())
    assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_st_planted_sign_error_fails_the_closed_form():
    # a surrogate with the sign of (e_sel - pi) flipped, planted in the oracle
    # on the CPU, is caught by the closed form's db_s
    inp, sel, nws, nwl, b_g, dout, w_s, b_s = _st_case(314)
    args = _args(inp, nws, nwl, b_g)
    good = ob.backward(sel=sel, dout=dout, w_s=w_s, b_s=b_s, **args)
    orig = ob.forward_st

    def flipped(x, sel_, *, chunk=64, pi_bar=None, **kw):
        out, o_s, o_l = ob.forward_torch(x, sel_, chunk=chunk, **kw)
        pi = ob.score_probs(x, chunk)
        chosen = pi.gather(-1, torch.as_tensor(np.asarray(sel_, np.int64))[..., None])[..., 0]
        f = (chosen.detach() / chosen).repeat_interleave(chunk, dim=-1)  # inverted factor
        return out * f[..., None], o_s, o_l

    ob.forward_st = flipped
    try:
        bad = ob.backward(sel=sel, dout=dout, w_s=w_s, b_s=b_s, **args)
    finally:
        ob.forward_st = orig
    assert not np.allclose(bad["db_s"], good["db_s"], rtol=1e-6)

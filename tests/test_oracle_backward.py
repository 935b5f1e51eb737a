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

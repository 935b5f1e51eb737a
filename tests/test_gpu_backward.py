"""The layer's backward pass (nats_hybrid_bwd) through the C ABI against the
fp64 backward oracle (oracle/backward.py), at the forward's selection:

* on the oracle's own activations (selection and branch outputs), so that
  only the backward's arithmetic is compared: every gradient within the bar
  of the dtype (fp32 layers compute in fp32; bf16 layers take the softmax
  branch on tensor cores with bf16 operands);
* end to end, on the activations the CUDA forward saved (its selection
  bit-exact with the oracle's), within the bar of the forward's dtype.
"""

import numpy as np
import pytest
import torch

import gen
import oracle
from oracle import backward as ob
from gpu_util import TOL, rel_err, to_device

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dg", "dbeta", "dw_g", "db_g", "dnorm_w_soft", "dnorm_w_lin")


def _case(B, H, L, d, dtype, seed):
    inp = gen.make_inputs(B, H, L, d, dtype=dtype, seed=seed, pattern="random", frac=0.5)
    rng = np.random.default_rng(seed + 500)
    nws = (1 + 0.2 * rng.standard_normal(d)).astype(np.float32)
    nwl = (1 + 0.2 * rng.standard_normal(d)).astype(np.float32)
    inp.b_g[:] = (0.3 * rng.standard_normal(H)).astype(np.float32)
    dout = rng.standard_normal((B, H, L, d)).astype(np.float32)
    if dtype == "bf16":
        dout = gen.round_to_bf16(dout)  # the values the device holds
    return inp, nws, nwl, dout


def _dev(x, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    return t.bfloat16() if dtype == "bf16" else t


def _oracle(inp, nws, nwl, dout, sel):
    return ob.backward(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.w_g, inp.b_g, sel, dout,
                       norm_w_soft=nws, norm_w_lin=nwl)


def _compare(got, ref, tol, label):
    errs = {n: rel_err(got[n].cpu().numpy(), ref[n]) for n in GRADS}
    print(f"[parity] backward {label}: " + " ".join(f"{n}={e:.1e}" for n, e in errs.items()))
    for n, e in errs.items():
        assert e <= tol, (n, e)


@pytest.mark.parametrize("B,H,L,d,dtype,seed", [
    (1, 2, 256, 64, "f32", 41), (1, 2, 256, 128, "f32", 42), (2, 2, 384, 128, "bf16", 43), (1, 3, 192, 64, "bf16", 44)])
def test_backward_on_oracle_activations(B, H, L, d, dtype, seed):
    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import build

    build.build()
    inp, nws, nwl, dout = _case(B, H, L, d, dtype, seed)
    sel = oracle.select_inputs(inp)[0].reshape(B, H, L // 64)
    ref = _oracle(inp, nws, nwl, dout, sel)
    t = to_device(inp)
    got = nats.hybrid_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_g"], t["b_g"],
                          torch.from_numpy(sel).cuda(), _dev(ref["o_s"], "f32"), _dev(ref["o_l"], "f32"),
                          _dev(dout, dtype), norm_w_soft=_dev(nws, "f32"), norm_w_lin=_dev(nwl, "f32"))
    torch.cuda.synchronize()
    # bf16 layers take the softmax branch on tensor cores with bf16 operands
    # (dO, P, dS rounded): the bar of the dtype
    _compare(got, ref, TOL[dtype], f"{dtype}-{d} (oracle activations)")


@pytest.mark.parametrize("B,H,L,d,dtype,seed", [(1, 2, 256, 64, "f32", 45), (2, 2, 320, 128, "bf16", 46)])
def test_backward_after_cuda_forward(B, H, L, d, dtype, seed):
    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import build

    build.build()
    inp, nws, nwl, dout = _case(B, H, L, d, dtype, seed)
    t = to_device(inp)
    nw = {"norm_w_soft": _dev(nws, "f32"), "norm_w_lin": _dev(nwl, "f32")}
    fwd = nats.hybrid_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_s"], t["b_s"], t["w_g"], t["b_g"],
                          return_sel=True, return_branches=True, check_errors=True, **nw)
    sel_ref = oracle.select_inputs(inp)[0].reshape(B, H, L // 64)
    assert np.array_equal(fwd["sel"].cpu().numpy(), sel_ref)
    got = nats.hybrid_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_g"], t["b_g"], fwd["sel"],
                          fwd["o_soft"], fwd["o_lin"], _dev(dout, dtype), **nw)
    torch.cuda.synchronize()
    _compare(got, _oracle(inp, nws, nwl, dout, sel_ref), TOL[dtype], f"{dtype}-{d} (after the CUDA forward)")


def test_backward_profiled_stages():
    # nats_hybrid_bwd_profiled: the same per-token gradients as without
    # events (the weight gradients are sums taken with atomics, in no fixed
    # order: equal to rounding), every stage's events recorded in order, and
    # the launch count
    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import _native, build

    build.build()
    inp, nws, nwl, dout = _case(1, 2, 256, 128, "bf16", 48)
    t = to_device(inp)
    nw = {"norm_w_soft": _dev(nws, "f32"), "norm_w_lin": _dev(nwl, "f32")}
    fwd = nats.hybrid_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_s"], t["b_s"], t["w_g"], t["b_g"],
                          return_sel=True, return_branches=True, **nw)
    args = (t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_g"], t["b_g"], fwd["sel"], fwd["o_soft"], fwd["o_lin"],
            _dev(dout, "bf16"))
    plain = nats.hybrid_bwd(*args, **nw)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in _native.BWD_STAGES]
    prof = _native.Profile()
    for i, (a, b) in enumerate(ev):
        a.record()  # materialise the event handles
        b.record()
        prof.start[i], prof.stop[i] = a.cuda_event, b.cuda_event
    timed = nats.hybrid_bwd(*args, **nw, profile=prof)
    torch.cuda.synchronize()
    for n in GRADS[:5]:  # dg, dbeta and dq / dk gather shared-memory sums taken with atomics
        assert torch.allclose(plain[n], timed[n], rtol=1e-5, atol=1e-6 * float(plain[n].abs().max())), n
    for n in GRADS[5:]:
        assert torch.allclose(plain[n], timed[n], rtol=1e-5, atol=1e-5 * float(plain[n].abs().max())), n
    # bf16: merge; the softmax-chunk lists, softmax dq, dk / dv (local and
    # retained key tiles); the Gated DeltaNet stage (chunk factors and scan of
    # the forward for the chunk-start states, the adjoint's chunk factors and
    # reverse scan); the adjoint's per-chunk products
    assert list(prof.stage_launches)[:len(_native.BWD_STAGES)] == [1, 4, 4, 1]
    assert prof.launches == 10
    ms = [a.elapsed_time(b) for a, b in ev]
    assert all(m > 0 for m in ms), ms
    # the softmax stage starts after the merge; the Gated DeltaNet stage's
    # state work needs no merge output and may start before it on a second
    # stream, beside the merge and the softmax stage; the per-chunk products
    # start after both
    merge, soft, gdn, comb = ev
    for a, b in ((merge[1], soft[0]), (soft[1], comb[0]), (gdn[1], comb[0])):
        assert a.elapsed_time(b) >= 0


def test_backward_all_softmax_and_all_linear():
    # the two degenerate selections: every chunk softmax (no Gated DeltaNet
    # state survives a chunk), every chunk Gated DeltaNet (only the own chunk
    # is attended by softmax)
    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import build

    build.build()
    inp, nws, nwl, dout = _case(1, 2, 256, 64, "f32", 47)
    t = to_device(inp)
    for fill in (0, 1):
        sel = np.full((1, 2, 4), fill, np.uint8)
        ref = _oracle(inp, nws, nwl, dout, sel)
        got = nats.hybrid_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_g"], t["b_g"],
                              torch.from_numpy(sel).cuda(), _dev(ref["o_s"], "f32"), _dev(ref["o_l"], "f32"),
                              _dev(dout, "f32"), norm_w_soft=_dev(nws, "f32"), norm_w_lin=_dev(nwl, "f32"))
        torch.cuda.synchronize()
        _compare(got, ref, TOL["f32"], f"all {'softmax' if fill == 0 else 'linear'}")


def test_backward_full_size_last_chunk():
    # the benchmark's workload (B=4 H=16 L=8192 d=128 bf16, 25 % softmax
    # chunks) through the CUDA forward and backward as bench.py runs them;
    # sampled: the last chunk of two heads, whose gradients (dq, dk, dv, dg,
    # dbeta) the oracle takes exactly from the retained keys / values before
    # it and the Gated DeltaNet state at its start
    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import build

    build.build()
    inp = gen.make_inputs(name="l8192", **gen.CONFIGS["l8192"])
    B, H, L, d = inp.B, inp.H, inp.L, inp.d
    N, L0 = L // 64, L - 64
    t = to_device(inp)
    fwd = nats.hybrid_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_s"], t["b_s"], t["w_g"], t["b_g"],
                          return_sel=True, return_branches=True, check_errors=True)
    dout = gen.round_to_bf16(np.random.default_rng(48).standard_normal((B, H, L, d)).astype(np.float32))
    got = nats.hybrid_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_g"], t["b_g"], fwd["sel"], fwd["o_soft"],
                          fwd["o_lin"], _dev(dout, "bf16"))
    torch.cuda.synchronize()
    sel = fwd["sel"].cpu().numpy()
    sl = slice(L0, L)
    for b, h in ((0, 3), (3, 13)):
        one = lambda a: np.ascontiguousarray(a[b:b + 1, h:h + 1])
        q, k, v, g, beta = (one(getattr(inp, n)) for n in ("q", "k", "v", "g", "beta"))
        assert np.array_equal(oracle.select(q, k, inp.w_s[h:h + 1], inp.b_s[h:h + 1])[0][0, 0], sel[b, h])
        state0 = oracle.forward(q[:, :, :L0], k[:, :, :L0], v[:, :, :L0], g[:, :, :L0], beta[:, :, :L0],
                                inp.w_s[h:h + 1], inp.b_s[h:h + 1], inp.w_g[h:h + 1], inp.b_g[h:h + 1],
                                sel_in=sel[b:b + 1, h:h + 1, :N - 1], outputs=("state",))["state"].reshape(1, 1, d, d)
        keep = np.flatnonzero(np.repeat(sel[b, h, :N - 1] == 0, 64))
        ref = ob.backward(q[:, :, sl], k[:, :, sl], v[:, :, sl], g[:, :, sl], beta[:, :, sl], inp.w_g[h:h + 1],
                          inp.b_g[h:h + 1], sel[b:b + 1, h:h + 1, N - 1:], dout[b:b + 1, h:h + 1, sl],
                          prefix_k=k[:, :, keep], prefix_v=v[:, :, keep], state0=state0)
        errs = {n: rel_err(got[n][b, h, sl].cpu().numpy(), ref[n][0, 0]) for n in ("dq", "dk", "dv", "dg", "dbeta")}
        print(f"[parity] backward l8192 head ({b}, {h}), last chunk, {len(keep)} retained keys: "
              + " ".join(f"{n}={e:.1e}" for n, e in errs.items()))
        for n, e in errs.items():
            assert e <= TOL["bf16"], (n, e)


@pytest.mark.parametrize("B,H,L,d,dtype,seed", [(1, 2, 256, 64, "f32", 61), (2, 2, 704, 128, "bf16", 62)])
def test_score_layer_gradient(B, H, L, d, dtype, seed):
    # nats_score_bwd after nats_hybrid_bwd: the straight-through surrogate's
    # gradient (reading BWD-2) against the oracle's, on the oracle's
    # activations, with the selection the score layer's own argmax; 704
    # tokens leave a partial group of chunks in the last CTA
    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import build

    build.build()
    inp, nws, nwl, dout = _case(B, H, L, d, dtype, seed)
    rng = np.random.default_rng(seed + 700)
    w_s = (0.5 * rng.standard_normal((H, 2, 2 * d))).astype(np.float32)
    b_s = (0.1 * rng.standard_normal((H, 2))).astype(np.float32)
    sel = oracle.select(inp.q, inp.k, w_s, b_s)[0]
    assert 0 < sel.mean() < 1  # both operations chosen somewhere
    ref = ob.backward(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.w_g, inp.b_g, sel, dout,
                      norm_w_soft=nws, norm_w_lin=nwl, w_s=w_s, b_s=b_s)
    t = to_device(inp)
    sel_d = torch.from_numpy(sel).cuda()
    dout_d = _dev(dout, dtype)
    grads = nats.hybrid_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_g"], t["b_g"], sel_d,
                            _dev(ref["o_s"], "f32"), _dev(ref["o_l"], "f32"), dout_d,
                            norm_w_soft=_dev(nws, "f32"), norm_w_lin=_dev(nwl, "f32"))
    before = {n: grads[n].clone() for n in ("dq", "dk")}
    nats.score_bwd(t["q"], t["k"], _dev(w_s, "f32"), _dev(b_s, "f32"), sel_d, _dev(ref["out"], dtype), dout_d,
                   grads)
    torch.cuda.synchronize()
    errs = {n: rel_err(grads[n].cpu().numpy(), ref[n]) for n in ("dq", "dk", "dw_s", "db_s")}
    # the score layer's share alone (what the call added), against the
    # oracle's surrogate minus its plain backward
    plain = ob.backward(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.w_g, inp.b_g, sel, dout,
                        norm_w_soft=nws, norm_w_lin=nwl)
    for n in ("dq", "dk"):
        errs[n + "_share"] = rel_err((grads[n] - before[n]).cpu().numpy(), ref[n] - plain[n])
    print(f"[parity] score-layer surrogate {dtype}-{d}: " + " ".join(f"{n}={e:.1e}" for n, e in errs.items()))
    for n, e in errs.items():
        assert e <= TOL[dtype], (n, e)


def test_backward_full_size_whole_head():
    # the benchmark's workload through the CUDA forward and backward as
    # bench.py runs them (the forward saves the row log-sum-exp, the backward
    # takes it); one whole head (all 8192 tokens, every chunk's state
    # gradient carried back through the reverse scan) against the oracle's
    # backward of that head, and every gradient against the backward that
    # recomputes the statistic
    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import build

    build.build()
    inp = gen.make_inputs(name="l8192", **gen.CONFIGS["l8192"])
    B, H, L, d = inp.B, inp.H, inp.L, inp.d
    t = to_device(inp)
    fwd = nats.hybrid_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_s"], t["b_s"], t["w_g"], t["b_g"],
                          return_sel=True, return_branches=True, return_lse=True, check_errors=True)
    dout = gen.round_to_bf16(np.random.default_rng(49).standard_normal((B, H, L, d)).astype(np.float32))
    args = (t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_g"], t["b_g"], fwd["sel"], fwd["o_soft"], fwd["o_lin"],
            _dev(dout, "bf16"))
    got = nats.hybrid_bwd(*args, lse=fwd["lse"])
    plain = nats.hybrid_bwd(*args)
    torch.cuda.synchronize()
    # the statistic differs from the recomputed one in its last bits, which
    # flips the bf16 rounding of a few P entries (dv sums P directly: up to
    # ~1e-4 of its max at this size)
    for n in GRADS:
        assert torch.allclose(got[n], plain[n], rtol=1e-3, atol=1e-3 * float(plain[n].abs().max())), n
    sel = fwd["sel"].cpu().numpy()
    b, h = 2, 7
    one = lambda a: a[b:b + 1, h:h + 1]
    ref = ob.backward(one(inp.q), one(inp.k), one(inp.v), one(inp.g), one(inp.beta), inp.w_g[h:h + 1],
                      inp.b_g[h:h + 1], sel[b:b + 1, h:h + 1], one(dout))
    errs = {n: rel_err(got[n][b:b + 1, h:h + 1].cpu().numpy(), ref[n]) for n in ("dq", "dk", "dv", "dg", "dbeta")}
    print("[parity] backward l8192 whole head: " + " ".join(f"{n}={e:.1e}" for n, e in errs.items()))
    for n, e in errs.items():
        assert e <= TOL["bf16"], (n, e)


@pytest.mark.parametrize("B,H,L,d,seed", [(2, 2, 320, 128, 47), (1, 3, 448, 64, 48)])
def test_backward_with_the_forward_row_statistic(B, H, L, d, seed):
    # hybrid_fwd(return_lse=True) saves the softmax rows' log-sum-exp;
    # hybrid_bwd(lse=...) then skips recomputing it: the same gradients as
    # without it (the statistic differs only by rounding order), and, for
    # d = 128, within the oracle's bar end to end
    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import build

    build.build()
    inp, nws, nwl, dout = _case(B, H, L, d, "bf16", seed)
    t = to_device(inp)
    nw = {"norm_w_soft": _dev(nws, "f32"), "norm_w_lin": _dev(nwl, "f32")}
    fwd = nats.hybrid_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_s"], t["b_s"], t["w_g"], t["b_g"],
                          return_sel=True, return_branches=True, return_lse=True, check_errors=True, **nw)
    plain = nats.hybrid_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_s"], t["b_s"], t["w_g"], t["b_g"],
                            return_sel=True, return_branches=True, **nw)
    torch.cuda.synchronize()
    for n in ("out", "sel", "o_soft", "o_lin"):  # the statistic's store changes nothing else
        assert torch.equal(plain[n], fwd[n]), n
    args = (t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_g"], t["b_g"], fwd["sel"], fwd["o_soft"],
            fwd["o_lin"], _dev(dout, "bf16"))
    ref = nats.hybrid_bwd(*args, **nw)
    got = nats.hybrid_bwd(*args, lse=fwd["lse"], **nw)
    torch.cuda.synchronize()
    for n in GRADS:  # (rounding flips of P in bf16, as in the full-size test)
        scale = float(ref[n].abs().max())
        assert torch.allclose(got[n], ref[n], rtol=1e-3, atol=1e-3 * scale), n
    if d == 128:  # the end-to-end bar, as after the CUDA forward above
        sel_ref = oracle.select_inputs(inp)[0].reshape(B, H, L // 64)
        _compare(got, _oracle(inp, nws, nwl, dout, sel_ref), TOL["bf16"], f"bf16-{d} (forward's row statistic)")

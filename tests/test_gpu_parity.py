"""CUDA path (through the C ABI) against the fp64 oracle.

Bars: chunk selection bit-exact; every compared tensor within
max|cuda - oracle| / max|oracle| <= 1e-2 (bf16 inputs) or 1e-4 (fp32 inputs).
Small workloads are compared element by element on every head and row; the
full-size workloads are run whole on the GPU and compared on sampled heads
and rows that the oracle computes one by one.
"""

import math

import numpy as np
import pytest
import torch

import gen
import oracle
from gpu_util import TOL, rel_err, run_cuda, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from linear_attention_nats_gb300 import build

    build.build()


def _compare(inp, got, ref, rows=None, tag=""):
    tol = TOL[inp.dtype]
    assert np.array_equal(got["sel"].reshape(ref["sel"].shape), ref["sel"]), f"{tag} selection differs"
    r = slice(None) if rows is None else rows
    errs = {
        "o_soft": rel_err(got["o_soft"][:, r], ref["o_s"][:, r]),
        "o_lin": rel_err(got["o_lin"], ref["o_l"]),
        "out": rel_err(got["out"][:, r], ref["out"][:, r]),
        "state": rel_err(got["state"], ref["state"]),
    }
    print(f"[parity] {tag}: " + " ".join(f"{k}={v:.2e}" for k, v in errs.items()))
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{tag} {bad} > {tol} (all: {errs})"
    return errs


def _flat(x, inp):
    return x.reshape(inp.B * inp.H, *x.shape[2:])


def _full_check(inp, sel_in=None, **kw):
    got = run_cuda(inp, sel_in=sel_in, **kw)
    okw = {k: kw[k] for k in ("scale", "eps") if k in kw}
    ref = oracle.forward_inputs(inp, sel_in=sel_in, **okw)
    got = {k: _flat(v, inp) for k, v in got.items()}
    return _compare(inp, got, ref, tag=inp.name)


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_workload_full_parity(name):
    inp = gen.config_inputs(name)
    _full_check(inp)


@pytest.mark.parametrize("name", ["tiny", "small", "l8192"])
def test_select_bit_exact(name):
    import linear_attention_nats_gb300 as nats

    inp = gen.config_inputs(name)
    t = to_device(inp)
    sel, sc = nats.select(t["q"], t["k"], t["w_s"], t["b_s"], scores=True)
    ref_sel, ref_sc = oracle.select_inputs(inp)
    assert np.array_equal(sel.cpu().numpy(), ref_sel)
    np.testing.assert_allclose(sc.cpu().numpy(), ref_sc, rtol=0, atol=2e-5)


PATTERNS = ["random", "all", "none", "alternating", "first", "last"]


@pytest.mark.parametrize("pattern", PATTERNS)
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("f32", 64), ("f32", 128)])
def test_patterns_ragged(pattern, dtype, d):
    # 7 chunks per head: an odd count, so a two-chunk query tile is left half full
    inp = gen.make_inputs(2, 2, 7 * 64, d, dtype=dtype, seed=21, pattern=pattern, frac=0.4,
                          name=f"{pattern}-{dtype}-{d}")
    _full_check(inp)


@pytest.mark.parametrize("L", [64, 128, 192])
def test_few_chunks(L):
    inp = gen.make_inputs(1, 3, L, 128, seed=L, pattern="random", frac=0.5, name=f"L{L}")
    _full_check(inp)


def test_sel_override_and_mirror():
    inp = gen.make_inputs(1, 4, 640, 128, seed=5, pattern="random", name="override")
    rng = np.random.default_rng(3)
    sel = rng.integers(0, 2, size=(1, 4, 10)).astype(np.uint8)
    _full_check(inp, sel_in=sel)
    got = run_cuda(inp, sel_in=sel)
    assert np.array_equal(got["sel"], sel)


def test_scale_eps_and_gate_saturation():
    inp = gen.make_inputs(1, 2, 512, 64, dtype="f32", seed=9, pattern="alternating", name="gate")
    _full_check(inp, scale=0.3, eps=1e-3)
    inp.b_g[:] = -1e4  # merge must reduce to the normalised linear branch
    got = run_cuda(inp)
    x = got["o_lin"].astype(np.float64)
    n = x / np.sqrt((x ** 2).mean(-1, keepdims=True) + 1e-6)
    assert rel_err(got["out"], n) <= 1e-4


def test_all_softmax_equals_causal_attention():
    inp = gen.make_inputs(1, 2, 1024, 128, seed=2, pattern="all", name="allsoft")
    t = to_device(inp)
    got = run_cuda(inp)
    ref = torch.nn.functional.scaled_dot_product_attention(
        t["q"].float(), t["k"].float(), t["v"].float(), is_causal=True)
    assert rel_err(got["o_soft"], ref.cpu().numpy()) <= 1e-2


def test_repeat_calls_are_deterministic():
    inp = gen.make_inputs(1, 2, 512, 128, seed=4, pattern="random", name="repeat")
    a = run_cuda(inp)
    b = run_cuda(inp)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_empty_inputs():
    import linear_attention_nats_gb300 as nats

    for B, H, L in ((0, 2, 128), (1, 2, 0)):
        q = torch.zeros((B, H, L, 64), dtype=torch.bfloat16, device="cuda")
        g = torch.zeros((B, H, L), device="cuda")
        out = nats.hybrid_fwd(q, q, q, g, g, torch.zeros((H, 2, 128), device="cuda"), None,
                              torch.zeros((H, 64), device="cuda"))
        assert out.shape == q.shape


def _sample_rows(L, n, seed):
    rng = np.random.default_rng(seed)
    rows = np.zeros(L, bool)
    rows[[0, 63, 64, L // 2, L - 65, L - 64, L - 1]] = True
    rows[rng.choice(L, size=n, replace=False)] = True
    return rows


@pytest.mark.parametrize("name", ["l8192", "sweep0", "sweep12", "sweep50", "sweep100", "long", "l128k"])
def test_full_size_sampled(name):
    inp = gen.config_inputs(name)
    got = run_cuda(inp)
    ref_sel, _ = oracle.select_inputs(inp)
    assert np.array_equal(got["sel"], ref_sel), "selection differs"
    if inp.planted is not None:
        assert np.array_equal(ref_sel == 0, inp.planted)
    rng = np.random.default_rng(17)
    heads = sorted(rng.choice(inp.B * inp.H, size=2, replace=False).tolist())
    rows = _sample_rows(inp.L, 96, 5)
    ref = oracle.forward_inputs(inp, heads=heads, rows=rows)
    sub = {k: _flat(v, inp)[heads] for k, v in got.items()}
    _compare(inp, sub, ref, rows=rows, tag=name)


@pytest.mark.parametrize("name", ["small", "l8192"])
def test_out_without_branch_outputs(name):
    """The call as the bench makes it: no branch outputs requested, so the
    Gated DeltaNet output stays in the workspace (bf16) until the merge."""
    import linear_attention_nats_gb300 as nats

    inp = gen.config_inputs(name)
    t = to_device(inp)
    r = nats.hybrid_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_s"], t["b_s"], t["w_g"], t["b_g"],
                        return_sel=True, check_errors=True)
    torch.cuda.synchronize()
    out = _flat(r["out"].float().cpu().numpy(), inp)
    ref_sel, _ = oracle.select_inputs(inp)
    assert np.array_equal(r["sel"].cpu().numpy(), ref_sel)
    if name == "small":
        ref = oracle.forward_inputs(inp, outputs=("out",))
        err = rel_err(out, ref["out"])
    else:
        rng = np.random.default_rng(23)
        heads = sorted(rng.choice(inp.B * inp.H, size=2, replace=False).tolist())
        rows = _sample_rows(inp.L, 96, 7)
        ref = oracle.forward_inputs(inp, heads=heads, rows=rows, outputs=("out",))
        err = rel_err(out[heads][:, rows], ref["out"][:, rows])
    print(f"[parity] {name} out only: out={err:.2e}")
    assert err <= TOL[inp.dtype]

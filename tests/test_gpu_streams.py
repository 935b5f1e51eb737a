"""Caller-owned concurrency of the layer forward (nats_hybrid_fwd_streams).

The two branches write disjoint outputs and every kernel's arithmetic is
fixed by its inputs, so the library's side stream, a caller's second stream
and both branches in order on one stream must give the same bits.
"""

import pytest
import torch

import gen
from gpu_util import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from linear_attention_nats_gb300 import build

    build.build()


@pytest.mark.parametrize("name", ["small", "l8192"])
def test_side_stream_modes_agree(name):
    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import _native

    inp = gen.config_inputs(name)
    t = to_device(inp)
    args = (t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_s"], t["b_s"], t["w_g"], t["b_g"])
    kw = dict(return_sel=True, return_state=True, return_branches=True, check_errors=True)
    ref = nats.hybrid_fwd(*args, **kw)
    side = torch.cuda.Stream()
    runs = {"caller side stream": nats.hybrid_fwd(*args, side_stream=side, **kw),
            "one stream": nats.hybrid_fwd(*args, side_stream="serial", **kw)}
    # the profiled form with the caller's stream: stages recorded, same launches
    prof = _native.Profile()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(_native.NUM_STAGES)]
    for i, (a, b) in enumerate(ev):
        a.record()
        b.record()
        prof.start[i], prof.stop[i] = a.cuda_event, b.cuda_event
    runs["caller side stream, profiled"] = nats.hybrid_fwd(*args, side_stream=side, profile=prof, **kw)
    torch.cuda.synchronize()
    for tag, got in runs.items():
        for n in ("out", "sel", "state", "o_soft", "o_lin"):
            assert torch.equal(got[n], ref[n]), (tag, n)
    assert prof.launches == 5  # chunk factors, compaction, scan, softmax, merge


def test_backward_side_stream_modes_agree():
    # nats_hybrid_bwd_streams: the library's side stream, a caller's second
    # stream and every kernel in order on one stream give the same gradients
    # (the per-token ones up to the order of their atomic sums)
    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import _native

    inp = gen.config_inputs("small")
    t = to_device(inp)
    fwd = nats.hybrid_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_s"], t["b_s"], t["w_g"], t["b_g"],
                          return_sel=True, return_branches=True)
    dout = torch.randn(t["q"].shape, generator=torch.Generator().manual_seed(5)).to(t["q"].dtype).cuda()
    args = (t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_g"], t["b_g"], fwd["sel"], fwd["o_soft"],
            fwd["o_lin"], dout)
    ref = nats.hybrid_bwd(*args)
    side = torch.cuda.Stream()
    prof = _native.Profile()
    runs = {"caller side stream": nats.hybrid_bwd(*args, side_stream=side),
            "one stream": nats.hybrid_bwd(*args, side_stream="serial"),
            "caller side stream, profiled": nats.hybrid_bwd(*args, side_stream=side, profile=prof)}
    torch.cuda.synchronize()
    for tag, got in runs.items():
        for n, x in ref.items():
            tol = float(x.abs().max()) * (1e-6 if n in ("dq", "dk", "dv", "dg", "dbeta") else 1e-5)
            assert torch.allclose(got[n], x, rtol=1e-5, atol=tol), (tag, n)
    assert prof.launches == 10

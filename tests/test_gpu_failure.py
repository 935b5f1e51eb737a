"""Failure detection without a GPU fault: an injected launch failure at each
stage of the layer forward surfaces as NATS_ERR_CUDA with the CUDA reason and
leaves the library usable; a bounded device wait that nothing completes gives
up, sets its flag and leaves the context usable."""

import ctypes

import pytest
import torch

import gen
from gpu_util import to_device

pytestmark = pytest.mark.gpu


def _fwd(t):
    import linear_attention_nats_gb300 as nats

    out = nats.hybrid_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_s"], t["b_s"], t["w_g"], t["b_g"])
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("stage", [3, 1, 4, 2, 5])  # gdn_prep, compact, gdn_scan, softmax, merge
def test_injected_stage_failure(stage):
    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import _native, build

    build.build()
    t = to_device(gen.make_inputs(1, 2, 512, 128, dtype="bf16", seed=51, pattern="random", frac=0.5))
    ref = _fwd(t).clone()
    _native.lib.nats_debug_fail_stage(stage)
    with pytest.raises(nats.NatsError) as e:
        _fwd(t)
    assert e.value.code == 7 and "invalid argument" in str(e.value)
    again = _fwd(t)  # the next call is clean
    assert torch.equal(again, ref)


def test_bounded_wait_gives_up():
    from linear_attention_nats_gb300 import _native, build

    build.build()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    code = _native.lib.nats_debug_bounded_wait(ctypes.c_void_p(flag.data_ptr()), 1_000_000,
                                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0
    torch.cuda.synchronize()
    assert int(flag.item()) == 1
    # the context is still usable
    t = to_device(gen.make_inputs(1, 2, 256, 64, dtype="bf16", seed=52, pattern="random", frac=0.5))
    out = _fwd(t)
    assert torch.isfinite(out.float()).all()

"""The layer with its projections (nats_hybrid_fwd_x) through the C ABI
against the fp64 oracle (oracle.forward_x): chunk selection bit-exact, y
within max|cuda - oracle| / max|oracle| <= 1e-2 (bf16)."""

import numpy as np
import pytest
import torch

import gen
import oracle
from gpu_util import TOL, rel_err

pytestmark = pytest.mark.gpu


def _bf16(a):
    return torch.from_numpy(gen.bf16_bits(np.ascontiguousarray(a, np.float32)).view(np.int16)).view(
        torch.bfloat16).cuda()


def _f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


@pytest.mark.parametrize("name", ["x_tiny", "x_small", "x_mid", "x_ragged"])
def test_x_path_parity(name):
    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import build

    build.build()
    inp = gen.x_config_inputs(name)
    r = nats.hybrid_fwd_x(_bf16(inp.x), _bf16(inp.w_qkv), _bf16(inp.w_ab), _f32(inp.w_s), _f32(inp.b_s),
                          _f32(inp.w_g), _f32(inp.b_g), heads=inp.H, b_a=_f32(inp.b_a), a_scale=_f32(inp.a_scale),
                          b_b=_f32(inp.b_b), w_o=_bf16(inp.w_o), return_sel=True, check_errors=True)
    torch.cuda.synchronize()
    ref = oracle.forward_x(inp.x, inp.w_qkv, inp.w_ab, inp.w_s, inp.b_s, inp.w_g, inp.b_g, inp.w_o, inp.H,
                           b_a=inp.b_a, a_scale=inp.a_scale, b_b=inp.b_b)
    margins = np.abs(ref["scores"][..., 0] - ref["scores"][..., 1])
    assert margins.min() >= 1e-3, "workload too close to a selection tie"
    assert np.array_equal(r["sel"].cpu().numpy(), ref["sel"])
    err = rel_err(r["y"].float().cpu().numpy(), ref["y"])
    print(f"[parity] {name} x path: y={err:.2e}")
    assert err <= TOL["bf16"]

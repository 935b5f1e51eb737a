"""Native Hybrid Attention on the GPU (nats_nha_fwd through the C ABI)
against the fp64 oracle (oracle/nha.py, reading CONV-16): every window
regime (w = 0: Gated Slot Attention; w >= L: causal attention; hybrid
windows), ragged chunk counts, and sampled heads of the measured workload,
within max|cuda - oracle| / max|oracle| <= 1e-2 (bf16)."""

import numpy as np
import pytest
import torch

import gen
from gpu_util import TOL, rel_err
from oracle import nha as oracle_nha

pytestmark = pytest.mark.gpu


def _bf16(a):
    return torch.from_numpy(gen.bf16_bits(np.ascontiguousarray(a, np.float32)).view(np.int16)).view(
        torch.bfloat16).cuda()


def _run(inp, window=None):
    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import build

    build.build()
    la = torch.from_numpy(np.ascontiguousarray(inp.log_alpha)).cuda()
    o = nats.nha_fwd(_bf16(inp.q), _bf16(inp.k), _bf16(inp.v), la, window=inp.window if window is None else window,
                     check_errors=True)
    torch.cuda.synchronize()
    return o.float().cpu().numpy()


@pytest.mark.parametrize("name", ["nha_tiny", "nha_w0", "nha_full", "nha_w256", "nha_mid"])
def test_nha_parity(name):
    inp = gen.nha_config_inputs(name)
    out = _run(inp)
    ref = oracle_nha.forward_inputs(inp)
    err = rel_err(out, ref)
    print(f"[parity] {name}: out={err:.2e}")
    assert np.isfinite(out).all()
    assert err <= TOL["bf16"]


@pytest.mark.parametrize("window", [0, 128, 384, 1024])
def test_nha_windows_ragged(window):
    """7 chunks (the last tile holds one chunk), every supported window regime."""
    inp = gen.make_nha_inputs(1, 2, 448, window=window, seed=40 + window)
    out = _run(inp)
    ref = oracle_nha.forward_inputs(inp)
    assert rel_err(out, ref) <= TOL["bf16"]


def test_nha_full_size_sampled_heads():
    """The measured launch configuration (B = 4, H = 16, L = 8192, w = 512):
    two whole heads against the oracle run on those heads alone."""
    inp = gen.nha_config_inputs("nha_l8192")
    out = _run(inp)
    for b, h in ((0, 0), (3, 11)):
        sub = gen.NhaInputs(B=1, H=1, L=inp.L, d=inp.d, m=inp.m, window=inp.window, dtype=inp.dtype,
                            q=inp.q[b:b + 1, h:h + 1], k=inp.k[b:b + 1, h:h + 1], v=inp.v[b:b + 1, h:h + 1],
                            log_alpha=inp.log_alpha[b:b + 1, h:h + 1])
        ref = oracle_nha.forward_inputs(sub)[0, 0]
        err = rel_err(out[b, h], ref)
        print(f"[parity] nha_l8192 head ({b}, {h}): out={err:.2e}")
        assert err <= TOL["bf16"]


def test_nha_repeat_calls_are_deterministic():
    inp = gen.nha_config_inputs("nha_w256")
    assert np.array_equal(_run(inp), _run(inp))

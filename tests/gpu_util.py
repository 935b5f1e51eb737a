"""Helpers shared by the GPU parity tests: upload seeded inputs, run the CUDA
path through the C ABI, compare with the oracle."""

from __future__ import annotations

import numpy as np
import torch

import gen

# Parity bars: max|cuda - oracle| / max|oracle| per compared tensor.
TOL = {"bf16": 1e-2, "f32": 1e-4}


def to_device(inp: gen.NatsInputs, device="cuda"):
    """Canonical inputs as CUDA tensors (Q, K, V in their storage dtype)."""
    if inp.dtype == "bf16":
        qkv = [torch.from_numpy(gen.bf16_bits(x).view(np.int16)).view(torch.bfloat16) for x in (inp.q, inp.k, inp.v)]
    else:
        qkv = [torch.from_numpy(x) for x in (inp.q, inp.k, inp.v)]
    d = {n: t.to(device) for n, t in zip(("q", "k", "v"), qkv)}
    for n in ("g", "beta", "w_s", "b_s", "w_g", "b_g"):
        d[n] = torch.from_numpy(np.ascontiguousarray(getattr(inp, n))).to(device)
    return d


def run_cuda(inp: gen.NatsInputs, sel_in=None, **kw):
    import linear_attention_nats_gb300 as nats

    t = to_device(inp)
    if sel_in is not None:
        kw["sel_in"] = torch.from_numpy(np.ascontiguousarray(sel_in, np.uint8)).cuda()
    r = nats.hybrid_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_s"], t["b_s"], t["w_g"],
                        t["b_g"], return_sel=True, return_state=True, return_branches=True, check_errors=True, **kw)
    torch.cuda.synchronize()
    return {k: v.float().cpu().numpy() if v.dtype != torch.uint8 else v.cpu().numpy() for k, v in r.items()}


def rel_err(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref).max()
    return float(np.abs(x - ref).max() / max(den, 1e-30))

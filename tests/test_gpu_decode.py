"""The layer in decode mode (nats_decode_step) through the C ABI against the
fp64 prefill oracle: stepped token by token from the empty state, every
token's output and both branch outputs match oracle.forward of the whole
sequence, chunk selections are bit-exact and the final state matches; and a
decode that continues a prefill (nats_hybrid_fwd's state and retained
chunks) matches the oracle over the whole sequence."""

import numpy as np
import pytest
import torch

import gen
import oracle
from gpu_util import TOL, rel_err, to_device

pytestmark = pytest.mark.gpu


def _decode(t_dev, inp, state, t0, t1, nws=None, nwl=None):
    import linear_attention_nats_gb300 as nats

    B, H, d = inp.B, inp.H, inp.d
    outs = {n: np.zeros((B, H, t1 - t0, d)) for n in ("out", "o_s", "o_l")}
    sel = []
    sel_buf = torch.zeros((B, H), dtype=torch.uint8, device="cuda")
    for t in range(t0, t1):
        q, k, v = (t_dev[n][:, :, t].contiguous() for n in ("q", "k", "v"))
        g, beta = (t_dev[n][:, :, t].contiguous() for n in ("g", "beta"))
        r = nats.decode_step(state, t, q, k, v, g, beta, t_dev["w_s"], t_dev["b_s"], t_dev["w_g"], t_dev["b_g"],
                             norm_w_soft=nws, norm_w_lin=nwl, sel_out=sel_buf, return_branches=True)
        for n in ("out", "o_s", "o_l"):
            outs[n][:, :, t - t0] = r[n].float().cpu().numpy()
        if t % 64 == 63:
            sel.append(sel_buf.cpu().numpy().copy())
    torch.cuda.synchronize()
    state.check()
    return outs, (np.stack(sel, axis=-1) if sel else np.zeros((B, H, 0), np.uint8))


@pytest.mark.parametrize("B,H,L,d,dtype,seed,norm", [
    (1, 2, 256, 64, "f32", 31, False), (2, 4, 384, 128, "bf16", 32, False),
    (1, 2, 256, 64, "bf16", 34, True), (1, 2, 192, 128, "f32", 35, True)])
def test_decode_from_empty_matches_prefill_oracle(B, H, L, d, dtype, seed, norm):
    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import build

    build.build()
    inp = gen.make_inputs(B, H, L, d, dtype=dtype, seed=seed, pattern="random", frac=0.5)
    t_dev = to_device(inp)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    state = nats.DecodeState(B, H, d, cap=L, dtype=tdt)
    nw = {}
    if norm:  # learnable RMSNorm weights of both branches
        rng = np.random.default_rng(seed + 100)
        nw = {"norm_w_soft": (1 + 0.2 * rng.standard_normal(d)).astype(np.float32),
              "norm_w_lin": (1 + 0.2 * rng.standard_normal(d)).astype(np.float32)}
    dev_nw = {k: torch.from_numpy(v).cuda() for k, v in nw.items()}
    outs, sel = _decode(t_dev, inp, state, 0, L, dev_nw.get("norm_w_soft"), dev_nw.get("norm_w_lin"))
    ref = oracle.forward_inputs(inp, **nw)
    assert np.array_equal(sel.reshape(ref["sel"].shape), ref["sel"])
    tol = TOL[dtype]
    errs = {n: rel_err(outs[n].reshape(ref[n].shape), ref[n]) for n in ("o_s", "o_l", "out")}
    errs["state"] = rel_err(state.S.cpu().numpy().reshape(ref["state"].shape), ref["state"])
    print(f"[parity] decode {dtype}-{d}{' norm' if norm else ''}: " + " ".join(f"{k}={v:.2e}" for k, v in errs.items()))
    for n, e in errs.items():
        assert e <= tol, (n, e)
    # the retained keys are those of the softmax chunks, in order
    n_kv = state.n_kv.cpu().numpy()
    assert np.array_equal(n_kv, 64 * (ref["sel"].reshape(B, H, -1) == 0).sum(-1))


@pytest.mark.parametrize("B,H,L,L0,seed", [(2, 4, 448, 256, 33), (1, 2, 2112, 2048, 36)])
def test_decode_continues_prefill(B, H, L, L0, seed):
    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import build

    build.build()
    d = 128
    inp = gen.make_inputs(B, H, L, d, dtype="bf16", seed=seed, pattern="random", frac=0.5)
    t_dev = to_device(inp)
    # prefill of the first L0 tokens through the layer forward
    pre = nats.hybrid_fwd(t_dev["q"][:, :, :L0].contiguous(), t_dev["k"][:, :, :L0].contiguous(),
                          t_dev["v"][:, :, :L0].contiguous(), t_dev["g"][:, :, :L0].contiguous(),
                          t_dev["beta"][:, :, :L0].contiguous(), t_dev["w_s"], t_dev["b_s"], t_dev["w_g"],
                          t_dev["b_g"], return_sel=True, return_state=True)
    # decode state after it: the chunk boundary state and the retained chunks
    state = nats.DecodeState(B, H, d, cap=L, dtype=torch.bfloat16)
    state.S.copy_(pre["state"])
    state.S0.copy_(pre["state"])
    sel0 = pre["sel"].cpu().numpy()
    for b in range(B):
        for h in range(H):
            keep = [c for c in range(L0 // 64) if sel0[b, h, c] == 0]
            for i, c in enumerate(keep):
                state.kv_k[b, h, 64 * i:64 * (i + 1)] = t_dev["k"][b, h, 64 * c:64 * (c + 1)]
                state.kv_v[b, h, 64 * i:64 * (i + 1)] = t_dev["v"][b, h, 64 * c:64 * (c + 1)]
            state.n_kv[b, h] = 64 * len(keep)
    outs, sel = _decode(t_dev, inp, state, L0, L)
    ref = oracle.forward_inputs(inp)
    N0 = L0 // 64
    assert np.array_equal(sel0.reshape(B * H, -1), ref["sel"][:, :N0])
    assert np.array_equal(sel.reshape(B * H, -1), ref["sel"][:, N0:])
    errs = {n: rel_err(outs[n].reshape(B * H, L - L0, d), ref[n][:, L0:]) for n in ("o_s", "o_l", "out")}
    print(f"[parity] decode after a {L0}-token prefill: " + " ".join(f"{k}={v:.2e}" for k, v in errs.items()))
    for n, e in errs.items():
        assert e <= TOL["bf16"], (n, e)

"""bf16 error budget of the Gated DeltaNet branch's tensor-core forward, on
the CPU.

The CUDA path ("Neural Attention Search Linear (NAtS-L)", technical summary,
"Kernmechanismen" item 3, in the chunkwise WY form) rounds to bf16 at seven
points: the chunk factors W = T diag(beta e^G) K, U = T diag(beta) V and
P = lower(e^{G_t - G_i} scale q_t . k_i) as stored; the scaled tiles
Q~ = diag(scale gamma) Q and K~ = diag(gamma_C / gamma) K; the bf16 copy of
the chunk-start state S0 that the products read; and Delta^T = U^T - S0 W^T
before it multiplies K~ and P^T.  Every product accumulates in fp32 and the
state itself stays fp32.  This model runs the same chunkwise steps in
float64 with each of those roundings applied (or all but one), against the
exact token recurrence with rollback, and states what each contributes and
how the error of o_l grows with the sequence length.  The bar of the GPU
parity tests is 1e-2 (max |error| / max |reference|).
"""

import numpy as np
import pytest

import gen

C = 64


def bf16(a):
    a = np.asarray(a, np.float32)
    b = a.view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16  # round to nearest even
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def exact(q, k, v, g, beta, sel, scale):
    L, d = q.shape
    S = np.zeros((d, d))
    out = np.empty((L, d))
    for c in range(L // C):
        S0 = S.copy()
        for t in range(c * C, (c + 1) * C):
            a = np.exp(g[t])
            S = a * S + beta[t] * np.outer(v[t] - a * (S @ k[t]), k[t])
            out[t] = S @ (scale * q[t])
        if sel[c] == 0:
            S = S0
    return out


def chunkwise(q, k, v, g, beta, sel, scale, rounded):
    """The CUDA path's chunkwise steps; `rounded` names the bf16 roundings applied."""
    R = {n: (bf16 if n in rounded else (lambda a: a)) for n in ("W", "U", "P", "Qt", "Kt", "S0", "Delta")}
    L, d = q.shape
    S = np.zeros((d, d))
    out = np.empty((L, d))
    for c in range(L // C):
        sl = slice(c * C, (c + 1) * C)
        Q, K, V, gg, bb = q[sl], k[sl], v[sl], g[sl], beta[sl]
        G = np.cumsum(gg)
        gam = np.exp(G)
        ratio = np.exp(G[:, None] - G[None, :])
        A = np.tril(ratio * (K @ K.T), -1) * bb[:, None]
        T = np.linalg.inv(np.eye(C) + A) * bb[None, :]
        W = R["W"](T @ (gam[:, None] * K))
        U = R["U"](T @ V)
        P = R["P"](np.tril(ratio * (scale * Q @ K.T)))
        Qt = R["Qt"](scale * gam[:, None] * Q)
        Kt = R["Kt"]((gam[-1] / gam)[:, None] * K)
        S0 = R["S0"](S)
        Delta = R["Delta"](U - W @ S0.T)
        out[sl] = Qt @ S0.T + P @ Delta
        if sel[c] != 0:
            S = gam[-1] * S + Delta.T @ Kt
    return out


POINTS = ("W", "U", "P", "Qt", "Kt", "S0", "Delta")


def _case(L, seed=4):
    inp = gen.make_inputs(1, 1, L, 128, dtype="bf16", seed=seed, pattern="random", frac=0.125)
    sel = gen.make_inputs(1, 1, L, 128, dtype="bf16", seed=seed, pattern="random", frac=0.125).planted
    q, k, v, g, beta = (a[0, 0].astype(np.float64) for a in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    sel = (~np.asarray(sel)[0, 0]).astype(np.uint8)  # planted chunks are the softmax ones
    return q, k, v, g, beta, sel, 128 ** -0.5


def _err(a, ref):
    return float(np.abs(a - ref).max() / np.abs(ref).max())


@pytest.mark.slow
def test_bf16_budget_of_the_gated_deltanet_branch():
    rows = {}
    for L in (8192, 65536):
        q, k, v, g, beta, sel, scale = _case(L)
        ref = exact(q, k, v, g, beta, sel, scale)
        full = _err(chunkwise(q, k, v, g, beta, sel, scale, set(POINTS)), ref)
        without = {p: _err(chunkwise(q, k, v, g, beta, sel, scale, set(POINTS) - {p}), ref) for p in POINTS}
        only = {p: _err(chunkwise(q, k, v, g, beta, sel, scale, {p}), ref) for p in POINTS}
        rows[L] = (full, without, only)
        print(f"[budget] L={L}: all roundings {full:.2e}; alone: "
              + " ".join(f"{p}={e:.1e}" for p, e in only.items())
              + "; all but: " + " ".join(f"{p}={e:.1e}" for p, e in without.items()))
    # the modelled error of o_l stays below the bar at both lengths, grows
    # slowly with L (the state's error is damped by the decay), and no
    # single rounding point carries it alone
    for L, (full, without, only) in rows.items():
        assert full < 1e-2, (L, full)
        assert max(only.values()) < full * 1.01
    assert rows[65536][0] < 2.5 * rows[8192][0]

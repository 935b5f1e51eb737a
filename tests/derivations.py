"""Independent float64 derivations used to pin the oracle.

Each function reaches the layer's result by a different route than the
oracle's token-by-token loops (a dense L x L mask, an explicit product of
transition matrices, the chunkwise WY/UT closed form), so that a slip in one
of them (a dropped term, a wrong sign or index, a transposed operand) shows
up as a mismatch.  Sizes are tiny; nothing here is fast.
"""

from __future__ import annotations

import numpy as np


def kv_mask(sel: np.ndarray, L: int, C: int) -> np.ndarray:
    """Boolean [L, L] mask M[t, j]: key j is visible to query t in the softmax branch.

    j <= t and (j is in t's own chunk or j's chunk chose softmax).
    """
    chunk = np.arange(L) // C
    t = np.arange(L)[:, None]
    j = np.arange(L)[None, :]
    same = chunk[:, None] == chunk[None, :]
    soft = (sel[chunk] == 0)[None, :]
    return (j <= t) & (same | soft)


def dense_masked_attention(q, k, v, sel, C, scale):
    """softmax(Q K^T * scale + log M) V for one head, float64."""
    L = q.shape[0]
    M = kv_mask(np.asarray(sel), L, C)
    s = (q.astype(np.float64) @ k.astype(np.float64).T) * scale
    s = np.where(M, s, -np.inf)
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    return p @ v.astype(np.float64)


def effective_tokens(sel, L, C, t):
    """Token indices whose writes are in the Gated DeltaNet state read at t.

    Tokens of earlier chunks that chose the linear operation, then the tokens
    of t's own chunk up to t (rolled-back chunks vanish entirely).
    """
    c = t // C
    toks = [j for j in range(c * C) if sel[j // C] == 1]
    toks += list(range(c * C, t + 1))
    return toks


def gdn_product_form(q, k, v, g, beta, sel, C, scale):
    """o_t = S_t (scale q_t) with S_t written as an explicit sum of products.

    S_t = sum_i beta_i v_i k_i^T  prod_{j after i} a_j (I - beta_j k_j k_j^T)
    over the effective token sequence of t (right-multiplied in time order).
    Also returns the final state (after the last chunk's commit or rollback).
    """
    L, dk = k.shape
    dv = v.shape[1]
    q, k, v = (x.astype(np.float64) for x in (q, k, v))
    beta = beta.astype(np.float64)
    a = np.exp(g.astype(np.float64))
    I = np.eye(dk)

    def state(toks):
        S = np.zeros((dv, dk))
        for n, i in enumerate(toks):
            term = beta[i] * np.outer(v[i], k[i])
            for j in toks[n + 1:]:
                term = term @ (a[j] * (I - beta[j] * np.outer(k[j], k[j])))
            S += term
        return S

    o = np.zeros((L, dv))
    for t in range(L):
        S = state(effective_tokens(sel, L, C, t))
        o[t] = S @ (scale * q[t].astype(np.float64))
    N = (L + C - 1) // C
    final = [j for j in range(L) if sel[j // C] == 1]
    return o, state(final)


def gdn_chunkwise(q, k, v, g, beta, sel, C, scale):
    """Chunkwise WY/UT closed form of the same branch, float64.

    Per chunk with start state S0 and in-chunk cumulative log-decay G:
      A    = strict_lower(beta_t e^{G_t - G_i} k_t . k_i)
      T    = (I + A)^{-1}
      U    = T diag(beta) V,  W = T diag(beta e^{G}) K
      Delta= U - W S0^T
      O    = e^{G} * (scale Q S0^T) + P Delta,  P = lower_incl(e^{G_t - G_i} scale q_t . k_i)
      S_C  = e^{G_C} S0 + Delta^T diag(e^{G_C - G}) K
    and S0 is kept (rollback) when the chunk chose softmax.
    """
    L, dk = k.shape
    dv = v.shape[1]
    q, k, v = (x.astype(np.float64) for x in (q, k, v))
    g, beta = g.astype(np.float64), beta.astype(np.float64)
    S = np.zeros((dv, dk))
    o = np.zeros((L, dv))
    N = (L + C - 1) // C
    for c in range(N):
        sl = slice(c * C, min(L, (c + 1) * C))
        Kc, Vc, Qc = k[sl], v[sl], q[sl]
        n = Kc.shape[0]
        G = np.cumsum(g[sl])
        D = np.exp(G[:, None] - G[None, :])
        A = np.tril(beta[sl][:, None] * D * (Kc @ Kc.T), -1)
        T = np.linalg.inv(np.eye(n) + A)
        U = T @ (beta[sl][:, None] * Vc)
        W = T @ ((beta[sl] * np.exp(G))[:, None] * Kc)
        Delta = U - W @ S.T
        P = np.tril(D * (Qc @ Kc.T)) * scale
        o[sl] = np.exp(G)[:, None] * (scale * Qc @ S.T) + P @ Delta
        S_end = np.exp(G[-1]) * S + Delta.T @ (np.exp(G[-1] - G)[:, None] * Kc)
        if sel[c] == 1:
            S = S_end
    return o, S

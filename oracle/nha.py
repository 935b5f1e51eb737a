"""fp64 CPU oracle of the Native Hybrid Attention (NHA) layer.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module; the library product
never does.  Plain numpy in float64, one token at a time.  It shares no code
with the CUDA path.

"Native Hybrid Attention for Efficient Sequence Modeling" (gist.science,
nl/paper/2510.07019), section "2. Methodologie", "Kernprincipes":
  * long-term information is compressed into a fixed number of slots (key /
    value pairs) by a linear RNN update inspired by Gated Slot Attention;
  * the slots are joined with the short-term tokens of a sliding window into
    one key / value set, and one softmax attention runs over that set;
  * the window size w is the only knob: w = 0 is a pure linear RNN, w equal
    to the sequence length is full attention.

The page gives no update rule, gate form or slot count.  The reading taken
here is CONV-16:
  * slot memory as in Gated Slot Attention (Zhang et al., 2024): m slots,
    K~, V~ in R^{m x d}, written by a token j as
        K~ <- diag(alpha_j) K~ + (1 - alpha_j) k_j^T,
        V~ <- diag(alpha_j) V~ + (1 - alpha_j) v_j^T,
    alpha_j in (0, 1)^m a per-slot forget gate, given as its logarithm
    (log_alpha, <= 0); K~ = V~ = 0 before the first write;
  * a token enters the slots when it leaves the window: the query at t sees
    the window tokens t - w < j <= t, and the slot memory after the writes
    of every token j <= t - w (none while t < w);
  * one softmax over the m slot keys (only once at least one token has been
    written) and the window keys, logits scale * q_t . key, scale = 1/sqrt(d)
    unless given; the output is the same weights over [V~; V_window];
  * no normalisation or gate after it.
With w = 0 the window is empty and every token is written before its own
query reads the slots: Gated Slot Attention.  With w >= L nothing is ever
written and the slots never take part: causal softmax attention.
"""

from __future__ import annotations

import numpy as np


def forward(q, k, v, log_alpha, window: int, scale: float = 0.0):
    """q, k, v [B, H, L, d]; log_alpha [B, H, L, m] (<= 0).  Returns o [B, H, L, d]
    (float64)."""
    q, k, v, la = (np.asarray(x, np.float64) for x in (q, k, v, log_alpha))
    B, H, L, d = q.shape
    m = la.shape[-1]
    if window < 0:
        raise ValueError("window must be >= 0")
    sc = scale if scale > 0 else 1.0 / np.sqrt(d)
    o = np.zeros((B, H, L, d))
    for b in range(B):
        for h in range(H):
            Ks = np.zeros((m, d))
            Vs = np.zeros((m, d))
            written = False
            for t in range(L):
                j = t - window  # the token leaving the window enters the slots
                if j >= 0:
                    a = np.exp(la[b, h, j])
                    Ks = a[:, None] * Ks + (1.0 - a)[:, None] * k[b, h, j][None, :]
                    Vs = a[:, None] * Vs + (1.0 - a)[:, None] * v[b, h, j][None, :]
                    written = True
                lo = max(0, t - window + 1)
                keys = [k[b, h, lo:t + 1]]
                vals = [v[b, h, lo:t + 1]]
                if written:
                    keys.insert(0, Ks)
                    vals.insert(0, Vs)
                K = np.concatenate(keys, 0)
                V = np.concatenate(vals, 0)
                z = sc * (K @ q[b, h, t])
                p = np.exp(z - z.max())
                o[b, h, t] = (p / p.sum()) @ V
    return o


def forward_inputs(inp, window=None, scale: float = 0.0):
    """The oracle on a generator record (gen.NhaInputs)."""
    return forward(inp.q, inp.k, inp.v, inp.log_alpha, inp.window if window is None else window, scale)

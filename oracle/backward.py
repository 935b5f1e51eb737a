"""fp64 CPU oracle of the NAtS-L layer's backward pass at a fixed selection.

TEST INFRASTRUCTURE ONLY: the tests and the benchmark's CPU-baseline leg may
import this module; the library product never does.  It shares no code with
the CUDA path.

The layer ("Neural Attention Search Linear (NAtS-L)", technical summary,
"Kernmechanismen" items 1, 3 and 4) is written out here a second time, in
plain PyTorch float64 on the CPU, as a function of its continuous inputs at
a given chunk selection:

* softmax branch: the dense masked form, softmax(q k^T scale + log M) v with
  M[t, j] = 1 when j <= t and j is in t's chunk or in an earlier chunk that
  chose softmax (the retained KV set of item 3);
* Gated DeltaNet branch: the token recurrence S <- a S + beta (v - a S k) k^T,
  o_l = S (scale q), with the state put back to the chunk start after every
  chunk that chose softmax (item 3's rollback);
* RMSNorm of each branch and the query-gated sum w N_s + (1 - w) N_l with
  w = sigmoid(q . W_g[h] + b_g[h]) (item 4).

The backward is the gradient of <dout, out> with respect to q, k, v, g, beta,
W_g, b_g and the two RMSNorm weights, taken by torch.autograd through that
forward.  The selection is the forward's argmax (item 1): a discrete choice
with no derivative; the pages state that the score layer is trained end to
end but give no estimator for it, so its gradient is not part of this
backward (the reading BWD-1).

Opt-in (the reading BWD-2, `backward(..., w_s=, b_s=)`): a straight-through
surrogate that lets the score layer learn.  With pi_c = softmax(s_c) over the
chunk's two scores s_c = W_s[h] p_c + b_s[h] (p_c the chunk mean of [q; k],
item 1) and sel_c the argmax, every output row of chunk c is multiplied by
pi_c[sel_c] / pi_c[sel_c] held constant: the value is unchanged, and
<dout, out> gains a gradient with respect to W_s, b_s and, through p_c, the
chunk's q and k.
"""

from __future__ import annotations

import numpy as np
import torch

NAMES = ("q", "k", "v", "g", "beta", "w_g", "b_g", "norm_w_soft", "norm_w_lin")


def _mask(sel_bh, L, chunk):
    """M[t, j] of one head: j <= t, and j in t's chunk or in an earlier chunk
    that chose softmax (sel = 0)."""
    t = torch.arange(L)
    ct = t // chunk
    causal = t[None, :] <= t[:, None]
    same = ct[None, :] == ct[:, None]
    soft = torch.as_tensor(np.asarray(sel_bh) == 0)[ct]  # chunk of key j chose softmax
    return causal & (same | soft[None, :])


def forward_torch(x, sel, *, chunk=64, scale=0.0, eps=1e-6, prefix_k=None, prefix_v=None, state0=None):
    """The layer at selection `sel` [B, H, N] on the float64 tensors of dict
    x (q, k, v [B, H, L, d]; g, beta [B, H, L]; w_g [H, d]; b_g [H]; norm
    weights [d]).  Returns (out, o_s, o_l), each [B, H, L, d].

    The tokens may continue a longer sequence: prefix_k, prefix_v
    [B, H, P, d] are the retained keys / values of its earlier softmax
    chunks (seen by every query here), state0 [B, H, dv, dk] its Gated
    DeltaNet state at this point (both constants)."""
    q, k, v, g, beta = x["q"], x["k"], x["v"], x["g"], x["beta"]
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    sc = scale if scale > 0 else dk ** -0.5
    N = (L + chunk - 1) // chunk
    outs, oss, ols = [], [], []
    for b in range(B):
        ob, osb, olb = [], [], []
        for h in range(H):
            qh, kh, vh = q[b, h], k[b, h], v[b, h]
            # softmax branch: dense masked attention over the retained set
            M = _mask(sel[b, h], L, chunk)
            logits = (qh @ kh.T) * sc
            logits = logits.masked_fill(~M, float("-inf"))
            if prefix_k is not None:  # the earlier retained keys, seen by every query
                pk = torch.as_tensor(prefix_k[b, h], dtype=q.dtype)
                pv = torch.as_tensor(prefix_v[b, h], dtype=q.dtype)
                o_s = torch.softmax(torch.cat([(qh @ pk.T) * sc, logits], dim=-1), dim=-1) @ torch.cat([pv, vh])
            else:
                o_s = torch.softmax(logits, dim=-1) @ vh
            # Gated DeltaNet branch: token recurrence with chunk rollback
            S = torch.zeros(dv, dk, dtype=q.dtype) if state0 is None else torch.as_tensor(state0[b, h], dtype=q.dtype)
            rows = []
            for c in range(N):
                S0 = S
                for t in range(c * chunk, min(L, (c + 1) * chunk)):
                    a = torch.exp(g[b, h, t])
                    kt, vt = kh[t], vh[t]
                    S = a * S + beta[b, h, t] * torch.outer(vt - a * (S @ kt), kt)
                    rows.append(S @ (qh[t] * sc))
                if sel[b, h, c] == 0:
                    S = S0
            o_l = torch.stack(rows)
            # RMSNorm of each branch, query-gated sum
            ns = o_s * torch.rsqrt((o_s * o_s).mean(-1, keepdim=True) + eps) * x["norm_w_soft"]
            nl = o_l * torch.rsqrt((o_l * o_l).mean(-1, keepdim=True) + eps) * x["norm_w_lin"]
            w = torch.sigmoid(qh @ x["w_g"][h] + x["b_g"][h])[:, None]
            ob.append(w * ns + (1 - w) * nl)
            osb.append(o_s)
            olb.append(o_l)
        outs.append(torch.stack(ob))
        oss.append(torch.stack(osb))
        ols.append(torch.stack(olb))
    return torch.stack(outs), torch.stack(oss), torch.stack(ols)


def score_probs(x, chunk=64):
    """pi [B, H, N, 2]: the softmax over the two operation scores of every
    chunk, s = W_s[h] p + b_s[h] with p the mean over the chunk's tokens of
    [q_t ; k_t] (unscaled q; a partial last chunk pools the tokens it has)."""
    q, k = x["q"], x["k"]
    L = q.shape[2]
    N = (L + chunk - 1) // chunk
    pooled = torch.stack([torch.cat([q[:, :, c * chunk:(c + 1) * chunk].mean(2),
                                     k[:, :, c * chunk:(c + 1) * chunk].mean(2)], dim=-1) for c in range(N)], dim=2)
    s = torch.einsum("bhnf,hof->bhno", pooled, x["w_s"]) + x["b_s"][None, :, None, :]
    return torch.softmax(s, dim=-1)


def forward_st(x, sel, *, chunk=64, pi_bar=None, **kw):
    """The straight-through surrogate of BWD-2: forward_torch's out with every
    row of chunk c multiplied by pi_c[sel_c] / pi_bar_c, pi_bar the same
    probability held constant (by default the one at x, so the value is
    unchanged; a finite-difference check passes the unperturbed one).
    Returns (out, o_s, o_l) like forward_torch."""
    out, o_s, o_l = forward_torch(x, sel, chunk=chunk, **kw)
    L = out.shape[2]
    pi = score_probs(x, chunk)
    chosen = pi.gather(-1, torch.as_tensor(np.asarray(sel, np.int64))[..., None])[..., 0]  # [B, H, N]
    bar = chosen.detach() if pi_bar is None else torch.as_tensor(np.asarray(pi_bar, np.float64))
    f = (chosen / bar).repeat_interleave(chunk, dim=-1)[..., :L]
    return out * f[..., None], o_s, o_l


def inputs64(q, k, v, g, beta, w_g, b_g=None, norm_w_soft=None, norm_w_lin=None):
    """float64 leaf tensors of the continuous inputs (absent bias / norm
    weights become zeros / ones)."""
    H, d = np.shape(w_g)
    dv = np.shape(v)[-1]
    vals = {"q": q, "k": k, "v": v, "g": g, "beta": beta, "w_g": w_g,
            "b_g": np.zeros(H) if b_g is None else b_g,
            "norm_w_soft": np.ones(dv) if norm_w_soft is None else norm_w_soft,
            "norm_w_lin": np.ones(dv) if norm_w_lin is None else norm_w_lin}
    return {n: torch.tensor(np.asarray(a, dtype=np.float64), requires_grad=True) for n, a in vals.items()}


def backward(q, k, v, g, beta, w_g, b_g, sel, dout, *, norm_w_soft=None, norm_w_lin=None, chunk=64,
             scale=0.0, eps=1e-6, prefix_k=None, prefix_v=None, state0=None, w_s=None, b_s=None):
    """Gradients of <dout, out> at selection `sel`, float64 numpy arrays named
    as the inputs (dq, dk, dv [B, H, L, d]; dg, dbeta [B, H, L]; dw_g [H, d];
    db_g [H]; dnorm_w_soft, dnorm_w_lin [d]); also the forward's out, o_s, o_l.
    prefix_k, prefix_v, state0: as for forward_torch (constants).
    With w_s [H, 2, 2d] (and b_s [H, 2], zero if absent): the BWD-2
    surrogate (forward_st), which adds dw_s, db_s and the score layer's
    share of dq, dk."""
    x = inputs64(q, k, v, g, beta, w_g, b_g, norm_w_soft, norm_w_lin)
    kw = dict(chunk=chunk, scale=scale, eps=eps, prefix_k=prefix_k, prefix_v=prefix_v, state0=state0)
    names = NAMES
    if w_s is not None:
        H = np.shape(w_s)[0]
        x["w_s"] = torch.tensor(np.asarray(w_s, np.float64), requires_grad=True)
        x["b_s"] = torch.tensor(np.zeros((H, 2)) if b_s is None else np.asarray(b_s, np.float64),
                                requires_grad=True)
        names = NAMES + ("w_s", "b_s")
        out, o_s, o_l = forward_st(x, np.asarray(sel), **kw)
    else:
        out, o_s, o_l = forward_torch(x, np.asarray(sel), **kw)
    grads = torch.autograd.grad(out, [x[n] for n in names], torch.as_tensor(np.asarray(dout, np.float64)))
    res = {"d" + n: gr.detach().numpy() for n, gr in zip(names, grads)}
    res.update(out=out.detach().numpy(), o_s=o_s.detach().numpy(), o_l=o_l.detach().numpy())
    return res

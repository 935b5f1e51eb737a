"""fp64 CPU oracle of the NAtS-L hybrid attention layer forward.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the library product
never does.  It wraps ``nats_oracle.cpp`` (plain C++17, float64, one thread per
(batch, head)) through ctypes.  It shares no code with the CUDA path.

Every function follows "Neural Attention Search Linear (NAtS-L)", technical
summary, section "Kernmechanismen", items 1, 3 and 4; the readings taken where
the page is silent carry the names CONV-1 ... CONV-15, DEC-1 and BWD-1
(each restated where it is used).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nats_oracle.cpp")
_LIB = os.path.join(_HERE, "libnats_oracle.so")
_lock = threading.Lock()
_lib = None


class _Dims(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("L", ctypes.c_int32),
        ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("chunk", ctypes.c_int32),
        ("scale", ctypes.c_double), ("eps", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (no GPU needed).  Returns the library path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            lib.nats_oracle_select.argtypes = [ctypes.POINTER(_Dims), P, P, P, P, P, P, ctypes.c_int32]
            lib.nats_oracle_select.restype = ctypes.c_int
            lib.nats_oracle_forward.argtypes = [ctypes.POINTER(_Dims)] + [P] * 13 + [
                ctypes.c_int32, P, P, P, P, P, P, P, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]
            lib.nats_oracle_forward.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f32(x):
    if x is None:
        return None
    return np.ascontiguousarray(x, dtype=np.float32)


def _ptr(x):
    return None if x is None else ctypes.c_void_p(x.ctypes.data)


def _dims(B, H, L, dk, dv, chunk, scale, eps):
    return _Dims(B, H, L, dk, dv, chunk, float(scale), float(eps))


def select(q, k, w_s, b_s=None, chunk: int = 64, threads: int = 0):
    """Score-layer selection for every (b, h).

    q, k: [B, H, L, dk]; w_s: [H, 2, 2dk]; b_s: [H, 2] or None.
    Returns (sel uint8 [B, H, N] with 0 = softmax, 1 = Gated DeltaNet,
    scores float64 [B, H, N, 2]).
    """
    lib = _load()
    q, k, w_s, b_s = _f32(q), _f32(k), _f32(w_s), _f32(b_s)
    B, H, L, dk = q.shape
    N = (L + chunk - 1) // chunk
    sel = np.zeros((B, H, N), np.uint8)
    scores = np.zeros((B, H, N, 2), np.float64)
    d = _dims(B, H, L, dk, dk, chunk, 0.0, 1e-6)
    rc = lib.nats_oracle_select(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(w_s), _ptr(b_s),
                                _ptr(sel), _ptr(scores), int(threads))
    if rc != 0:
        raise RuntimeError(f"nats_oracle_select failed ({rc})")
    return sel, scores


def forward(q, k, v, g, beta, w_s, b_s, w_g, b_g=None, *, chunk: int = 64, scale: float = 0.0,
            eps: float = 1e-6, norm_w_soft=None, norm_w_lin=None, sel_in=None, heads=None,
            rows=None, outputs=("sel", "scores", "o_s", "o_l", "out", "state"), threads: int = 0):
    """Layer forward in float64.

    Shapes: q, k [B, H, L, dk]; v [B, H, L, dv]; g, beta [B, H, L]; w_s [H, 2, 2dk];
    b_s [H, 2]; w_g [H, dk]; b_g [H]; norm weights [dv]; sel_in [B, H, N] uint8.
    heads: iterable of (b, h) pairs or flat indices (default: all, in order).
    rows: optional [L] bool mask of the rows whose softmax output and merged
    output are computed (others are NaN).
    Returns a dict with the requested outputs, each packed over the listed
    heads: sel [n, N], scores [n, N, 2], o_s / o_l / out [n, L, dv], state
    [n, dv, dk]; plus "threads" (threads used).
    """
    lib = _load()
    q, k, v, g, beta = _f32(q), _f32(k), _f32(v), _f32(g), _f32(beta)
    w_s, b_s, w_g, b_g = _f32(w_s), _f32(b_s), _f32(w_g), _f32(b_g)
    nws, nwl = _f32(norm_w_soft), _f32(norm_w_lin)
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    N = (L + chunk - 1) // chunk
    if heads is None:
        flat = np.arange(B * H, dtype=np.int32)
    else:
        flat = np.array([h if np.isscalar(h) else h[0] * H + h[1] for h in heads], dtype=np.int32)
    n = len(flat)
    res = {}
    want = set(outputs)
    res_sel = np.zeros((n, N), np.uint8) if "sel" in want else None
    res_scores = np.zeros((n, N, 2), np.float64) if "scores" in want else None
    fill = np.nan if rows is not None else 0.0
    res_os = np.full((n, L, dv), fill) if "o_s" in want else None
    res_ol = np.zeros((n, L, dv)) if "o_l" in want else None
    res_out = np.full((n, L, dv), fill) if "out" in want else None
    res_state = np.zeros((n, dv, dk)) if "state" in want else None
    sel_arr = None if sel_in is None else np.ascontiguousarray(sel_in, np.uint8).reshape(B * H, N)
    rows_arr = None if rows is None else np.ascontiguousarray(rows, np.uint8).reshape(L)
    used = ctypes.c_int32(0)
    d = _dims(B, H, L, dk, dv, chunk, scale, eps)
    rc = lib.nats_oracle_forward(
        ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(w_s), _ptr(b_s),
        _ptr(w_g), _ptr(b_g), _ptr(nws), _ptr(nwl), _ptr(sel_arr), _ptr(flat), n, _ptr(rows_arr),
        _ptr(res_sel), _ptr(res_scores), _ptr(res_os), _ptr(res_ol), _ptr(res_out),
        _ptr(res_state), int(threads), ctypes.byref(used))
    if rc != 0:
        raise RuntimeError(f"nats_oracle_forward failed ({rc})")
    for name, arr in (("sel", res_sel), ("scores", res_scores), ("o_s", res_os), ("o_l", res_ol),
                      ("out", res_out), ("state", res_state)):
        if arr is not None:
            res[name] = arr
    res["threads"] = used.value
    return res


def forward_inputs(inp, **kw):
    """forward() on a gen.NatsInputs workload."""
    return forward(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.w_s, inp.b_s, inp.w_g, inp.b_g,
                   chunk=inp.chunk, **kw)


def select_inputs(inp, threads: int = 0):
    """select() on a gen.NatsInputs workload."""
    return select(inp.q, inp.k, inp.w_s, inp.b_s, chunk=inp.chunk, threads=threads)


def _bf16(a):
    """Round to the nearest bf16 value (ties to even), returned as float64.

    The value goes through float32 first (round to nearest), then keeps the
    top 16 bits of its encoding with round-to-nearest-even on the rest."""
    f = np.ascontiguousarray(np.asarray(a, np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def _softplus(z):
    return np.where(z > 20.0, z, np.log1p(np.exp(np.minimum(z, 20.0))))


def project(x, w_qkv, w_ab, heads, *, b_a=None, a_scale=None, b_b=None):
    """Inputs of the layer from hidden states x [B, L, hidden] (fp64 products).

    The projections are not spelled out by the pages ("Kernmechanismen"
    item 4 only says the merge weights come from projections of the query);
    the reading is the plain Gated DeltaNet form:
      [q | k' | v] = bf16(x W_qkv), head h at columns h d .. h d + d - 1;
      k = bf16(k' / |k'|) per head (a zero k' stays zero);
      [a | b] = x W_ab;  g = -a_scale softplus(a + b_a);  beta = sigmoid(b + b_b).
    Returns q, k, v [B, H, L, d] and g, beta [B, H, L] (float64)."""
    x = np.asarray(x, np.float64)
    B, L, hidden = x.shape
    H = int(heads)
    P = x.reshape(B * L, hidden) @ np.asarray(w_qkv, np.float64)
    d = P.shape[1] // (3 * H)
    P = P.reshape(B, L, 3, H, d).transpose(2, 0, 3, 1, 4)  # part, B, H, L, d
    q, kr, v = _bf16(P[0]), _bf16(P[1]), _bf16(P[2])
    nrm = np.sqrt((kr * kr).sum(-1, keepdims=True))
    k = _bf16(np.where(nrm > 0, kr / np.where(nrm > 0, nrm, 1.0), 0.0))
    AB = (x.reshape(B * L, hidden) @ np.asarray(w_ab, np.float64)).reshape(B, L, 2, H).transpose(2, 0, 3, 1)
    zero = np.zeros(H)
    b_a = zero if b_a is None else np.asarray(b_a, np.float64)
    b_b = zero if b_b is None else np.asarray(b_b, np.float64)
    a_scale = np.ones(H) if a_scale is None else np.asarray(a_scale, np.float64)
    g = -a_scale[None, :, None] * _softplus(AB[0] + b_a[None, :, None])
    beta = 1.0 / (1.0 + np.exp(-(AB[1] + b_b[None, :, None])))
    return q, k, v, g, beta


def forward_x(x, w_qkv, w_ab, w_s, b_s, w_g, b_g, w_o, heads, *, b_a=None, a_scale=None, b_b=None,
              threads: int = 0):
    """The layer with its projections, float64: y = bf16(o_flat W_o) where o is
    the layer output (rounded to bf16, as the layer emits it) with the heads of
    a token side by side.  Returns {"y": [B, L, hidden], "sel": [B, H, N],
    "scores": [B, H, N, 2], "q", "k", "v", "g", "beta", "o"}."""
    q, k, v, g, beta = project(x, w_qkv, w_ab, heads, b_a=b_a, a_scale=a_scale, b_b=b_b)
    B, H, L, d = q.shape
    r = forward(q, k, v, g, beta, w_s, b_s, w_g, b_g, outputs=("sel", "scores", "out"), threads=threads)
    o = _bf16(r["out"]).reshape(B, H, L, d)
    of = o.transpose(0, 2, 1, 3).reshape(B * L, H * d)
    y = _bf16(of @ np.asarray(w_o, np.float64)).reshape(B, L, -1)
    N = r["sel"].shape[-1]
    return {"y": y, "sel": r["sel"].reshape(B, H, N), "scores": r["scores"].reshape(B, H, N, 2),
            "q": q, "k": k, "v": v, "g": g, "beta": beta, "o": o}


class Decoder:
    """The same layer in decode mode, one token per step, in float64.

    "Neural Attention Search Linear (NAtS-L)", technical summary,
    "Kernmechanismen" items 1, 3 and 4, read token by token (the prefill
    oracle's readings CONV-1 ... CONV-12 hold, plus the decode reading DEC-1):

    * every new token is appended to the keys / values of its chunk and sees
      the retained keys / values (those of earlier softmax chunks) plus its
      own chunk up to itself;
    * the Gated DeltaNet state takes the token's update at once (the
      pseudo-update) and the readout uses it;
    * when a chunk is complete its score (mean of [q; k] over the chunk
      through the linear score layer, ties to softmax) decides: softmax keeps
      the chunk's keys / values and returns the state to the chunk start;
      Gated DeltaNet keeps the state and drops the chunk's keys / values.

    Run from an empty state over a whole sequence, it reproduces ``forward``.
    """

    def __init__(self, B, H, dk, dv, w_s, b_s, w_g, b_g=None, *, chunk: int = 64, scale: float = 0.0,
                 eps: float = 1e-6, norm_w_soft=None, norm_w_lin=None):
        self.B, self.H, self.dk, self.dv, self.C = B, H, dk, dv, chunk
        self.scale = scale if scale > 0 else 1.0 / np.sqrt(dk)
        self.eps = eps
        self.w_s = np.asarray(w_s, np.float64).reshape(H, 2, 2 * dk)
        self.b_s = np.zeros((H, 2)) if b_s is None else np.asarray(b_s, np.float64).reshape(H, 2)
        self.w_g = np.asarray(w_g, np.float64).reshape(H, dk)
        self.b_g = np.zeros(H) if b_g is None else np.asarray(b_g, np.float64).reshape(H)
        self.nws = np.ones(dv) if norm_w_soft is None else np.asarray(norm_w_soft, np.float64)
        self.nwl = np.ones(dv) if norm_w_lin is None else np.asarray(norm_w_lin, np.float64)
        self.S = np.zeros((B, H, dv, dk))   # state after the last token
        self.S0 = np.zeros((B, H, dv, dk))  # state at the start of the current chunk
        self.kv_k = [[np.zeros((0, dk)) for _ in range(H)] for _ in range(B)]  # retained
        self.kv_v = [[np.zeros((0, dv)) for _ in range(H)] for _ in range(B)]
        self.ck = np.zeros((B, H, chunk, dk))  # current chunk
        self.cv = np.zeros((B, H, chunk, dv))
        self.psum = np.zeros((B, H, 2 * dk))  # sum of [q; k] over the current chunk
        self.t = 0
        self.sel = [[[] for _ in range(H)] for _ in range(B)]  # selection of each completed chunk

    def _rms(self, o, w):
        return o / np.sqrt(np.mean(o * o) + self.eps) * w

    def step(self, q, k, v, g, beta):
        """One token for every (b, h): q, k [B, H, dk], v [B, H, dv], g, beta [B, H].
        Returns (out, o_s, o_l), each [B, H, dv]; completed chunks append to ``sel``."""
        q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
        g, beta = np.asarray(g, np.float64), np.asarray(beta, np.float64)
        B, H, C = self.B, self.H, self.C
        p = self.t % C
        out = np.zeros((B, H, self.dv))
        o_s = np.zeros((B, H, self.dv))
        o_l = np.zeros((B, H, self.dv))
        for b in range(B):
            for h in range(H):
                qt, kt, vt = q[b, h], k[b, h], v[b, h]
                self.ck[b, h, p], self.cv[b, h, p] = kt, vt
                # Gated DeltaNet: S <- a S (I - beta k k^T) + beta v k^T, readout with the new S
                a, bt = np.exp(g[b, h]), beta[b, h]
                S = self.S[b, h]
                S = a * S - a * bt * np.outer(S @ kt, kt) + bt * np.outer(vt, kt)
                self.S[b, h] = S
                o_l[b, h] = S @ (qt * self.scale)
                # softmax over the retained keys and this chunk up to the token
                K = np.concatenate([self.kv_k[b][h], self.ck[b, h, :p + 1]])
                V = np.concatenate([self.kv_v[b][h], self.cv[b, h, :p + 1]])
                lg = (K @ qt) * self.scale
                e = np.exp(lg - lg.max())
                o_s[b, h] = (e / e.sum()) @ V
                # per-branch RMSNorm and the query-gated sum
                w = 1.0 / (1.0 + np.exp(-(qt @ self.w_g[h] + self.b_g[h])))
                out[b, h] = w * self._rms(o_s[b, h], self.nws) + (1 - w) * self._rms(o_l[b, h], self.nwl)
                self.psum[b, h] += np.concatenate([qt, kt])
                if p == C - 1:
                    s = self.w_s[h] @ (self.psum[b, h] / C) + self.b_s[h]
                    sel = 0 if s[0] >= s[1] else 1
                    self.sel[b][h].append(sel)
                    if sel == 0:  # softmax: keep the chunk's keys / values, roll the state back
                        self.kv_k[b][h] = np.concatenate([self.kv_k[b][h], self.ck[b, h]])
                        self.kv_v[b][h] = np.concatenate([self.kv_v[b][h], self.cv[b, h]])
                        self.S[b, h] = self.S0[b, h]
                    else:  # Gated DeltaNet: commit the state
                        self.S0[b, h] = self.S[b, h]
                    self.psum[b, h] = 0.0
        self.t += 1
        return out, o_s, o_l

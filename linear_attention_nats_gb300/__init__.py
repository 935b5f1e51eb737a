"""libnats: NAtS-L token-level hybrid attention layer forward on GB300 (sm_103a).

Thin torch-facing binding of the C ABI in include/nats.h.  Tensors must be
CUDA tensors; work is enqueued on the current torch CUDA stream (or the one
given).  The functions here only marshal arguments: selection, both branches
and the merge all run in libnats' CUDA kernels.
"""

from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _native
from ._native import NATS_BF16, NATS_F32, NatsError, check, dims  # noqa: F401

__all__ = ["select", "hybrid_fwd", "hybrid_fwd_x", "nha_fwd", "DecodeState", "decode_step", "workspace_size", "NatsError",
           "dims", "NATS_BF16", "NATS_F32"]


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return NATS_BF16
    if t.dtype == torch.float32:
        return NATS_F32
    raise TypeError(f"unsupported dtype {t.dtype}; use bfloat16 or float32")


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _req(t: Optional[torch.Tensor], name: str, dtype=None, shape=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def check_workspace(dm, workspace, stream=None) -> None:
    """Synchronise and raise NatsError if a kernel of the last call gave up."""
    check(_native.lib.nats_workspace_check(ctypes.byref(dm), _p(workspace), _stream(stream)),
          "nats_workspace_check")


def workspace_size(B: int, H: int, L: int, d: int, dtype=NATS_BF16) -> int:
    """Bytes of workspace hybrid_fwd needs (0 for unsupported sizes)."""
    dm = dims(B, H, L, d, dtype)
    return int(_native.lib.nats_workspace_size(ctypes.byref(dm)))


def select(q, k, w_s, b_s=None, *, scores: bool = False, stream=None):
    """Chunk selection: uint8 [B, H, L/64] (0 softmax, 1 Gated DeltaNet)."""
    _req(q, "q")
    B, H, L, d = q.shape
    _req(k, "k", q.dtype, q.shape)
    _req(w_s, "w_s", torch.float32, (H, 2, 2 * d))
    _req(b_s, "b_s", torch.float32, (H, 2))
    N = L // 64
    sel = torch.empty((B, H, N), dtype=torch.uint8, device=q.device)
    sc = torch.empty((B, H, N, 2), dtype=torch.float32, device=q.device) if scores else None
    dm = dims(B, H, L, d, _dtype_code(q))
    check(_native.lib.nats_select(ctypes.byref(dm), _p(q), _p(k), _p(w_s), _p(b_s), _p(sel), _p(sc),
                                  _stream(stream)), "nats_select")
    return (sel, sc) if scores else sel


def _streams_of(side_stream):
    """nats_streams for a torch.cuda.Stream (fork / join events made here) or
    "serial" (everything in order on the call's stream), and the events,
    which the caller keeps alive until the call has been enqueued."""
    streams = _native.Streams()
    ev = []
    if side_stream != "serial":
        ev = [torch.cuda.Event(), torch.cuda.Event()]
        for e in ev:  # materialise the event handles
            e.record(side_stream)
        streams.side, streams.fork, streams.join = side_stream.cuda_stream, ev[0].cuda_event, ev[1].cuda_event
    return streams, ev


def hybrid_fwd(q, k, v, g, beta, w_s, b_s, w_g, b_g=None, *, norm_w_soft=None, norm_w_lin=None,
               sel_in=None, scale: float = 0.0, eps: float = 1e-6, out=None, workspace=None,
               return_sel: bool = False, return_state: bool = False,
               return_branches: bool = False, return_lse: bool = False, check_errors: bool = False,
               stream=None, profile=None, side_stream=None):
    """NAtS-L hybrid attention layer forward (nats_hybrid_fwd; with `profile`,
    a _native.Profile, nats_hybrid_fwd_profiled; with `side_stream` or
    `return_lse`, nats_hybrid_fwd_streams).

    side_stream: a torch.cuda.Stream for the softmax branch (fork / join
    events are made here), or the string "serial" for both branches in order
    on `stream`; None uses the library's per-device side stream.
    return_lse (bf16 layers): also return "lse" ([B, H, L] fp32), the softmax
    branch's row statistic that hybrid_bwd(lse=...) reuses.

    q, k, v: [B, H, L, d] bf16 or fp32 (same dtype); g, beta: fp32 [B, H, L];
    w_s: fp32 [H, 2, 2d]; b_s: fp32 [H, 2] or None; w_g: fp32 [H, d];
    b_g: fp32 [H] or None; norm weights fp32 [d] or None; sel_in: uint8
    [B, H, L/64] or None.  Returns `out` alone, or a dict with "out" and the
    requested "sel", "state" ([B, H, d, d] fp32), "o_soft", "o_lin".
    check_errors=True synchronises and raises if a kernel gave up on a bounded wait.
    """
    _req(q, "q")
    B, H, L, d = q.shape
    N = L // 64
    for name, t in (("k", k), ("v", v)):
        _req(t, name, q.dtype, q.shape)
    _req(g, "g", torch.float32, (B, H, L))
    _req(beta, "beta", torch.float32, (B, H, L))
    _req(w_s, "w_s", torch.float32, (H, 2, 2 * d))
    _req(b_s, "b_s", torch.float32, (H, 2))
    _req(w_g, "w_g", torch.float32, (H, d))
    _req(b_g, "b_g", torch.float32, (H,))
    _req(norm_w_soft, "norm_w_soft", torch.float32, (d,))
    _req(norm_w_lin, "norm_w_lin", torch.float32, (d,))
    _req(sel_in, "sel_in", torch.uint8, (B, H, N))
    dt = _dtype_code(q)
    dm = dims(B, H, L, d, dt, scale, eps)
    if out is None:
        out = torch.empty_like(q)
    _req(out, "out", q.dtype, q.shape)
    need = int(_native.lib.nats_workspace_size(ctypes.byref(dm)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _req(workspace, "workspace", torch.uint8)
    dev = q.device
    sel = torch.empty((B, H, N), dtype=torch.uint8, device=dev) if return_sel else None
    state = torch.empty((B, H, d, d), dtype=torch.float32, device=dev) if return_state else None
    o_soft = torch.empty((B, H, L, d), dtype=torch.float32, device=dev) if return_branches else None
    o_lin = torch.empty((B, H, L, d), dtype=torch.float32, device=dev) if return_branches else None
    lse = torch.empty((B, H, L), dtype=torch.float32, device=dev) if return_lse else None
    args = (ctypes.byref(dm), _p(q), _p(k), _p(v), _p(g), _p(beta), _p(w_s), _p(b_s), _p(w_g), _p(b_g),
            _p(norm_w_soft), _p(norm_w_lin), _p(sel_in), _p(out), _p(sel), _p(state), _p(o_soft),
            _p(o_lin))
    tail = (_p(workspace), ctypes.c_size_t(workspace.numel()), _stream(stream))
    if side_stream is not None or return_lse:
        streams, _events = _streams_of(side_stream) if side_stream is not None else (None, [])
        prof = ctypes.byref(profile) if profile is not None else None
        check(_native.lib.nats_hybrid_fwd_streams(*args, _p(lse), *tail,
                                                  ctypes.byref(streams) if streams is not None else None, prof),
              "nats_hybrid_fwd_streams")
    elif profile is None:
        check(_native.lib.nats_hybrid_fwd(*args, *tail), "nats_hybrid_fwd")
    else:
        check(_native.lib.nats_hybrid_fwd_profiled(*args, *tail, ctypes.byref(profile)), "nats_hybrid_fwd_profiled")
    if check_errors:
        check_workspace(dm, workspace, stream)
    if not (return_sel or return_state or return_branches or return_lse):
        return out
    res = {"out": out}
    if return_lse:
        res["lse"] = lse
    if return_sel:
        res["sel"] = sel
    if return_state:
        res["state"] = state
    if return_branches:
        res["o_soft"] = o_soft
        res["o_lin"] = o_lin
    return res


def hybrid_fwd_x(x, w_qkv, w_ab, w_s, b_s, w_g, b_g=None, *, heads: int, b_a=None, a_scale=None, b_b=None,
                 w_o, y=None, workspace=None, return_sel: bool = False, check_errors: bool = False, stream=None):
    """The layer with its projections: x [B, L, hidden] bf16 -> y [B, L, hidden] bf16.

    w_qkv: bf16 [hidden, 3 H d]; w_ab: bf16 [hidden, 2 H]; b_a, a_scale, b_b:
    fp32 [H] or None; w_s, b_s, w_g, b_g as for hybrid_fwd; w_o: bf16
    [H d, hidden].  The definitions are those of nats_hybrid_fwd_x in
    include/nats.h.  Returns y, or {"y": y, "sel": sel} with return_sel.
    check_errors synchronises and raises if a bounded device wait expired."""
    _req(x, "x", torch.bfloat16)
    B, L, hidden = x.shape
    H = int(heads)
    d = w_qkv.shape[1] // (3 * H)
    N = L // 64
    _req(w_qkv, "w_qkv", torch.bfloat16, (hidden, 3 * H * d))
    _req(w_ab, "w_ab", torch.bfloat16, (hidden, 2 * H))
    for name, t in (("b_a", b_a), ("a_scale", a_scale), ("b_b", b_b), ("b_g", b_g)):
        _req(t, name, torch.float32, (H,))
    _req(w_s, "w_s", torch.float32, (H, 2, 2 * d))
    _req(b_s, "b_s", torch.float32, (H, 2))
    _req(w_g, "w_g", torch.float32, (H, d))
    _req(w_o, "w_o", torch.bfloat16, (H * d, hidden))
    dm = dims(B, H, L, d, NATS_BF16)
    if y is None:
        y = torch.empty((B, L, hidden), dtype=torch.bfloat16, device=x.device)
    _req(y, "y", torch.bfloat16, (B, L, hidden))
    need = int(_native.lib.nats_x_workspace_size(ctypes.byref(dm), hidden))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    _req(workspace, "workspace", torch.uint8)
    sel = torch.empty((B, H, N), dtype=torch.uint8, device=x.device) if return_sel else None
    check(_native.lib.nats_hybrid_fwd_x(
        ctypes.byref(dm), hidden, _p(x), _p(w_qkv), _p(w_ab), _p(b_a), _p(a_scale), _p(b_b), _p(w_s), _p(b_s),
        _p(w_g), _p(b_g), _p(w_o), _p(y), _p(sel), _p(workspace), ctypes.c_size_t(workspace.numel()),
        _stream(stream)), "nats_hybrid_fwd_x")
    if check_errors:
        check(_native.lib.nats_x_workspace_check(ctypes.byref(dm), hidden, _p(workspace), _stream(stream)),
              "nats_x_workspace_check")
    return {"y": y, "sel": sel} if return_sel else y


def hybrid_bwd(q, k, v, g, beta, w_g, b_g, sel, o_soft, o_lin, dout, *, norm_w_soft=None, norm_w_lin=None,
               scale: float = 0.0, eps: float = 1e-6, weight_grads: bool = True, workspace=None, stream=None,
               profile=None, side_stream=None, lse=None):
    """Backward pass of the layer at the forward's selection
    (nats_hybrid_bwd_streams; `profile`, a _native.Profile, or None).

    side_stream: a torch.cuda.Stream for the Gated DeltaNet state work of a
    bf16 layer (fork / join events are made here), or "serial" for every
    kernel in order on `stream`; None uses the library's per-device side
    stream.
    lse: the forward's "lse" (hybrid_fwd(..., return_lse=True)) for the same
    inputs; a bf16 backward then reads the softmax row statistic instead of
    recomputing it.

    sel, o_soft, o_lin: the forward's selection and branch outputs
    (hybrid_fwd(..., return_sel=True, return_branches=True)); dout like q.
    Returns a dict of fp32 gradients: dq, dk, dv [B, H, L, d]; dg, dbeta
    [B, H, L]; and, with weight_grads, dw_g [H, d], db_g [H], dnorm_w_soft,
    dnorm_w_lin [d].  The score layer (W_s, b_s) gets none: the selection is
    an argmax.
    """
    _req(q, "q")
    B, H, L, d = q.shape
    N = L // 64
    for name, t in (("k", k), ("v", v), ("dout", dout)):
        _req(t, name, q.dtype, q.shape)
    _req(g, "g", torch.float32, (B, H, L))
    _req(beta, "beta", torch.float32, (B, H, L))
    _req(w_g, "w_g", torch.float32, (H, d))
    _req(b_g, "b_g", torch.float32, (H,))
    _req(norm_w_soft, "norm_w_soft", torch.float32, (d,))
    _req(norm_w_lin, "norm_w_lin", torch.float32, (d,))
    _req(sel, "sel", torch.uint8, (B, H, N))
    _req(o_soft, "o_soft", torch.float32, (B, H, L, d))
    _req(o_lin, "o_lin", torch.float32, (B, H, L, d))
    _req(lse, "lse", torch.float32, (B, H, L))
    dm = dims(B, H, L, d, _dtype_code(q), scale, eps)
    need = int(_native.lib.nats_bwd_workspace_size(ctypes.byref(dm)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _req(workspace, "workspace", torch.uint8)
    f32 = dict(dtype=torch.float32, device=q.device)
    res = {"dq": torch.empty((B, H, L, d), **f32), "dk": torch.empty((B, H, L, d), **f32),
           "dv": torch.empty((B, H, L, d), **f32), "dg": torch.empty((B, H, L), **f32),
           "dbeta": torch.empty((B, H, L), **f32)}
    if weight_grads:
        res.update(dw_g=torch.empty((H, d), **f32), db_g=torch.empty((H,), **f32),
                   dnorm_w_soft=torch.empty((d,), **f32), dnorm_w_lin=torch.empty((d,), **f32))
    streams, _events = _streams_of(side_stream) if side_stream is not None else (None, [])
    check(_native.lib.nats_hybrid_bwd_streams(
        ctypes.byref(dm), _p(q), _p(k), _p(v), _p(g), _p(beta), _p(w_g), _p(b_g), _p(norm_w_soft),
        _p(norm_w_lin), _p(sel), _p(o_soft), _p(o_lin), _p(lse), _p(dout), _p(res["dq"]), _p(res["dk"]), _p(res["dv"]),
        _p(res["dg"]), _p(res["dbeta"]), _p(res.get("dw_g")), _p(res.get("db_g")), _p(res.get("dnorm_w_soft")),
        _p(res.get("dnorm_w_lin")), _p(workspace), ctypes.c_size_t(workspace.numel()), _stream(stream),
        ctypes.byref(streams) if streams is not None else None,
        ctypes.byref(profile) if profile is not None else None), "nats_hybrid_bwd")
    return res


def score_bwd(q, k, w_s, b_s, sel, out, dout, grads, *, stream=None):
    """The score layer's gradient under the straight-through surrogate
    (nats_score_bwd, reading BWD-2), after hybrid_bwd: `grads` is
    hybrid_bwd's dict; its dq, dk gain the score layer's share in place and
    it gains dw_s [H, 2, 2d] and db_s [H, 2].  out: the forward's output."""
    _req(q, "q")
    B, H, L, d = q.shape
    for name, t in (("k", k), ("out", out), ("dout", dout)):
        _req(t, name, q.dtype, q.shape)
    _req(w_s, "w_s", torch.float32, (H, 2, 2 * d))
    _req(b_s, "b_s", torch.float32, (H, 2))
    _req(sel, "sel", torch.uint8, (B, H, L // 64))
    for name in ("dq", "dk"):
        _req(grads[name], name, torch.float32, (B, H, L, d))
    f32 = dict(dtype=torch.float32, device=q.device)
    grads["dw_s"] = torch.empty((H, 2, 2 * d), **f32)
    grads["db_s"] = torch.empty((H, 2), **f32)
    check(_native.lib.nats_score_bwd(
        ctypes.byref(dims(B, H, L, d, _dtype_code(q))), _p(q), _p(k), _p(w_s), _p(b_s), _p(sel), _p(out), _p(dout),
        _p(grads["dq"]), _p(grads["dk"]), _p(grads["dw_s"]), _p(grads["db_s"]), _stream(stream)), "nats_score_bwd")
    return grads


class DecodeState:
    """Device state of the layer in decode mode (nats_decode_state): the
    Gated DeltaNet state S and its chunk-start copy S0 (fp32 [B, H, d, d]), the
    current chunk's keys / values ck, cv ([B, H, 64, d]), the running sum of
    [q; k] over the chunk (fp32 [B, H, 2 d]), the retained keys / values kv_k,
    kv_v ([B, H, cap, d]) and their count n_kv (int32 [B, H]), and the error
    flag err (int32 [1], set by a step whose bounded wait for its copies ran
    out; `check()` reads it).  New states are empty (zeros)."""

    def __init__(self, B: int, H: int, d: int, cap: int, dtype=torch.bfloat16, device="cuda"):
        z = dict(device=device)
        self.B, self.H, self.d, self.cap, self.dtype = B, H, d, int(cap), dtype
        self.S = torch.zeros((B, H, d, d), dtype=torch.float32, **z)
        self.S0 = torch.zeros((B, H, d, d), dtype=torch.float32, **z)
        self.ck = torch.zeros((B, H, 64, d), dtype=dtype, **z)
        self.cv = torch.zeros((B, H, 64, d), dtype=dtype, **z)
        self.psum = torch.zeros((B, H, 2 * d), dtype=torch.float32, **z)
        self.kv_k = torch.zeros((B, H, self.cap, d), dtype=dtype, **z)
        self.kv_v = torch.zeros((B, H, self.cap, d), dtype=dtype, **z)
        self.n_kv = torch.zeros((B, H), dtype=torch.int32, **z)
        self.err = torch.zeros((1,), dtype=torch.int32, **z)

    def c_struct(self) -> _native.DecodeState:
        return _native.DecodeState(self.S.data_ptr(), self.S0.data_ptr(), self.ck.data_ptr(), self.cv.data_ptr(),
                                   self.psum.data_ptr(), self.kv_k.data_ptr(), self.kv_v.data_ptr(),
                                   self.n_kv.data_ptr(), self.cap, self.err.data_ptr())

    def check(self) -> None:
        """Raises if a step since the state was made gave up waiting for its
        key / value copies (synchronises with the device)."""
        if int(self.err.item()) != 0:
            raise _native.NatsError(8, "nats_decode_step (a bounded wait ran out)")


def decode_step(state: DecodeState, t: int, q, k, v, g, beta, w_s, b_s, w_g, b_g=None, *, norm_w_soft=None,
                norm_w_lin=None, out=None, sel_out=None, return_branches: bool = False, scale: float = 0.0,
                eps: float = 1e-6, stream=None):
    """One decode step at position t: q, k, v [B, H, d] (the state's dtype), g,
    beta fp32 [B, H]; weights as for hybrid_fwd.  Updates `state` in place and
    returns out [B, H, d] (or {"out", "o_s", "o_l"} with return_branches).
    sel_out (uint8 [B, H]) receives the chunk's selection when t completes a
    chunk.  The definitions are those of nats_decode_step in include/nats.h."""
    B, H, d = state.B, state.H, state.d
    for name, x in (("q", q), ("k", k), ("v", v)):
        _req(x, name, state.dtype, (B, H, d))
    _req(g, "g", torch.float32, (B, H))
    _req(beta, "beta", torch.float32, (B, H))
    _req(w_s, "w_s", torch.float32, (H, 2, 2 * d))
    _req(b_s, "b_s", torch.float32, (H, 2))
    _req(w_g, "w_g", torch.float32, (H, d))
    _req(b_g, "b_g", torch.float32, (H,))
    if out is None:
        out = torch.empty((B, H, d), dtype=state.dtype, device=q.device)
    _req(out, "out", state.dtype, (B, H, d))
    _req(sel_out, "sel_out", torch.uint8, (B, H))
    o_s = o_l = None
    if return_branches:
        o_s = torch.empty((B, H, d), dtype=torch.float32, device=q.device)
        o_l = torch.empty((B, H, d), dtype=torch.float32, device=q.device)
    dm = dims(B, H, 0, d, _dtype_code(q), scale=scale, eps=eps)
    st = state.c_struct()
    check(_native.lib.nats_decode_step(
        ctypes.byref(dm), int(t), _p(q), _p(k), _p(v), _p(g), _p(beta), _p(w_s), _p(b_s), _p(w_g), _p(b_g),
        _p(norm_w_soft), _p(norm_w_lin), ctypes.byref(st), _p(out), _p(sel_out), _p(o_s), _p(o_l),
        _stream(stream)), "nats_decode_step")
    return {"out": out, "o_s": o_s, "o_l": o_l} if return_branches else out


def nha_fwd(q, k, v, log_alpha, *, window: int, scale: float = 0.0, out=None, workspace=None,
            check_errors: bool = False, stream=None):
    """Native Hybrid Attention forward (nats_nha_fwd): q, k, v [B, H, L, 128]
    bf16, log_alpha [B, H, L, 64] fp32 (log of the slot forget gate); one
    softmax over the slot memory and the window of the last `window` tokens.
    Returns out [B, H, L, 128] bf16.  The definitions are those of
    nats_nha_fwd in include/nats.h."""
    _req(q, "q", torch.bfloat16)
    B, H, L, d = q.shape
    for name, t in (("k", k), ("v", v)):
        _req(t, name, torch.bfloat16, q.shape)
    _req(log_alpha, "log_alpha", torch.float32)
    if log_alpha.dim() != 4 or tuple(log_alpha.shape[:3]) != (B, H, L):
        raise ValueError("log_alpha must be [B, H, L, slots]")
    dm = _native.nha_dims(B, H, L, d, log_alpha.shape[3], window, NATS_BF16, scale)
    if out is None:
        out = torch.empty_like(q)
    _req(out, "out", torch.bfloat16, q.shape)
    need = int(_native.lib.nats_nha_workspace_size(ctypes.byref(dm)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _req(workspace, "workspace", torch.uint8)
    check(_native.lib.nats_nha_fwd(ctypes.byref(dm), _p(q), _p(k), _p(v), _p(log_alpha), _p(out), _p(workspace),
                                   ctypes.c_size_t(workspace.numel()), _stream(stream)), "nats_nha_fwd")
    if check_errors:
        check(_native.lib.nats_nha_workspace_check(ctypes.byref(dm), _p(workspace), _stream(stream)),
              "nats_nha_workspace_check")
    return out

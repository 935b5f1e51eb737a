"""The C ABI: the library loads, exports what include/nats.h declares, and
rejects bad arguments on the host before any launch (no GPU needed)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def nat():
    from linear_attention_nats_gb300 import build as b

    b.build()
    from linear_attention_nats_gb300 import _native

    return _native


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(nats_\w+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(nat):
    declared = _declared()
    assert {"nats_select", "nats_hybrid_fwd", "nats_workspace_size", "nats_status_string"} <= declared
    assert declared == set(nat.EXPORTS)
    for name in sorted(declared):
        assert hasattr(nat.lib, name), name


def test_status_strings(nat):
    for code, name in nat.STATUS.items():
        s = nat.lib.nats_status_string(code).decode()
        assert s.startswith(name), (code, s)


def test_workspace_size(nat):
    ws = lambda *a, **k: nat.lib.nats_workspace_size(ctypes.byref(nat.dims(*a, **k)))
    assert ws(4, 16, 8192, 128) > 4 * 16 * 8192 * 128 * 4 * 2
    assert ws(1, 1, 64, 64) > 0
    assert ws(1, 1, 100, 64) == 0  # L % 64 != 0
    assert ws(1, 1, 64, 96) == 0  # unsupported head size
    # the largest TMA row coordinate, (B H N + c) d, must fit a 32-bit int
    assert ws(1, 1 << 14, 1 << 16, 128) == 0
    assert ws(1, 1 << 14, 1 << 16, 64) > 0
    assert ws(1, (1 << 14) - 1, 1 << 16, 128) > 0
    assert ws(0, 4, 256, 64) >= 0
    small, big = ws(1, 2, 256, 64), ws(2, 2, 256, 64)
    assert big > small


def _fwd(nat, dm, **ptrs):
    names = ["q", "k", "v", "g", "beta", "w_s", "b_s", "w_g", "b_g", "nws", "nwl", "sel_in", "out",
             "sel_out", "state", "o_soft", "o_lin", "ws"]
    args = [ptrs.get(n) for n in names]
    args = [None if a is None else ctypes.c_void_p(a) for a in args]
    return nat.lib.nats_hybrid_fwd(ctypes.byref(dm), *args[:17], args[17],
                                   ctypes.c_size_t(ptrs.get("ws_bytes", 1 << 40)), None)


# Fake but 256-aligned addresses: validation must reject before touching them.
A = 0x10000000
FULL = dict(q=A, k=A + 0x1000, v=A + 0x2000, g=A + 0x3000, beta=A + 0x4000, w_s=A + 0x5000,
            w_g=A + 0x6000, out=A + 0x7000, ws=A + 0x8000)


@pytest.mark.parametrize("case,code", [
    (dict(B=-1), 2), (dict(L=100), 2), (dict(d=96), 6), (dict(dtype=7), 3), (dict(chunk=32), 2),
    (dict(scale=float("nan")), 9), (dict(eps=-1.0), 9),
])
def test_shape_errors(nat, case, code):
    kw = dict(B=1, H=2, L=256, d=64, dtype=0, scale=0.0, eps=1e-6, chunk=64)
    kw.update(case)
    dm = nat.dims(kw["B"], kw["H"], kw["L"], kw["d"], kw["dtype"], kw["scale"], kw["eps"], kw["chunk"])
    assert _fwd(nat, dm, **FULL) == code
    assert nat.lib.nats_select(ctypes.byref(dm), *[ctypes.c_void_p(A)] * 3, None,
                               ctypes.c_void_p(A), None, None) == code


def test_dk_ne_dv(nat):
    dm = nat.Dims(1, 2, 256, 64, 128, 64, 0, 0.0, 1e-6)
    assert _fwd(nat, dm, **FULL) == 2


@pytest.mark.parametrize("missing", ["q", "k", "v", "g", "beta", "w_g", "out", "ws"])
def test_null_errors(nat, missing):
    dm = nat.dims(1, 2, 256, 64)
    p = dict(FULL)
    p[missing] = None
    assert _fwd(nat, dm, **p) == 1


def test_w_s_optional_only_with_override(nat):
    dm = nat.dims(1, 2, 256, 64)
    p = dict(FULL)
    p["w_s"] = None
    assert _fwd(nat, dm, **p) == 1


def test_alignment_error(nat):
    dm = nat.dims(1, 2, 256, 64)
    p = dict(FULL)
    p["v"] = A + 0x2008
    assert _fwd(nat, dm, **p) == 4


def test_workspace_too_small(nat):
    dm = nat.dims(1, 2, 256, 64)
    need = nat.lib.nats_workspace_size(ctypes.byref(dm))
    assert _fwd(nat, dm, ws_bytes=need - 1, **FULL) == 5


def test_empty_is_a_no_op(nat):
    # zero extents return NATS_OK without touching any pointer (all NULL here)
    for B, H, L in ((0, 2, 256), (1, 0, 256), (1, 2, 0)):
        assert _fwd(nat, nat.dims(B, H, L, 64)) == 0


def test_x_path_validation(nat):
    # the layer with its projections: argument checks before any launch
    dm = nat.dims(1, 2, 256, 64)
    assert nat.lib.nats_x_workspace_size(ctypes.byref(dm), 100) == 0  # hidden % 8
    assert nat.lib.nats_x_workspace_size(ctypes.byref(dm), 128) > nat.lib.nats_workspace_size(ctypes.byref(dm))
    f32 = nat.dims(1, 2, 256, 64, 1)
    null = [None] * 14
    assert nat.lib.nats_hybrid_fwd_x(ctypes.byref(f32), 128, *null, ctypes.c_size_t(0), None) == 3
    assert nat.lib.nats_hybrid_fwd_x(ctypes.byref(dm), 100, *null, ctypes.c_size_t(0), None) == 2
    assert nat.lib.nats_hybrid_fwd_x(ctypes.byref(dm), 128, *null, ctypes.c_size_t(0), None) == 1
    bad = nat.dims(1, 2, 100, 64)  # L % 64
    assert nat.lib.nats_hybrid_fwd_x(ctypes.byref(bad), 128, *null, ctypes.c_size_t(0), None) == 2


def test_decode_validation(nat):
    # the decode step: argument checks before any launch (no device memory is touched)
    dm = nat.dims(1, 2, 0, 64)
    fake = ctypes.c_void_p(256)  # 16-byte aligned, never dereferenced on these paths
    odd = ctypes.c_void_p(264)   # 8-byte aligned only
    st = nat.DecodeState(fake.value, fake.value, fake.value, fake.value, fake.value, fake.value, fake.value,
                         fake.value, 64, fake.value)
    no_err = nat.DecodeState(fake.value, fake.value, fake.value, fake.value, fake.value, fake.value, fake.value,
                             fake.value, 64, None)
    args = [fake] * 11
    tail = [fake, None, None, None, None]

    def call(d=dm, t=0, a=args, s=st, tl=tail):
        return nat.lib.nats_decode_step(ctypes.byref(d), t, *a, ctypes.byref(s) if s is not None else None, *tl)

    assert call(t=-1) == 9                       # NATS_ERR_VALUE
    assert call(t=64) == 5                       # cap 64 cannot take a second chunk: NATS_ERR_WORKSPACE
    assert call(a=[None] + args[1:]) == 1        # q NULL
    assert call(s=None) == 1                     # state NULL
    assert call(s=no_err) == 1                   # state without its error flag
    assert call(a=[odd] + args[1:]) == 4         # q misaligned: NATS_ERR_ALIGN
    bad = nat.dims(1, 2, 0, 96)
    assert call(d=bad) == 6                      # head size: NATS_ERR_UNSUPPORTED
    empty = nat.dims(0, 2, 0, 64)
    assert call(d=empty) == 0                    # nothing to do


def test_backward_validation(nat):
    # the backward pass: argument checks before any launch
    dm = nat.dims(1, 2, 128, 64)
    need = nat.lib.nats_bwd_workspace_size(ctypes.byref(dm))
    rows, dd, chunks = 2 * 128, 64 * 64, 2 * 2
    al = lambda b: (b + 255) // 256 * 256
    common = al(rows * 64 * 4) + 2 * al(rows * 4)  # d o_l, delta, lse; then d o_s (fp32 layers) or its bf16 copy
    common_f32, common = common + al(rows * 64 * 4), common + al(rows * 64 * 2)
    # fp32 layers: 2 chunk-start states, one chunk of states, one held gradient, then the two state halves'
    # per-token column sums and scalars
    f32 = nat.lib.nats_bwd_workspace_size(ctypes.byref(nat.dims(1, 2, 128, 64, nat.NATS_F32)))
    assert f32 == common_f32 + (al(chunks * dd * 4) + al(2 * 64 * dd * 4) + al(2 * dd * 4) + al(2 * rows * 2 * 64 * 4)
                            + al(2 * rows * 4 * 4))
    # bf16 layers: the compacted softmax-chunk lists, the forward's chunk factors (G, W, U^T, P, gate, o_l,
    # error flag), then the chunkwise adjoint's chunk-start states and state gradients, G, Linv and P (fp32),
    # W, Q_eff, K~ (fp16) and their scales
    assert need == common + (2 * al(chunks * 4) + al(rows * 4) + 2 * al(rows * 64 * 2) + al(rows * 64 * 2)
                             + al(rows * 4)
                             + al(rows * 64 * 2) + al(16)
                             + 2 * al(chunks * dd * 4) + al(rows * 4) + 2 * al(rows * 64 * 4)
                             + 3 * al(rows * 64 * 2) + al(chunks * 16))
    fake = ctypes.c_void_p(256)
    odd = ctypes.c_void_p(264)
    args = [fake] * 23  # q ... dnorm_w_lin, then the workspace

    def call(d=dm, a=args, ws_bytes=need):
        return nat.lib.nats_hybrid_bwd(ctypes.byref(d), *a, ctypes.c_size_t(ws_bytes), None)

    assert call(ws_bytes=need - 1) == 5           # NATS_ERR_WORKSPACE
    assert call(a=[None] + args[1:]) == 1         # q NULL
    assert call(a=args[:9] + [None] + args[10:]) == 1   # sel NULL
    assert call(a=args[:12] + [odd] + args[13:]) == 4   # dout misaligned
    assert call(a=args[:22] + [None]) == 1        # workspace NULL
    for optional in (6, 7, 8, 18, 19, 20, 21):    # b_g, norm weights, weight gradients may be NULL
        a = list(args)
        a[optional] = None
        assert call(a=a, ws_bytes=0) == 5          # passes the NULL checks, stops at the workspace
    assert call(d=nat.dims(1, 2, 100, 64)) == 2   # L % 64: NATS_ERR_SHAPE
    assert call(d=nat.dims(0, 2, 128, 64)) == 0   # nothing to do
    assert nat.lib.nats_bwd_workspace_size(ctypes.byref(nat.dims(1, 2, 100, 64))) == 0


def test_backward_streams_validation(nat):
    # nats_hybrid_bwd_streams: a second stream other than `stream` needs both
    # events (checked after the shape and pointer checks, before the workspace)
    dm = nat.dims(1, 2, 128, 64)
    need = nat.lib.nats_bwd_workspace_size(ctypes.byref(dm))
    fake = ctypes.c_void_p(256)
    args = [fake] * 24  # q ... o_lin, lse, dout ... dnorm_w_lin, the workspace

    def call(streams, d=dm, a=args, ws_bytes=1 << 40):
        return nat.lib.nats_hybrid_bwd_streams(ctypes.byref(d), *a, ctypes.c_size_t(ws_bytes), None,
                                               ctypes.byref(streams) if streams is not None else None, None)

    side = ctypes.c_void_p(0x7000).value
    for fork, join in ((None, None), (256, None), (None, 256)):
        assert call(nat.Streams(side, fork, join)) == 1                      # NATS_ERR_NULL
    assert call(nat.Streams(side, None, None), d=nat.dims(1, 2, 100, 64)) == 2  # shapes first
    assert call(nat.Streams(side, None, None), a=[None] + args[1:]) == 1      # q NULL
    # no second stream (or the caller's own): events not needed, the workspace check comes next
    for st in (nat.Streams(None, None, None), None):
        assert call(st, ws_bytes=need - 1) == 5
    assert call(nat.Streams(side, 256, 256), ws_bytes=need - 1) == 5
    assert call(nat.Streams(side, None, None), d=nat.dims(0, 2, 128, 64)) == 0  # nothing to do
    # the forward's row statistic: optional, 16-byte aligned
    assert call(None, a=args[:12] + [None] + args[13:], ws_bytes=need - 1) == 5
    assert call(None, a=args[:12] + [ctypes.c_void_p(264)] + args[13:]) == 4


def test_debug_hook_validation(nat):
    # the bounded-wait hook checks its arguments before any launch
    assert nat.lib.nats_debug_bounded_wait(None, 1000, None) == 1           # NATS_ERR_NULL
    assert nat.lib.nats_debug_bounded_wait(ctypes.c_void_p(256), 0, None) == 9  # NATS_ERR_VALUE
    assert nat.lib.nats_debug_bounded_wait(ctypes.c_void_p(256), 2 * 10**9, None) == 9
    nat.lib.nats_debug_fail_stage(-1)  # cancelling an injection is always allowed


def test_noalloc_validation_order(nat):
    """The allocation-free forward checks its arguments like nats_hybrid_fwd,
    in the same order, and only then its fixed scratch limit; all of it on
    the host, before any CUDA call."""
    P = lambda a: ctypes.c_void_p(a)
    good = [P(0x10000000)] * 5 + [P(0x10001000), None, P(0x10002000), None, None, None, None, P(0x10003000)]
    tail = [None] * 5 + [None]

    def call(dm, ptrs):
        return nat.lib.nats_hybrid_fwd_noalloc(ctypes.byref(dm), *ptrs, *tail)

    big = nat.dims(1, 16, 16384, 128)
    assert nat.lib.nats_workspace_size(ctypes.byref(big)) > nat.NOALLOC_SCRATCH_BYTES
    assert call(nat.dims(1, 1, 100, 64), good) == 2  # NATS_ERR_SHAPE
    assert call(nat.dims(0, 4, 256, 64), good) == 0  # empty problem: no-op
    no_out = list(good)
    no_out[12] = None
    assert call(big, no_out) == 1  # NATS_ERR_NULL comes before the size limit
    odd = list(good)
    odd[0] = P(0x10000008)
    assert call(big, odd) == 4  # NATS_ERR_ALIGN comes before the size limit
    assert call(big, good) == 5  # NATS_ERR_WORKSPACE
    assert nat.lib.nats_noalloc_check(ctypes.byref(big), None) == 5


def test_nha_validation(nat):
    """nats_nha_fwd rejects bad arguments on the host, before any launch."""
    P = lambda a: ctypes.c_void_p(a)
    ok_ptrs = [P(0x10000000)] * 5 + [P(0x20000000)]

    def call(dm, ptrs=ok_ptrs, nbytes=1 << 40):
        return nat.lib.nats_nha_fwd(ctypes.byref(dm), *ptrs, ctypes.c_size_t(nbytes), None)

    d = nat.nha_dims
    assert nat.lib.nats_nha_workspace_size(ctypes.byref(d(1, 2, 512))) > 0
    assert call(d(1, 2, 500)) == 2  # L % 64
    assert call(d(1, 2, 512, d=64)) == 6  # head size
    assert call(d(1, 2, 512, slots=32)) == 6  # slot count
    assert call(d(1, 2, 512, window=64)) == 6  # window not a multiple of 128 (and < L)
    assert call(d(1, 2, 512, window=-1)) == 2
    assert call(d(1, 2, 512, dtype=nat.NATS_F32)) == 3
    assert call(d(1, 2, 512, scale=float("nan"))) == 9
    assert call(d(0, 2, 512)) == 0  # empty: no-op
    assert call(d(1, 2, 512), [None] + ok_ptrs[1:]) == 1
    assert call(d(1, 2, 512), [P(0x10000004)] + ok_ptrs[1:]) == 4
    assert call(d(1, 2, 512), nbytes=16) == 5


def test_score_bwd_validation(nat):
    """nats_score_bwd rejects bad arguments on the host, before any launch."""
    P = lambda a: ctypes.c_void_p(a)
    ok = [P(0x10000000)] * 11  # q, k, w_s, b_s, sel, out, dout, dq, dk, dw_s, db_s

    def call(dm, ptrs=ok):
        return nat.lib.nats_score_bwd(ctypes.byref(dm), *ptrs, None)

    assert call(nat.dims(1, 2, 500, 128, 0)) == 2  # L % 64
    assert call(nat.dims(1, 2, 512, 96, 0)) == 6  # head size
    for i in (0, 1, 2, 4, 5, 6, 7, 8, 9, 10):  # every pointer but b_s is required
        assert call(nat.dims(1, 2, 512, 128, 0), ok[:i] + [None] + ok[i + 1:]) == 1, i
    for i in (0, 1, 5, 6, 7, 8):  # q, k, out, dout, dq, dk 16-byte aligned
        assert call(nat.dims(1, 2, 512, 128, 0), ok[:i] + [P(0x10000004)] + ok[i + 1:]) == 4, i


def test_streams_validation(nat):
    # nats_hybrid_fwd_streams: a second stream other than `stream` needs both
    # events (checked after the shape and pointer checks, before the workspace)
    dm = nat.dims(1, 2, 256, 64)
    names = ["q", "k", "v", "g", "beta", "w_s", "b_s", "w_g", "b_g", "nws", "nwl", "sel_in", "out",
             "sel_out", "state", "o_soft", "o_lin", "ws"]

    def call(dmx, streams, ws_bytes=1 << 40, lse=None, **ptrs):
        args = [None if ptrs.get(n) is None else ctypes.c_void_p(ptrs[n]) for n in names]
        return nat.lib.nats_hybrid_fwd_streams(ctypes.byref(dmx), *args[:17], lse, args[17],
                                               ctypes.c_size_t(ws_bytes), None,
                                               ctypes.byref(streams) if streams is not None else None, None)

    side = ctypes.c_void_p(0x7000).value
    for fork, join in ((None, None), (A, None), (None, A)):
        assert call(dm, nat.Streams(side, fork, join), **FULL) == 1
    assert call(nat.dims(1, 2, 100, 64), nat.Streams(side, None, None), **FULL) == 2  # shapes first
    need = nat.lib.nats_workspace_size(ctypes.byref(dm))
    # no second stream (or the caller's own): events not needed, the workspace check comes next
    for st in (nat.Streams(None, None, None), None):
        assert call(dm, st, ws_bytes=need - 1, **FULL) == 5
    assert call(dm, nat.Streams(side, A, A), ws_bytes=need - 1, **FULL) == 5
    # the saved row statistic exists for bf16 layers only
    f32 = nat.dims(1, 2, 256, 64, nat.NATS_F32)
    assert call(f32, None, lse=ctypes.c_void_p(A), **FULL) == 3
    assert call(dm, None, ws_bytes=need - 1, lse=ctypes.c_void_p(A), **FULL) == 5

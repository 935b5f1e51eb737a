"""nats_hybrid_fwd_noalloc: the entry point for callers that cannot allocate
device memory (a plugin whose host owns all device memory through its own
pool, a loop that must never block on an allocation, a plain C caller with no
allocator).  It uses a scratch array built into the library instead of a
caller workspace.  Checked through the C ABI against nats_hybrid_fwd on the
same inputs, on two calls in a row with different inputs, so that the second
call also shows that whatever the first left in the shared scratch does not
leak into its result.  This file is collected last on purpose."""

import ctypes

import numpy as np
import pytest
import torch

import gen
from gpu_util import TOL, rel_err, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nat():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from linear_attention_nats_gb300 import build

    build.build()
    from linear_attention_nats_gb300 import _native

    return _native


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _run(nat, inp, no_alloc):
    t = to_device(inp)
    B, H, L, d = inp.B, inp.H, inp.L, inp.d
    dm = nat.dims(B, H, L, d, nat.NATS_BF16 if inp.dtype == "bf16" else nat.NATS_F32)
    out = torch.empty_like(t["q"])
    sel = torch.empty((B, H, L // 64), dtype=torch.uint8, device="cuda")
    state = torch.empty((B, H, d, d), dtype=torch.float32, device="cuda")
    common = [ctypes.byref(dm), _ptr(t["q"]), _ptr(t["k"]), _ptr(t["v"]), _ptr(t["g"]), _ptr(t["beta"]),
              _ptr(t["w_s"]), _ptr(t["b_s"]), _ptr(t["w_g"]), _ptr(t["b_g"]), None, None, None, _ptr(out),
              _ptr(sel), _ptr(state), None, None]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if no_alloc:
        code = nat.lib.nats_hybrid_fwd_noalloc(*common, stream)
    else:
        need = nat.lib.nats_workspace_size(ctypes.byref(dm))
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        code = nat.lib.nats_hybrid_fwd(*common, _ptr(ws), ctypes.c_size_t(need), stream)
    assert code == 0, nat.STATUS.get(code, code)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), sel.cpu().numpy(), state.cpu().numpy()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_no_alloc_matches_workspace_entry_on_two_calls(nat, dtype):
    cases = [gen.make_inputs(1, 4, 512, 128, dtype=dtype, seed=31, pattern="random", frac=0.5),
             gen.make_inputs(2, 2, 384, 64, dtype=dtype, seed=32, pattern="alternating")]
    for inp in cases:  # two calls in a row, different shapes and selections
        ref_out, ref_sel, ref_state = _run(nat, inp, no_alloc=False)
        out, sel, state = _run(nat, inp, no_alloc=True)
        # the same kernels on the same inputs: the results agree bit for bit
        assert np.array_equal(sel, ref_sel)
        assert np.array_equal(out, ref_out)
        assert np.array_equal(state, ref_state)
        assert rel_err(out, ref_out) <= TOL[dtype]
        dm = nat.dims(inp.B, inp.H, inp.L, inp.d, nat.NATS_BF16 if dtype == "bf16" else nat.NATS_F32)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        assert nat.lib.nats_noalloc_check(ctypes.byref(dm), stream) == 0  # no bounded wait expired


def test_no_alloc_rejects_problems_beyond_its_scratch(nat):
    B, H, L, d = 1, 16, 16384, 128  # needs more than the built-in scratch
    dm = nat.dims(B, H, L, d)
    assert nat.lib.nats_workspace_size(ctypes.byref(dm)) > nat.NOALLOC_SCRATCH_BYTES
    # valid device buffers for every input and the output: only the size is wrong
    x = torch.zeros((B, H, L, d), dtype=torch.bfloat16, device="cuda")
    out = torch.full_like(x, 7.0)
    gb = torch.zeros((B, H, L), dtype=torch.float32, device="cuda")
    w_s = torch.zeros((H, 2, 2 * d), dtype=torch.float32, device="cuda")
    w_g = torch.zeros((H, d), dtype=torch.float32, device="cuda")
    args = [ctypes.byref(dm), _ptr(x), _ptr(x), _ptr(x), _ptr(gb), _ptr(gb), _ptr(w_s), None, _ptr(w_g), None,
            None, None, None, _ptr(out), None, None, None, None, None]
    assert nat.lib.nats_hybrid_fwd_noalloc(*args) == 5  # NATS_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert bool((out.float() == 7.0).all())  # the output was not touched
    assert nat.lib.nats_noalloc_check(ctypes.byref(dm), None) == 5
    # the regular checks come first: a NULL output is reported as such
    args[13] = None
    assert nat.lib.nats_hybrid_fwd_noalloc(*args) == 1  # NATS_ERR_NULL

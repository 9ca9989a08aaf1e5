"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Engines that own every device allocation, or systems that freeze their memory budget at
start-up, cannot hand the backward a freshly allocated workspace.  attn_bwd_noalloc takes its
float32 scratch from a fixed static array in the library instead.  This file checks, through
the C ABI, that on two calls in a row with different inputs it returns bit for bit what
attn_bwd returns on the same inputs (the same kernels run; only the scratch differs, so a
stale or aliased table would show as a changed bit), that it allocates no device memory, and
that it refuses problems larger than its array.  It is collected last on purpose.
"""
import ctypes
import gc

import pytest
import torch

import exact_io_aware_gb300 as ea
from synth import Workload

from helpers import head_inputs, to_dev

pytestmark = pytest.mark.gpu


def _noalloc(lib):
    f = lib.attn_bwd_noalloc
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    f.argtypes = [i32, i32, i32, i32, i32, f32, vp, vp, vp, vp, vp, vp, i32, vp, i64, i64, i32,
                  vp, vp, vp, vp]
    f.restype = i32
    return f


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _free_device_bytes_unchanged(before, tries=3):
    """True if the device's free memory is back at `before` in one of a few readings (another
    process on a shared GPU may move it for a moment; a leak by this call would not go away)."""
    for _ in range(tries):
        torch.cuda.synchronize()
        if torch.cuda.mem_get_info()[0] >= before:
            return True
    return False


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_attn_bwd_on_two_calls(dtype):
    lib = ea.load()
    noalloc = _noalloc(lib)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # two problems of different shapes and seeds, run back to back through the one array
    for call, (seed, H, n) in enumerate(((21, 3, 777), (22, 2, 300))):
        wl = Workload("noalloc", seed, 2, H, n, 64, dtype, "causal", 0.125)
        inp = head_inputs(wl)
        dev = {t: to_dev(inp[t], dtype) for t in inp}
        q, k, v, g = dev["q"], dev["k"], dev["v"], dev["do"]
        o, lse = ea.attn_fwd(q, k, v, wl.c, mask="causal")
        ref = ea.attn_bwd(q, k, v, o, lse, g, wl.c, mask="causal")
        code = ea.DTYPE_CODE[q.dtype]
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        # garbage from earlier tests must not be collected (and freed) inside the measured window
        gc.collect()
        gc.disable()
        try:
            torch.cuda.synchronize()
            torch_bytes = torch.cuda.memory_allocated()
            free_before = torch.cuda.mem_get_info()[0]
            rc = noalloc(code, wl.B, wl.H, wl.n, wl.d, wl.c, _p(q), _p(k), _p(v), _p(o), _p(lse),
                         _p(g), 1, ctypes.c_void_p(0), 0, 0, 0, _p(dq), _p(dk), _p(dv), stream)
            assert rc == 0, ea.attn_last_error()
            assert ea.attn_device_status() == ea.ATTN_OK
            assert torch.cuda.memory_allocated() == torch_bytes
        finally:
            gc.enable()
        if call == 1:  # the first call may load the library's module data on this device
            assert _free_device_bytes_unchanged(free_before)
        for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            assert torch.equal(got, want), f"call {call}: {name} differs from attn_bwd"


def test_noalloc_refuses_problems_larger_than_its_scratch():
    lib = ea.load()
    noalloc = _noalloc(lib)
    need = lib.attn_bwd_workspace_bytes(2, 1, 128, 70000, 128)
    assert need > (32 << 20)
    buf = torch.empty(64, dtype=torch.bfloat16, device="cuda")
    p = _p(buf)
    rc = noalloc(2, 1, 128, 70000, 128, 0.1, p, p, p, p, p, p, 0, ctypes.c_void_p(0), 0, 0, 0,
                 p, p, p, ctypes.c_void_p(0))
    assert rc == ea.ATTN_ERR_WORKSPACE
    assert "attn_bwd_noalloc" in ea.attn_last_error()

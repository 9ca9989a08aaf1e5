"""The C ABI library loads, exports every entry point the header declares, and rejects bad
arguments on the host (no GPU needed: argument checks run before any CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "exactattn.h")


@pytest.fixture(scope="module")
def lib():
    from exact_io_aware_gb300.build import build

    path = build()
    import exact_io_aware_gb300 as ea

    return ea.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("attn_fwd", "attn_bwd", "attn_bwd_workspace_bytes", "attn_device_status",
                 "attn_last_error"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def _fwd(lib, **kw):
    args = dict(dtype=2, B=1, H=1, n=128, d=64, c=0.125, q=16, k=32, v=48, mask=0, bits=0,
                row_words=0, head_stride=0, kvb=0, o=64, lse=80, stream=0)
    args.update(kw)
    vp = ctypes.c_void_p
    return lib.attn_fwd(args["dtype"], args["B"], args["H"], args["n"], args["d"], args["c"],
                        vp(args["q"]), vp(args["k"]), vp(args["v"]), args["mask"], vp(args["bits"]),
                        args["row_words"], args["head_stride"], args["kvb"], vp(args["o"]),
                        vp(args["lse"]), vp(args["stream"]))


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=7), -1),
    (dict(n=0), -1),
    (dict(B=-1), -1),
    (dict(d=48), -2),
    (dict(d=256), -2),
    (dict(kvb=96), -2),
    (dict(B=300, H=300), -2),
    (dict(q=0), -1),
    (dict(o=0), -1),
    (dict(lse=0), -1),
    (dict(q=18), -3),
    (dict(o=72), -3),
    (dict(lse=82), -3),
    (dict(mask=5), -1),
    (dict(mask=2, bits=0), -1),
    (dict(mask=2, bits=16, row_words=3), -1),
    (dict(mask=2, bits=18, row_words=4), -3),
    (dict(mask=2, bits=16, row_words=4, head_stride=-1), -1),
])
def test_forward_rejects_bad_arguments_on_host(lib, kw, code):
    assert _fwd(lib, **kw) == code
    assert lib.attn_last_error().decode() != ""


def test_backward_workspace_check_on_host(lib):
    need = lib.attn_bwd_workspace_bytes(2, 2, 3, 1000, 64)
    rows = 2 * 3 * 1000
    assert need >= 2 * (2 * 3 * 1024) * 4  # per-row table: LSE and D, n padded to 128 rows
    assert lib.attn_bwd_workspace_bytes(0, 2, 3, 1000, 64) >= rows * 4
    assert lib.attn_bwd_workspace_bytes(2, 0, 3, 1000, 64) == 0
    vp = ctypes.c_void_p
    rc = lib.attn_bwd(2, 2, 3, 1000, 64, 0.125, vp(16), vp(32), vp(48), vp(64), vp(80), vp(96),
                      0, vp(0), 0, 0, 0, vp(112), vp(128), vp(144), vp(160), need - 1, vp(0))
    assert rc == -4
    rc = lib.attn_bwd(2, 2, 3, 1000, 64, 0.125, vp(16), vp(32), vp(48), vp(64), vp(80), vp(0),
                      0, vp(0), 0, 0, 0, vp(112), vp(128), vp(144), vp(160), need, vp(0))
    assert rc == -1


def test_value_width_entries_reject_bad_arguments_on_host(lib):
    vp = ctypes.c_void_p
    fwd = lambda d, vw, o=64, p_drop=0.0: lib.attn_fwd_vdim(
        2, 1, 1, 128, d, vw, 0.125, vp(16), vp(32), vp(48), 0, vp(0), 0, 0, 0, p_drop, 0, vp(o),
        vp(80), vp(0))
    assert fwd(64, 32) == -2 and fwd(128, 16) == -2 and fwd(64, 96) == -2  # pairs not built
    assert fwd(64, 128, o=0) == -1          # null output (a supported pair gets that far)
    assert fwd(128, 64, o=72) == -3         # misaligned output
    assert fwd(64, 128, p_drop=1.0) == -1   # p_drop must lie in [0, 1)
    bwd = lambda d, vw, ws=4096: lib.attn_bwd_vdim(
        2, 1, 1, 128, d, vw, 0.125, vp(16), vp(32), vp(48), vp(64), vp(80), vp(96), 0, vp(0), 0,
        0, 0, 0.0, 0, vp(112), vp(128), vp(144), vp(160), ws, vp(0))
    assert bwd(64, 32) == -2
    assert bwd(64, 128, ws=0) == -4         # workspace too small


def test_fp8_block_entries_reject_bad_arguments_on_host(lib):
    vp = ctypes.c_void_p
    quant = lambda dtype=2, d=64, n=128, q=16, sq=256: lib.attn_fp8_quantize(
        dtype, 1, 1, n, d, vp(q), vp(32), vp(48), vp(0), vp(64), vp(80), vp(96), vp(sq),
        vp(272), vp(288), vp(0))
    assert quant(dtype=0) == -2             # float32 inputs
    assert quant(d=96) == -2 and quant(d=32) == -2
    assert quant(n=100) == -2               # n not a multiple of 16
    assert quant(q=0) == -1
    assert quant(q=24) == -3                # misaligned input
    assert quant(sq=258) == -3              # misaligned scales
    fwd = lambda d=64, n=128, sk=272, o=64: lib.attn_fwd_fp8_blocks(
        1, 1, n, d, 0.125, vp(16), vp(32), vp(48), vp(256), vp(sk), vp(288), 0, vp(0), 0, 0,
        vp(o), vp(80), vp(0))
    assert fwd(d=16) == -2
    assert fwd(n=120) == -2
    assert fwd(sk=0) == -1                  # null scale pointer
    assert fwd(sk=274) == -3                # misaligned scale pointer
    assert fwd(o=72) == -3


def test_ring_depth_cap_is_checked(lib):
    assert lib.attn_debug_set_ring_stages(5) == -1
    assert lib.attn_debug_set_ring_stages(-1) == -1
    assert lib.attn_debug_set_ring_stages(2) == 0
    assert lib.attn_debug_set_ring_stages(0) == 0


def test_ring_stage_division_is_exact():
    """The kernels' stage / parity of ring use i: a multiply-high by ceil(2^32 / n) must equal
    i // n (n = 2, 3, 4) for every i a kernel can reach (step counts below 2^31)."""
    import numpy as np
    rng = np.random.default_rng(1)
    i = np.concatenate([np.arange(0, 1 << 16), rng.integers(0, 1 << 31, 1 << 16),
                        [(1 << 31) - 1, (1 << 31) - 2]]).astype(np.uint64)
    for n in (2, 3, 4):
        magic = np.uint64(((1 << 32) + n - 1) // n)
        q = (i * magic) >> np.uint64(32)
        assert np.array_equal(q, i // np.uint64(n)), n

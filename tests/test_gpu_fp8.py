"""FP8 (E4M3) forward on the GPU against the oracle's exact attention on the dequantized inputs.

The inputs are quantized per tensor (scale = max |x| / 448), the kernel gets the E4M3 bytes, and
the oracle computes exact attention on the dequantized values.  The only rounding the FP8 path
adds is that of the probabilities to E4M3 before the P V product, bounded elementwise by
sum_j (2^-4 P_ij + 2^-18) |V_ja| (oracle/fp8.py); the tolerance is that bound plus bfloat16
output rounding (2^-8 relative) and float32 slack.
"""
import numpy as np
import pytest
import torch

import exact_io_aware_gb300 as ea
from oracle import fp8 as ofp8
from oracle import masks
from synth import Workload, draw_head, pack_bitmap

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not hasattr(torch, "float8_e4m3fn"), reason="torch without float8")]


def _quant(x):
    s = float(np.abs(x).max()) / 448.0
    q, deq = ofp8.quantize(x, s)
    t = torch.from_numpy(q.astype(np.float32)).to(torch.float8_e4m3fn)
    assert np.array_equal(t.to(torch.float64).numpy(), q)  # the codes carry the oracle's values
    return t, deq, s


def _run(B, H, n, d, mask, c_mult=1.0, q_mult=1.0, seed=71):
    wl = Workload("fp8", seed, B, H, n, d, "f32", mask, d ** -0.5)
    raw = {t: np.stack([draw_head(wl, t, bh) for bh in range(wl.heads)]).reshape(B, H, n, d)
           for t in ("q", "k", "v")}
    raw["q"] = raw["q"] * q_mult
    q8, dq_, sq = _quant(raw["q"])
    k8, dk_, sk = _quant(raw["k"])
    v8, dv_, sv = _quant(raw["v"])
    vt8 = v8.transpose(2, 3).contiguous()
    c = wl.c * c_mult
    if mask == "bitmap":
        rng = np.random.default_rng(seed)
        allowed = rng.random((n, n)) < 0.3
        allowed[np.arange(n), np.arange(n)] = True
        words = pack_bitmap(allowed)
        mk = masks.bitmap(words, n)
        bits = torch.from_numpy(words.view(np.int32)).cuda()
    else:
        mk, bits = masks.for_kind(mask, n), None
    o, lse = ea.attn_fwd_fp8(q8.cuda(), k8.cuda(), vt8.cuda(), c, sq, sk, sv, mask=mask,
                             mask_bits=bits)
    status = ea.attn_device_status()
    o = o.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    worst = 0.0
    for bh in range(B * H):
        b, h = divmod(bh, H)
        Y, L, bound = ofp8.forward_rows_bound(dq_[b, h], dk_[b, h], dv_[b, h], c,
                                              mk(bh, np.arange(n)))
        err = np.abs(o[b, h] - Y)
        tol = 1.02 * bound + 2.0 ** -8 * np.abs(Y) + 1e-5
        assert np.all(err <= tol), (f"head {bh}: O off at {np.argwhere(err > tol)[:4].tolist()}, "
                                    f"max err/tol {np.max(err / tol):.3f}")
        fin = np.isfinite(L)
        assert np.array_equal(np.isfinite(lse[b, h]), fin)
        assert np.max(np.abs(lse[b, h][fin] - L[fin]), initial=0.0) <= 2e-3
        worst = max(worst, float(np.linalg.norm(o[b, h] - Y) / max(np.linalg.norm(Y), 1e-30)))
    return status, worst


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mask", ["none", "causal", "bitmap"])
@pytest.mark.parametrize("n", [128, 336])
def test_fp8_forward_within_the_rounding_bound(d, mask, n):
    status, worst = _run(1, 2, n, d, mask)
    assert status == ea.ATTN_OK
    assert worst < 0.05  # relative Frobenius error of O: FP8 probabilities, a few per cent


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_forward_high_scores(d):
    """Scores of 20-30 (the overflow workload's range): the exact running maximum keeps every
    E4M3 probability at most 2^8."""
    status, _ = _run(1, 2, 256, d, "causal", c_mult=2.5, q_mult=2.5, seed=72)
    assert status == ea.ATTN_OK


def test_fp8_forward_several_tiles():
    status, worst = _run(2, 2, 1024, 128, "causal", seed=73)
    assert status == ea.ATTN_OK and worst < 0.05


def test_fp8_forward_rejects_unsupported_shapes():
    lib = ea.load()
    x = torch.zeros(64, dtype=torch.uint8, device="cuda")
    p = ea._ptr(x)
    assert lib.attn_fwd_fp8(1, 1, 100, 64, 0.1, p, p, p, 1.0, 1.0, 1.0, 0, None, 0, 0, p, p,
                            None) == ea.ATTN_ERR_UNSUPPORTED  # n not a multiple of 16
    assert lib.attn_fwd_fp8(1, 1, 128, 32, 0.1, p, p, p, 1.0, 1.0, 1.0, 0, None, 0, 0, p, p,
                            None) == ea.ATTN_ERR_UNSUPPORTED  # d = 32
    assert lib.attn_fwd_fp8(1, 1, 128, 64, 0.1, p, p, p, 0.0, 1.0, 1.0, 0, None, 0, 0, p, p,
                            None) == ea.ATTN_ERR_INVALID_ARG  # zero scale

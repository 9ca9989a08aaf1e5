"""Pins of the oracle's E4M3 rounding and FP8 error bound."""
import numpy as np
import pytest
import torch

from oracle import fp8


def test_e4m3_special_values():
    r = fp8.round_e4m3
    assert r(448.0) == 448.0 and r(460.0) == 448.0 and r(1e6) == 448.0 and r(-1e6) == -448.0
    assert r(2.0 ** -9) == 2.0 ** -9  # smallest subnormal
    assert r(2.0 ** -10) == 0.0  # halfway to zero: ties to even (zero)
    assert r(1.5 * 2.0 ** -9) == 2.0 * 2.0 ** -9  # halfway between f = 1 and 2: even f = 2
    assert r(1.0625) == 1.0 and r(1.1875) == 1.25  # ties to even fraction
    assert r(1.0626) == 1.125 and r(-3.3) == -3.25
    assert r(2.0 ** -6) == 2.0 ** -6 and r(7 * 2.0 ** -9) == 7 * 2.0 ** -9  # normal/subnormal edge
    assert r(0.0) == 0.0


@pytest.mark.skipif(not hasattr(torch, "float8_e4m3fn"), reason="torch without float8")
def test_e4m3_matches_torch_conversion():
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.normal(size=20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 300.0)])
    x = x[np.abs(x) <= 448.0]  # torch's conversion is not saturating; inside the range they agree
    want = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.round_e4m3(x.astype(np.float32).astype(np.float64))
    assert np.array_equal(got, want)


def test_bound_covers_the_rounded_probabilities():
    # brute force: round P' = 2^8 e^{s - m} to E4M3 as the kernel does and check the bound
    rng = np.random.default_rng(9)
    for trial in range(20):
        n, d = 200, 16
        q, k, v = rng.normal(size=(n, d)), rng.normal(size=(n, d)), rng.normal(size=(n, d))
        a = rng.random((n, n)) < 0.5
        a[np.arange(n), np.arange(n)] = True
        c = 0.25 * (trial + 1)
        Y, lse, bound = fp8.forward_rows_bound(q, k, v, c, a)
        s = np.where(a, c * (q @ k.T), -np.inf)
        m = s.max(axis=1, keepdims=True)
        Pp = np.where(a, 256.0 * np.exp(s - m), 0.0)
        Yq = (fp8.round_e4m3(Pp) @ v) / Pp.sum(axis=1, keepdims=True)
        assert np.all(np.abs(Yq - Y) <= bound * (1 + 1e-12) + 1e-15)
        assert np.max(np.abs(Yq - Y)) > 0  # the rounding is visible


# ---------------------------------------------------------------- block scaling, incoherent processing


def test_hadamard_closed_forms():
    h4 = np.array([[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]], float)
    assert np.array_equal(fp8.hadamard(4), h4)  # Sylvester's order-4 matrix, written out
    for d in (1, 2, 16, 64, 128):
        h = fp8.hadamard(d)
        assert np.array_equal(h @ h.T, d * np.eye(d))  # rows orthogonal, norm^2 = d
        assert np.array_equal(h, h.T) and np.all(np.abs(h) == 1)
        # row i, column j of Sylvester's matrix: (-1)^popcount(i & j)
        i, j = np.meshgrid(np.arange(d), np.arange(d), indexing="ij")
        pc = np.vectorize(lambda x: bin(x).count("1"))(i & j)
        assert np.array_equal(h, (-1.0) ** pc)
    with pytest.raises(ValueError):
        fp8.hadamard(96)


def test_rotation_preserves_products_and_flattens_outliers():
    rng = np.random.default_rng(21)
    d = 128
    sg = rng.choice([-1.0, 1.0], d)
    q, k = rng.normal(size=(50, d)), rng.normal(size=(60, d))
    assert np.allclose(fp8.rotate(q, sg) @ fp8.rotate(k, sg).T / d, q @ k.T, atol=1e-11)
    e = np.zeros(d)
    e[37] = 5.0
    assert np.array_equal(np.abs(fp8.rotate(e, sg)), np.full(d, 5.0))  # one spike spreads flat


def test_block_quantization_definition():
    rng = np.random.default_rng(22)
    x = (rng.normal(size=(300, 64)) * np.array([1e-3, 1.0, 40.0])[np.arange(300) // 128][:, None])
    x = x.astype(np.float32).astype(np.float64)
    x[260:270] = 0.0
    codes, scales = fp8.quantize_blocks(x)
    assert scales.shape == (3,)
    for b, (lo, hi) in enumerate(((0, 128), (128, 256), (256, 300))):
        blk = x[lo:hi]
        amax = np.abs(blk).max()
        assert abs(scales[b] * 448.0 - amax) <= 2.0 ** -22 * amax  # scale = absmax / 448
        assert np.abs(codes[lo:hi]).max() == 448.0  # the block's largest entry maps to 448
        deq = codes[lo:hi] * scales[b]
        # dequantization error within half an E4M3 ulp (relative 2^-4) or the subnormal half-step
        err = np.abs(deq - blk)
        assert np.all(err <= np.maximum(2.0 ** -4 * np.abs(blk), 2.0 ** -10 * scales[b]) * (1 + 1e-6))
    z, sz = fp8.quantize_blocks(np.zeros((5, 16)))
    assert np.array_equal(z, np.zeros((5, 16))) and np.array_equal(sz, [1.0])  # zero block
    _, s2 = fp8.quantize_blocks(x[:128], divide=128.0)
    assert s2[0] == scales[0] / 128.0


def test_block_quantized_operands_stand_for_the_inputs():
    rng = np.random.default_rng(23)
    n, d = 260, 64
    q, k, v = (rng.normal(size=(n, d)) for _ in range(3))
    sg = rng.choice([-1.0, 1.0], d)
    for signs in (None, sg):
        h = fp8.block_quantized_head(q, k, v, signs)
        s_true = q @ k.T
        assert np.abs(h["q"] @ h["k"].T - s_true).max() <= 0.15 * np.abs(s_true).max()
        assert np.allclose(h["v"], v, rtol=2.0 ** -4, atol=1e-2)
        assert h["r"].max() == 1.0 and np.all(h["r"] > 0)
    # with no rotation the codes are the per-block quantization of the inputs themselves
    h = fp8.block_quantized_head(q, k, v)
    c8, s = fp8.quantize_blocks(q)
    assert np.array_equal(h["q8"], c8) and np.array_equal(h["sq"], s)


def test_incoherent_processing_lowers_the_error_on_outlier_channels():
    """Q and K with a few channels 30x larger than the rest (the case incoherent processing is
    for): the rotated, block-scaled scores are closer to the exact ones."""
    rng = np.random.default_rng(24)
    n, d = 256, 128
    boost = np.ones(d)
    boost[[3, 50, 90]] = 30.0
    q, k = rng.normal(size=(n, d)) * boost, rng.normal(size=(n, d)) * boost
    v = rng.normal(size=(n, d))
    s_true = q @ k.T
    err = {}
    for name, signs in (("plain", None), ("rotated", rng.choice([-1.0, 1.0], d))):
        h = fp8.block_quantized_head(q, k, v, signs)
        err[name] = np.sqrt(np.mean((h["q"] @ h["k"].T - s_true) ** 2))
    assert err["rotated"] < 0.7 * err["plain"], err


def test_block_scaled_bound_covers_the_rounded_probabilities():
    # brute force: the kernel's arithmetic with block-scaled values, P' = 2^8 e^{s - m} r_J
    rng = np.random.default_rng(25)
    for trial in range(10):
        n, d = 300, 16
        q, k = rng.normal(size=(n, d)), rng.normal(size=(n, d))
        v = rng.normal(size=(n, d)) * np.repeat(2.0 ** rng.integers(-12, 1, 3), 128)[:n, None]
        h = fp8.block_quantized_head(q, k, v)
        a = rng.random((n, n)) < 0.6
        a[np.arange(n), np.arange(n)] = True
        c = 0.3 * (trial + 1)
        Y, lse, bound = fp8.forward_rows_bound(h["q"], h["k"], h["v"], c, a, h["r"])
        s = np.where(a, c * (h["q"] @ h["k"].T), -np.inf)
        m = s.max(axis=1, keepdims=True)
        P0 = np.where(a, 256.0 * np.exp(s - m), 0.0)
        svmax = h["sv"].max()
        Yq = (fp8.round_e4m3(P0 * h["r"][None, :]) @ (h["v8"] * svmax)) / P0.sum(axis=1, keepdims=True)
        assert np.all(np.abs(Yq - Y) <= bound * (1 + 1e-12) + 1e-15)
        assert np.max(np.abs(Yq - Y)) > 0


def test_bound_holds_with_a_stale_running_maximum():
    """The FP8 forward raises its running maximum only when a block's maximum exceeds it by more
    than 0.75 in log2 units.  Brute force with the maximum anywhere in that window below the
    true one: P' = 2^8 e^{s - m} stays below 448 (no saturation), and the output with P'
    rounded to E4M3 stays within the same bound sum_j (2^-4 P_ij + 2^-18) |V_j|."""
    rng = np.random.default_rng(26)
    for trial in range(20):
        n, d = 150, 16
        q, k, v = rng.normal(size=(n, d)), rng.normal(size=(n, d)), rng.normal(size=(n, d))
        a = rng.random((n, n)) < 0.5
        a[np.arange(n), np.arange(n)] = True
        c = 0.3 * (trial + 1)
        Y, lse, bound = fp8.forward_rows_bound(q, k, v, c, a)
        s = np.where(a, c * (q @ k.T), -np.inf)
        lag = rng.uniform(0.0, 0.75, size=(n, 1)) * np.log(2.0)  # natural-log units
        m = s.max(axis=1, keepdims=True) - lag
        Pp = np.where(a, 256.0 * np.exp(s - m), 0.0)
        assert Pp.max() < 448.0 and np.all(Pp.max(axis=1) >= 256.0)
        Yq = (fp8.round_e4m3(Pp) @ v) / Pp.sum(axis=1, keepdims=True)
        assert np.all(np.abs(Yq - Y) <= bound * (1 + 1e-12) + 1e-15)

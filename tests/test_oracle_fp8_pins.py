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

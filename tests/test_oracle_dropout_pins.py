"""Pins of the oracle's dropout extension: the generator against its published known-answer
vectors, the mask's keep rate, the reduction to no dropout at p = 0, and the reverse pass
against central finite differences of the function with the realised mask held fixed."""
import math
import os

import numpy as np
import pytest

from oracle import attention, dropout, masks

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _kat():
    rows = []
    for line in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        ctr, key, out = (tuple(int(w, 16) for w in part.split()) for part in line.split("|"))
        rows.append((ctr, key, out))
    return rows


@pytest.mark.parametrize("ctr,key,out", _kat())
def test_philox_known_answers(ctr, key, out):
    got = dropout.philox4x32(np.array(ctr, dtype=np.uint64), key)
    assert tuple(int(x) for x in got) == out


def test_philox_rounds_matter():
    # a dropped round changes the output (guards against a loop that runs one round short)
    ctr, key, out = _kat()[2]
    assert tuple(int(x) for x in dropout.philox4x32(np.array(ctr, dtype=np.uint64), key, 9)) != out


@pytest.mark.parametrize("p", [0.1, 0.3, 0.5])
def test_keep_rate_and_independence(p):
    keep = dropout.keep_mask(0x1234_5678_9ABC, 3, np.arange(300), 1000, p)
    pe = dropout.effective_p(p)
    n = keep.size
    sd = math.sqrt(pe * (1 - pe) / n)
    assert abs(keep.mean() - (1 - pe)) < 5 * sd
    # pairs one generator call decides together are not correlated: neighbouring keys of a
    # row and neighbouring rows of a key
    for a, b in ((keep[:, 0::4], keep[:, 1::4]), (keep[0::4, :], keep[1::4, :])):
        a, b = a.ravel(), b.ravel()
        assert abs(np.mean(a & b) - (1 - pe) ** 2) < 5 * math.sqrt((1 - pe) ** 2 / a.size)
    # different seeds or heads give different masks
    other = dropout.keep_mask(0x1234_5678_9ABD, 3, np.arange(300), 1000, p)
    assert np.mean(other != keep) > 0.5 * 2 * pe * (1 - pe)
    assert np.any(dropout.keep_mask(0x1234_5678_9ABC, 4, np.arange(300), 1000, p) != keep)


def test_threshold_edges():
    assert dropout.threshold(0.0) == 0
    assert dropout.threshold(0.5) == 128
    assert dropout.threshold(0.1) == 26 and dropout.effective_p(0.1) == 26 / 256
    assert dropout.threshold(0.998) == 255
    for bad in (0.999, 1.0, -0.1):
        with pytest.raises(ValueError):
            dropout.threshold(bad)
    assert dropout.keep_mask(7, 0, np.arange(5), 9, 0.0).all()


@pytest.mark.parametrize("p", [0.25, 0.5, 0.9])
def test_patch_layout_from_the_published_vector(p):
    """Rows 0-3 x keys 0-3 of head 0 under seed 0 are one generator call: counter (0,0,0,0),
    key (0,0), the first published known-answer vector.  Row x reads word x, key y byte y
    (least significant first); the pair is kept iff the byte reaches the 8-bit threshold."""
    ctr, key, out = _kat()[0]
    assert ctr == (0, 0, 0, 0) and key == (0, 0)
    t = int(math.floor(p * 256 + 0.5))
    want = [[((out[x] >> (8 * y)) & 0xFF) >= t for y in range(4)] for x in range(4)]
    got = dropout.keep_mask(0, 0, np.arange(4), 4, p)
    assert got.tolist() == want


def test_zero_probability_is_plain_attention():
    rng = np.random.default_rng(3)
    n, d = 23, 5
    q, k, v, g = (rng.normal(size=(n, d)) for _ in range(4))
    a = masks.causal(n)(0, np.arange(n))
    keep = dropout.keep_mask(9, 0, np.arange(n), n, 0.0)
    y, lse = dropout.forward_rows(q, k, v, 0.6, a, keep, 0.0)
    y0, lse0, _, _ = attention.forward_rows(q, k, v, 0.6, a)
    assert np.max(np.abs(y - y0)) < 1e-13 and np.max(np.abs(lse - lse0)) < 1e-13
    grads = dropout.backward_head(q, k, v, 0.6, a, keep, 0.0, g)
    ref = attention.backward_head(q, k, v, 0.6, a, g)
    for x, r in zip(grads, ref):
        assert np.max(np.abs(x - r)) < 1e-12


def test_dropout_gradient_matches_central_differences():
    rng = np.random.default_rng(4)
    n, d, p, c = 7, 3, 0.4, 0.8
    q, k, v, g = (rng.normal(size=(n, d)) for _ in range(4))
    a = masks.causal(n)(0, np.arange(n))
    keep = dropout.keep_mask(21, 1, np.arange(n), n, p)
    assert 0 < keep[a].sum() < a.sum()  # some allowed pairs dropped, some kept

    def phi(qq, kk, vv):
        y, _ = dropout.forward_rows(qq, kk, vv, c, a, keep, p)
        return float((g * y).sum())

    dQ, dK, dV = dropout.backward_head(q, k, v, c, a, keep, p, g)
    h = 1e-6
    for name, x, grad in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            fp = phi(args["q"], args["k"], args["v"])
            args[name] = xm
            fm = phi(args["q"], args["k"], args["v"])
            fd[idx] = (fp - fm) / (2 * h)
        assert np.max(np.abs(fd - grad)) <= 1e-7 * max(1.0, np.max(np.abs(grad))), name


def test_dropout_key_gradient_sums_to_zero_and_output_is_unbiased():
    rng = np.random.default_rng(5)
    n, d, p = 40, 4, 0.3
    q, k, v, g = (rng.normal(size=(n, d)) for _ in range(4))
    a = np.ones((n, n), bool)
    keep = dropout.keep_mask(5, 2, np.arange(n), n, p)
    _, dK, _ = dropout.backward_head(q, k, v, 0.5, a, keep, p, g)
    assert np.max(np.abs(dK.sum(axis=0))) < 1e-12
    # averaged over many seeds the dropped output approaches the plain one
    y0, _, _, _ = attention.forward_rows(q, k, v, 0.5, a)
    acc = np.zeros_like(y0)
    seeds = 400
    for s in range(seeds):
        acc += dropout.forward_rows(q, k, v, 0.5, a, dropout.keep_mask(s, 0, np.arange(n), n, p),
                                    p)[0]
    assert np.max(np.abs(acc / seeds - y0)) < 0.1


def test_gamma_pieces_agree_with_the_reverse_pass():
    rng = np.random.default_rng(6)
    n, d, p, c = 12, 4, 0.35, 0.7
    q, k, v, g = (rng.normal(size=(n, d)) for _ in range(4))
    a = masks.causal(n)(0, np.arange(n))
    keep = dropout.keep_mask(3, 1, np.arange(n), n, p)
    P, dPt, gamma = dropout.probabilities_and_gamma(q, k, v, c, a, keep, p, g)
    dQ, dK, _ = dropout.backward_head(q, k, v, c, a, keep, p, g)
    assert np.max(np.abs(c * gamma @ k - dQ)) < 1e-12
    assert np.max(np.abs(c * gamma.T @ q - dK)) < 1e-12
    assert np.array_equal(P[~a], np.zeros(np.count_nonzero(~a)))

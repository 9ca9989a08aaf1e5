"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test ties the oracle to something other than itself: the worked examples printed on
the pages (fixtures under tests/golden/, each with its citation), closed forms, invariants,
brute-force finite differences on tiny inputs, and a negative control.
"""
import math
import os

import numpy as np
import pytest

from oracle import attention, io_model, masks, tiled
from synth import bitmap_mask, draw_head, pack_bitmap, workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _random_allowed(rng, n, p=0.4):
    a = rng.random((n, n)) < p
    a[np.arange(n), rng.integers(0, n, n)] = True  # every row nonempty
    return a


# ---------------------------------------------------------------- worked examples (page 1)

def _golden_examples():
    rows = []
    with open(os.path.join(GOLDEN, "streaming_softmax_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, blocks, qty, val = [x.strip() for x in line.split("|")]
            blks = [[float(t) for t in b.split(",")] for b in blocks.split(";")]
            rows.append((name, blks, qty, float(val)))
    return rows


@pytest.mark.parametrize("name,blocks,qty,printed", _golden_examples())
def test_streaming_worked_examples(name, blocks, qty, printed):
    b1, b2 = (np.array(b) for b in blocks)
    s1 = tiled.block_summary(b1, np.zeros((b1.size, 0)))
    s2 = tiled.block_summary(b2, np.zeros((b2.size, 0)))
    m, ell = tiled.streaming_normaliser([b1, b2])
    one = tiled.block_summary(np.concatenate([b1, b2]), np.zeros((b1.size + b2.size, 0)))
    got = {
        "m_after_block_1": s1[0],
        "l_after_block_1": s1[1],
        "rescaled_old_sum": s1[1] * math.exp(s1[0] - m),
        "new_block_sum": s2[1] * math.exp(s2[0] - m),
        "m_final": m,
        "l_final": ell,
        "l_one_shot": one[1],
    }[qty]
    assert abs(got - printed) <= 5e-4  # the page prints three decimals


def test_streaming_examples_exact_values():
    m, ell = tiled.streaming_normaliser([[2, 1], [3, 0]])
    assert m == 3
    assert abs(ell - (math.exp(-1) + math.exp(-2) + 1 + math.exp(-3))) < 1e-14
    assert abs(ell - 1.5530017928) < 1e-9
    m, ell = tiled.streaming_normaliser([[1, 4], [2, 2, 5]])
    assert m == 5
    assert abs(ell - 1.4857692168) < 1e-9


# ---------------------------------------------------------------- merge algebra (page 5)

def _rand_summary(rng, v=4):
    s = rng.normal(size=rng.integers(1, 6)) * 3
    return tiled.block_summary(s, rng.normal(size=(s.size, v)))


def _close(a, b, tol=1e-12):
    return (abs(a[0] - b[0]) <= tol * max(1, abs(a[0]))
            and abs(a[1] - b[1]) <= tol * max(1, abs(a[1]))
            and np.allclose(a[2], b[2], rtol=tol, atol=tol))


def test_merge_associative_commutative_identity():
    rng = _rng(11)
    for _ in range(200):
        a, b, c = (_rand_summary(rng) for _ in range(3))
        assert _close(tiled.merge(a, b), tiled.merge(b, a))
        assert _close(tiled.merge(tiled.merge(a, b), c), tiled.merge(a, tiled.merge(b, c)))
        assert tiled.merge(a, tiled.BOTTOM) is a
        assert tiled.merge(tiled.BOTTOM, a) is a


def test_merge_of_disjoint_sets_is_summary_of_union():
    rng = _rng(12)
    for _ in range(100):
        s = rng.normal(size=9) * 4
        v = rng.normal(size=(9, 3))
        cut = rng.integers(1, 9)
        u = tiled.merge(tiled.block_summary(s[:cut], v[:cut]),
                        tiled.block_summary(s[cut:], v[cut:]))
        assert _close(u, tiled.block_summary(s, v))
        assert u[0] == s.max()


# ---------------------------------------------------------------- key shares (page 5)

def _shard_results(q, k, val, c, a, shares):
    """Each share's normalised (O_g, LSE_g) from the dense definition on that share alone."""
    out = []
    for idx in shares:
        keep = np.zeros(a.shape[1], bool)
        keep[idx[idx < a.shape[1]]] = True
        y, lse, _, _ = attention.forward_rows(q, k, val, c, a & keep[None, :])
        out.append((y, lse))
    return out


@pytest.mark.parametrize("kind", ["none", "causal", "random"])
def test_merged_key_shares_equal_dense(kind):
    rng = _rng(31)
    n, d, v, b = 45, 4, 3, 4
    q, k = rng.normal(size=(n, d)), rng.normal(size=(n, d)) * 2
    val = rng.normal(size=(n, v))
    c = 0.9
    if kind == "none":
        a = np.ones((n, n), bool)
    elif kind == "causal":
        a = masks.causal(n)(0, np.arange(n))
    else:
        a = _random_allowed(rng, n, 0.15)  # many (row, share) pairs with no allowed key
    y, lse, _, _ = attention.forward_rows(q, k, val, c, a)
    reach = -(-n // b)
    for parts in (1, 2, 3, 5, 12, 20):
        shares = tiled.key_shares(reach, parts, b)
        assert sorted(np.concatenate(shares).tolist()) == list(range(reach * b))
        res = _shard_results(q, k, val, c, a, shares)
        for i in range(n):
            o_i, l_i = tiled.merge_normalised([(yg[i], lg[i]) for yg, lg in res])
            assert abs(l_i - lse[i]) <= 1e-12
            assert np.max(np.abs(o_i - y[i])) <= 1e-12


def test_merge_normalised_worked_example_and_empty_parts():
    # page 1's blocks {2, 1} and {3, 0} as two shares of one row (zero-width values)
    l1, l2 = math.log(math.exp(2) + math.exp(1)), math.log(math.exp(3) + 1.0)
    o, lse = tiled.merge_normalised([(np.zeros(0), l1), (np.zeros(0), l2)])
    assert abs(lse - (3 + math.log(1.5530017928))) < 1e-9  # m = 3, l = 1.553 as printed
    assert abs(lse - 3.4401896986) < 1e-9
    # values: the merged output is the softmax-weighted mean of the shares' outputs
    o, lse = tiled.merge_normalised([(np.array([1.0, -2.0]), 0.0), (np.array([3.0, 4.0]), math.log(3)),
                                     (np.array([9.0, 9.0]), -math.inf)])
    assert abs(lse - math.log(4)) < 1e-15
    assert np.allclose(o, [(1 + 3 * 3) / 4, (-2 + 3 * 4) / 4], atol=1e-15)
    o, lse = tiled.merge_normalised([(np.ones(3), -math.inf), (np.ones(3), -math.inf)])
    assert lse == -math.inf and np.all(o == 0)


# ---------------------------------------------------------------- exactness (page 5)

@pytest.mark.parametrize("kind", ["none", "causal", "random"])
def test_tiled_forward_equals_dense_for_every_block_size(kind):
    rng = _rng(21)
    n, d, v = 37, 5, 6
    q, k = rng.normal(size=(n, d)), rng.normal(size=(n, d))
    val = rng.normal(size=(n, v))
    c = 0.7
    if kind == "none":
        a = np.ones((n, n), bool)
    elif kind == "causal":
        a = masks.causal(n)(0, np.arange(n))
    else:
        a = _random_allowed(rng, n)
    y, lse, m, ell = attention.forward_rows(q, k, val, c, a)
    for b in (1, 3, 8, 32, 37, 64):
        ty, tm, tl = tiled.forward_head(q, k, val, c, a, b)
        assert np.max(np.abs(ty - y)) <= 1e-12
        assert np.max(np.abs(tm - m)) <= 1e-12
        assert np.max(np.abs(tl - ell) / ell) <= 1e-12
        assert np.max(np.abs(tm + np.log(tl) - lse)) <= 1e-12


@pytest.mark.parametrize("vw", [4, 7, 2])
def test_reverse_procedure_equals_dense_backward(vw):
    """Value width vw = d and vw != d (the general shape: V and G have their own width)."""
    rng = _rng(22)
    n, d = 23, 4
    q, k = (rng.normal(size=(n, d)) for _ in range(2))
    val, g = (rng.normal(size=(n, vw)) for _ in range(2))
    c = 0.9
    a = _random_allowed(rng, n)
    dq, dk, dv, y, lse = attention.backward_head(q, k, val, c, a, g)
    for b in (1, 5, 23):
        ty, tm, tl = tiled.forward_head(q, k, val, c, a, b)
        rq, rk, rv = tiled.reverse_head(q, k, val, c, a, b, ty, tm, tl, g)
        for x, ref in ((rq, dq), (rk, dk), (rv, dv)):
            assert np.max(np.abs(x - ref)) <= 1e-11 * max(1.0, np.max(np.abs(ref)))


def _phi(q, k, v, c, a, g):
    y, _, _, _ = attention.forward_rows(q, k, v, c, a)
    return float((g * y).sum())


@pytest.mark.parametrize("tied,vw", [(False, 3), (True, 3), (False, 5), (False, 2)])
def test_gradient_matches_central_differences(tied, vw):
    rng = _rng(23 + tied)
    n, d = 7, 3
    q, k = (rng.normal(size=(n, d)) for _ in range(2))
    v, g = (rng.normal(size=(n, vw)) for _ in range(2))
    c = 0.8
    a = _random_allowed(rng, n, 0.6)
    a[2, :] = True
    if tied:  # two keys with the same, maximal score in row 2 (the theorem allows ties)
        k[4] = k[5] = 3.0 * q[2] / np.linalg.norm(q[2])
    dq, dk, dv, _, _ = attention.backward_head(q, k, v, c, a, g)
    if tied:
        s = c * (k @ q[2])
        assert s[4] == s[5] == s.max()
    h = 1e-6
    for x, grad in ((q, dq), (k, dk), (v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + h
            fp = _phi(q, k, v, c, a, g)
            x[idx] = old - h
            fm = _phi(q, k, v, c, a, g)
            x[idx] = old
            fd[idx] = (fp - fm) / (2 * h)
        assert np.linalg.norm(fd - grad) <= 1e-7 * np.linalg.norm(grad) + 1e-9


# ---------------------------------------------------------------- closed forms and invariants

def test_zero_scale_gives_mean_and_log_count():
    rng = _rng(31)
    n, d = 50, 6
    q, k, v, g = (rng.normal(size=(n, d)) for _ in range(4))
    a = _random_allowed(rng, n)
    y, lse, _, _ = attention.forward_rows(q, k, v, 0.0, a)
    for i in range(n):
        assert np.allclose(y[i], v[a[i]].mean(axis=0), atol=1e-13)
        assert abs(lse[i] - math.log(a[i].sum())) <= 1e-13
    dq, dk, _, _, _ = attention.backward_head(q, k, v, 0.0, a, g)
    assert np.all(dq == 0) and np.all(dk == 0)


def test_single_allowed_key_and_causal_first_row():
    rng = _rng(32)
    n, d = 20, 5
    q, k, v = (rng.normal(size=(n, d)) for _ in range(3))
    c = 1.3
    a = np.zeros((n, n), bool)
    pick = rng.integers(0, n, n)
    a[np.arange(n), pick] = True
    y, lse, _, _ = attention.forward_rows(q, k, v, c, a)
    assert np.allclose(y, v[pick], atol=1e-15)
    assert np.allclose(lse, c * np.einsum("ir,ir->i", q, k[pick]), atol=1e-13)
    yc, lc, _, _ = attention.forward_rows(q, k, v, c, masks.causal(n)(0, np.arange(n)))
    assert np.allclose(yc[0], v[0], atol=1e-15)
    assert abs(lc[0] - c * float(q[0] @ k[0])) <= 1e-13


def test_gradient_sum_rules():
    rng = _rng(33)
    n, d = 40, 8
    q, k, v, g = (rng.normal(size=(n, d)) for _ in range(4))
    a = _random_allowed(rng, n)
    dq, dk, dv, _, _ = attention.backward_head(q, k, v, 0.5, a, g)
    # Σ_j γ_ij = 0 for every row, so the key gradients sum to zero ...
    assert np.max(np.abs(dk.sum(axis=0))) <= 1e-12
    # ... and Σ_j p_ij = 1, so the value gradients sum to the upstream rows.
    assert np.allclose(dv.sum(axis=0), g.sum(axis=0), atol=1e-12)


def test_shift_and_permutation_invariances():
    rng = _rng(34)
    n, d = 30, 4
    q, k, v = (rng.normal(size=(n, d)) for _ in range(3))
    c = 0.6
    a = _random_allowed(rng, n)
    y, lse, _, _ = attention.forward_rows(q, k, v, c, a)
    u, w = rng.normal(size=d), rng.normal(size=d)
    y2, lse2, _, _ = attention.forward_rows(q, k + u, v, c, a)
    assert np.allclose(y2, y, atol=1e-12)
    assert np.allclose(lse2 - lse, c * (q @ u), atol=1e-12)
    y3, _, _, _ = attention.forward_rows(q, k, v + w, c, a)
    assert np.allclose(y3 - y, np.broadcast_to(w, y.shape), atol=1e-12)
    perm = rng.permutation(n)
    y4, lse4, _, _ = attention.forward_rows(q, k[perm], v[perm], c, a[:, perm])
    assert np.allclose(y4, y, atol=1e-12) and np.allclose(lse4, lse, atol=1e-12)


def test_multi_head_layout():
    rng = _rng(35)
    B, H, n, d = 2, 3, 9, 4
    Q, K, V, G = (rng.normal(size=(B, H, n, d)) for _ in range(4))
    mk = masks.causal(n)
    Y, L = attention.forward(Q, K, V, 0.5, mk)
    dQ, dK, dV = attention.backward(Q, K, V, 0.5, mk, G)
    for bh in range(B * H):
        b, h = divmod(bh, H)
        a = mk(bh, np.arange(n))
        y, lse, _, _ = attention.forward_rows(Q[b, h], K[b, h], V[b, h], 0.5, a)
        dq, dk, dv, _, _ = attention.backward_head(Q[b, h], K[b, h], V[b, h], 0.5, a, G[b, h])
        assert np.array_equal(Y[b, h], y) and np.array_equal(L[b, h], lse)
        assert np.array_equal(dQ[b, h], dq) and np.array_equal(dK[b, h], dk)
        assert np.array_equal(dV[b, h], dv)


def test_empty_row_reading():
    a = np.zeros((3, 3), bool)
    a[0, 0] = a[2, 1] = True
    rng = _rng(36)
    q, k, v, g = (rng.normal(size=(3, 2)) for _ in range(4))
    y, lse, _, _ = attention.forward_rows(q, k, v, 1.0, a)
    assert np.all(y[1] == 0) and lse[1] == -np.inf
    dq, dk, dv, _, _ = attention.backward_head(q, k, v, 1.0, a, g)
    assert np.all(dq[1] == 0)
    ty, tm, tl = tiled.forward_head(q, k, v, 1.0, a, 2)
    assert np.all(ty[1] == 0) and tm[1] == -np.inf


# ---------------------------------------------------------------- negative control (page 4)

def _broken_forward(q, k, v, c, b):
    """The tiled forward with the running-total rescale e^{m-m'} left out on purpose."""
    n = q.shape[0]
    Y = np.zeros((n, v.shape[1]))
    for i in range(n):
        m, ell, z = -np.inf, 0.0, np.zeros(v.shape[1])
        for J in tiled.key_blocks(n, b):
            s = c * (k[J] @ q[i])
            mn = max(m, s.max())
            w = np.exp(s - mn)
            ell, z, m = ell + w.sum(), z + w @ v[J], mn  # old ℓ, z not rescaled
        Y[i] = z / ell
    return Y


def test_broken_rescale_fails_unless_max_in_first_block():
    rng = _rng(41)
    n, d, b = 32, 4, 8
    q, k, v = (rng.normal(size=(n, d)) for _ in range(3))
    a = np.ones((n, n), bool)
    y, _, _, _ = attention.forward_rows(q, k, v, 1.0, a)
    yb = _broken_forward(q, k, v, 1.0, b)
    s = q @ k.T
    first = s.argmax(axis=1) < b
    assert first.any() and (~first).any()
    err = np.max(np.abs(yb - y), axis=1)
    assert np.all(err[first] <= 1e-12)  # no running max change: nothing to forget
    assert np.all(err[~first] > 1e-6)  # later maxima: the forgotten rescale shows


# ---------------------------------------------------------------- fp16 overflow (page 4)

def test_fp16_overflow_threshold():
    with np.errstate(over="ignore"):
        assert np.isfinite(np.float16(math.exp(10.32)))
        assert np.isinf(np.float16(math.exp(math.log(65520.0) + 1e-9)))
        assert np.isinf(np.float16(math.exp(23.41)))
    assert abs(math.exp(10.32) - 30320) < 20  # the page prints 30,320


def test_overflow_workload_needs_the_running_max():
    wl = workload("overflow_f16_d64_hot")
    q, k, v = (draw_head(wl, t, 0, n=1024) for t in ("q", "k", "v"))
    a = masks.causal(1024)(0, np.arange(1024))
    s = attention.masked_scores(q, k, wl.c, a)
    rowmax = s.max(axis=1)
    assert 18.0 < np.median(rowmax[512:]) < 26.0
    with np.errstate(over="ignore"):
        naive = np.float16(np.exp(np.where(a, s, 0.0)))
    assert np.isinf(naive).any()  # exp of raw scores does not fit fp16
    y, lse, m, _ = attention.forward_rows(q, k, v, wl.c, a)
    shifted = np.exp(np.where(a, s - m[:, None], -np.inf))
    assert shifted.max() == 1.0 and np.isfinite(np.float16(shifted)).all()
    assert np.isfinite(y).all() and np.isfinite(lse).all()


# ---------------------------------------------------------------- IO model (page 4)

def test_io_model_reproduces_printed_counts():
    with open(os.path.join(GOLDEN, "io_counts.txt")) as f:
        rows = [l.split("|") for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) == 2
    for n, d, unfused, fused in rows:
        n, d = int(n), int(d)
        assert io_model.unfused_bytes(n, d) == int(unfused)
        assert io_model.fused_bytes(n, d) == int(fused)
    assert round(io_model.unfused_bytes(4096, 64) / 2**20) == 514
    assert round(io_model.fused_bytes(4096, 64) / 2**20) == 258
    assert io_model.unfused_bytes(4096, 16) / 2**20 == pytest.approx(272.5, abs=0.05)
    assert io_model.fused_bytes(4096, 16) / 2**20 == pytest.approx(16.5, abs=0.05)


# ---------------------------------------------------------------- mask storage

def test_rectangular_causal_is_the_tail_of_square_attention():
    # a key/value cache: the last m queries against all n keys give the last m rows of square
    # causal attention over the n positions
    rng = np.random.default_rng(61)
    n, d = 50, 6
    q, k, v = (rng.normal(size=(n, d)) for _ in range(3))
    y, lse, _, _ = attention.forward_rows(q, k, v, 0.7, masks.causal(n)(0, np.arange(n)))
    for m in (1, 3, 17, n):
        mk = masks.causal_rect(m, n)
        ym, lm, _, _ = attention.forward_rows(q[n - m:], k, v, 0.7, mk(0, np.arange(m)))
        assert np.max(np.abs(ym - y[n - m:])) < 1e-13 and np.max(np.abs(lm - lse[n - m:])) < 1e-13
    assert np.array_equal(masks.causal_rect(n, n)(0, np.arange(n)), masks.causal(n)(0, np.arange(n)))
    assert masks.causal_rect(1, 9)(0, [0]).all()
    a = masks.causal_rect(7, 4)(0, np.arange(7))  # more queries than keys: the first 3 see none
    assert not a[:3].any() and a[3, :1].all() and not a[3, 1:].any() and a[6].all()


def test_bitmap_membership_hand_built():
    n = 70
    words = np.zeros((2, 3), np.uint32)
    words[0, 0] = 0b1011  # keys 0, 1, 3
    words[0, 1] = 1 << 31  # key 63
    words[1, 2] = 1 << 5  # key 69
    mk = masks.bitmap(words, n)
    a = mk(0, [0, 1])
    assert sorted(np.flatnonzero(a[0])) == [0, 1, 3, 63]
    assert sorted(np.flatnonzero(a[1])) == [69]


def test_bitmap_head_stride_and_pack_roundtrip():
    rng = _rng(51)
    n = 100
    a0, a1 = _random_allowed(rng, n), _random_allowed(rng, n)
    w = np.concatenate([pack_bitmap(a0, 5), pack_bitmap(a1, 5)])
    mk = masks.bitmap(w, n, head_stride_words=n * 5)
    assert np.array_equal(mk(0, np.arange(n)), a0)
    assert np.array_equal(mk(1, np.arange(n)), a1)


def test_block_sparse_workload_bitmap():
    a = bitmap_mask(2048, 5)
    i = np.arange(2048)
    assert a[i, i].all()
    assert a[1000, 1000 - 128] and a[1000, 1000 + 127]
    assert 0.3 < a.mean() < 0.5
    blocks = a.reshape(32, 64, 32, 64).all(axis=(1, 3))
    assert 0.2 < blocks.mean() < 0.45

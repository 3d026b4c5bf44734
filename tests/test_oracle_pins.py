"""Pins for the fp64 CPU oracle, each against something other than the oracle.

Every test here checks the oracle against a fact the method pages or the
mathematics fix: a library routine the definition reduces to, a closed form,
an invariant, or brute-force enumeration on tiny inputs.  A dropped term,
wrong sign, wrong index or transposed operand anywhere in the oracle fails at
least one of them (see the comment on each test).
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_inputs(L, Hq, Hkv, D, T, W, seed, dtype="f32", scale=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (scale * torch.randn(L, Hq, W, D, generator=g)).float()
    k = torch.randn(L, Hkv, T, D, generator=g).float()
    if dtype == "bf16":
        q, k = q.bfloat16(), k.bfloat16()
    return q, k


# --------------------------------------------------------------------------- a1
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_score_equals_library_attention(seed):
    """The mean attention row of the window queries equals what torch's own
    scaled-dot-product attention returns when V is the identity (so the output
    IS the probability matrix), with the causal window mask and GQA mapping
    expanded explicitly.  Catches: wrong scale (1/D vs 1/sqrt(D)), mask offset
    (j<=i instead of j<=P+i), GQA mapping (h % H_kv instead of h // G), mean
    over the wrong axis, missing normalisation."""
    L, Hq, Hkv, D, T, W = 2, 4, 2, 8, 37, 5
    q, k = _rand_inputs(L, Hq, Hkv, D, T, W, seed, scale=2.0)
    s = O.shape_of(L, Hq, Hkv, D, T, W, "f32")
    c = O.score(s, q, k)
    G, P = Hq // Hkv, T - W
    kk = k.double().repeat_interleave(G, dim=1)                 # [L][Hq][T][D]
    eye = torch.eye(T, dtype=torch.float64).expand(L, Hq, T, T)
    pos = torch.arange(T)
    mask = pos[None, :] <= (P + torch.arange(W))[:, None]       # [W][T]
    probs = torch.nn.functional.scaled_dot_product_attention(
        q.double(), kk, eye, attn_mask=mask)                    # [L][Hq][W][T]
    ref = probs.view(L, Hkv, G, W, T).mean(dim=(2, 3)).numpy()
    np.testing.assert_allclose(c, ref, rtol=1e-12, atol=1e-15)


def test_score_single_row_is_softmax():
    """W=1, G=1: the score is one textbook softmax row over all T keys."""
    L, H, D, T = 1, 3, 16, 50
    q, k = _rand_inputs(L, H, H, D, T, 1, 7)
    s = O.shape_of(L, H, H, D, T, 1, "f32")
    c = O.score(s, q, k)
    for h in range(H):
        logits = (k[0, h].double() @ q[0, h, 0].double()).numpy() / math.sqrt(D)
        np.testing.assert_allclose(c[0, h], scipy.special.softmax(logits), rtol=1e-12)


def test_score_equal_keys_closed_form():
    """All keys equal: window row i attends uniformly to its P+i+1 visible
    keys, so c_j = (1/W) sum_{i : j <= P+i} 1/(P+i+1)."""
    L, H, D, T, W = 1, 2, 4, 20, 6
    q, _ = _rand_inputs(L, H, H, D, T, W, 3)
    k = torch.ones(L, H, T, D) * 0.37
    s = O.shape_of(L, H, H, D, T, W, "f32")
    c = O.score(s, q, k)
    P = T - W
    want = np.array([sum(1.0 / (P + i + 1) for i in range(W) if j <= P + i) / W
                     for j in range(T)])
    for h in range(H):
        np.testing.assert_allclose(c[0, h], want, rtol=1e-13)


def test_score_rows_sum_to_one_and_bf16_widening_is_exact():
    """Each softmax row sums to 1, so the window mean sums to 1; bf16 bytes
    decode to exactly the fp32 values they round to."""
    L, Hq, Hkv, D, T, W = 1, 4, 1, 16, 64, 8
    q, k = _rand_inputs(L, Hq, Hkv, D, T, W, 11, dtype="bf16")
    sb = O.shape_of(L, Hq, Hkv, D, T, W, "bf16")
    sf = O.shape_of(L, Hq, Hkv, D, T, W, "f32")
    cb = O.score(sb, q, k)
    cf = O.score(sf, q.float(), k.float())
    assert np.array_equal(cb, cf)
    np.testing.assert_allclose(cb.sum(axis=-1), 1.0, rtol=0, atol=1e-13)


def test_score_unit_matches_all():
    L, Hq, Hkv, D, T, W = 2, 6, 3, 8, 30, 4
    q, k = _rand_inputs(L, Hq, Hkv, D, T, W, 5)
    s = O.shape_of(L, Hq, Hkv, D, T, W, "f32")
    c = O.score(s, q, k)
    assert np.array_equal(O.score_unit(s, q, k, 1, 2), c[1, 2])


# --------------------------------------------------------------------------- a2
def _mba_bruteforce(c, num, den):
    """Fewest entries whose sum reaches num/den of the total, by enumerating
    every subset in exact rational arithmetic (no sorting)."""
    fr = [Fraction(x) for x in c]
    need = Fraction(num, den) * sum(fr)
    for m in range(0, len(c) + 1):
        for sub in itertools.combinations(range(len(c)), m):
            if sum((fr[j] for j in sub), Fraction(0)) >= need:
                return m
    raise AssertionError


@pytest.mark.parametrize("seed", range(12))
def test_mba_bruteforce_subsets(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 12))
    c = rng.dirichlet(np.full(n, 0.3 + seed % 3))
    num, den = [(9, 10), (1, 2), (3, 4)][seed % 3]
    assert O.mba(c, num, den) == _mba_bruteforce(c, num, den)


def test_mba_special_cases():
    # one-hot: a single token holds all the mass
    assert O.mba(np.eye(1, 40, 17).ravel()) == 1
    # uniform over n tokens: ceil(0.9 n) of them are needed
    for n in (1, 7, 10, 33, 1000):
        assert O.mba(np.full(n, 1.0 / n)) == math.ceil(0.9 * n)
    # "reaches" is inclusive: 1/2 + 1/4 is exactly 3/4 of the mass
    assert O.mba(np.array([0.25, 0.5, 0.25]), 3, 4) == 2
    # dyadic masses: 1/2+1/4+1/8 = 0.875 < 0.9, all four are needed
    assert O.mba(np.array([0.125, 0.5, 0.125, 0.25])) == 4
    # no mass at all needs no tokens
    assert O.mba(np.zeros(5)) == 0


def test_mba_permutation_invariant_and_rejects_bad_scores():
    rng = np.random.default_rng(4)
    c = rng.dirichlet(np.ones(300))
    m = O.mba(c)
    for _ in range(3):
        assert O.mba(rng.permutation(c)) == m
    with pytest.raises(ValueError):
        O.mba(np.array([0.5, -0.1, 0.6]))
    with pytest.raises(ValueError):
        O.mba(np.array([0.5, np.nan]))


def test_negative_zero_is_the_score_zero():
    """-0.0 compares equal to +0.0: MBA counts it as no mass and top-K ranks it
    as a zero (ties to the lower position), against the brute-force
    definitions."""
    c = np.zeros(10)
    c[[2, 5, 8]] = [0.5, 0.3, 0.2]
    neg = c.copy()
    neg[[0, 3, 4, 9]] = -0.0
    assert np.signbit(neg).sum() == 4
    for num, den in ((9, 10), (1, 1)):
        assert O.mba(neg, num, den) == O.mba(c, num, den) == _mba_bruteforce(c, num, den)
    for B in (2, 3, 5, 10):
        assert O.topk(neg, 10, B).tolist() == O.topk(c, 10, B).tolist() == _topk_bruteforce(c, B)


# --------------------------------------------------------------------------- a3
def _hamilton_ok(S, R, a):
    """a is a largest-remainder apportionment of R by weights S: every entry
    is floor or ceil of its exact quota and sum(|a-q|) is minimal over all
    non-negative integer vectors summing to R (checked by enumeration)."""
    tot = sum(S) or len(S)
    w = S if sum(S) else [1] * len(S)
    q = [Fraction(R * x, tot) for x in w]
    best = None
    for vec in itertools.product(range(R + 1), repeat=len(S)):
        if sum(vec) != R:
            continue
        dev = sum(abs(v - qq) for v, qq in zip(vec, q))
        if best is None or dev < best[0]:
            best = (dev, [vec])
        elif dev == best[0]:
            best[1].append(vec)
    return tuple(a) in best[1], max(best[1])


@pytest.mark.parametrize("seed", range(10))
def test_budget_bruteforce_largest_remainder(seed):
    rng = np.random.default_rng(100 + seed)
    L = int(rng.integers(1, 5))
    H = int(rng.integers(1, 3))
    mba = rng.integers(0, 9, size=(L, H)).astype(np.int32)
    floor = int(rng.integers(0, 3))
    R = int(rng.integers(0, 10))
    total = L * floor + R
    P = 10_000                                   # no cap
    b = O.budget(mba, P, total, floor)
    a = [int(x) - floor for x in b]
    S = [int(x) for x in mba.sum(axis=1)]
    ok, lex_max = _hamilton_ok(S, R, a)
    assert ok, (S, R, a)
    # remainder ties go to the lower layer: the lexicographically largest
    # optimum
    assert tuple(a) == lex_max


def test_budget_invariants_random():
    rng = np.random.default_rng(9)
    for _ in range(200):
        L = int(rng.integers(1, 40))
        H = int(rng.integers(1, 9))
        P = int(rng.integers(1, 500))
        floor = int(rng.integers(0, P + 1))
        total = int(rng.integers(L * floor, L * P + 50))
        mba = rng.integers(0, 2 * P, size=(L, H)).astype(np.int32)
        b = O.budget(mba, P, total, floor)
        assert b.min() >= floor and b.max() <= P
        assert b.sum() == min(total, L * P)


def test_budget_worked_examples():
    with open(os.path.join(GOLDEN, "budget_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        got = O.budget(np.array(c["mba"], dtype=np.int32), c["prefix"], c["total"], c["floor"])
        assert got.tolist() == c["budget"], c["why"]


def test_budget_equal_lmba_and_errors():
    mba = np.full((8, 4), 17, dtype=np.int32)
    assert O.budget(mba, 1000, 8 * 300, 100).tolist() == [300] * 8
    # 2403 = 8*300 + 3 spare tokens go to the three lowest layers
    assert O.budget(mba, 1000, 2403, 100).tolist() == [301] * 3 + [300] * 5
    # total >= L*P keeps everything
    assert O.budget(mba, 50, 10**6, 10).tolist() == [50] * 8
    with pytest.raises(ValueError):
        O.budget(mba, 1000, 8 * 100 - 1, 100)      # below the floors
    with pytest.raises(ValueError):
        O.budget(mba, 50, 1000, 51)                # floor above the prefix


# --------------------------------------------------------------------------- a4
def _topk_bruteforce(c, B):
    """Among all B-subsets, the largest exact score sum; among those, the
    lexicographically smallest sorted index tuple (lowest indices win ties)."""
    fr = [Fraction(x) for x in c]
    best = None
    for sub in itertools.combinations(range(len(c)), B):
        key = (sum((fr[j] for j in sub), Fraction(0)), tuple(-j for j in sub))
        if best is None or key > best[0]:
            best = (key, sub)
    return list(best[1])


@pytest.mark.parametrize("seed", range(12))
def test_topk_bruteforce(seed):
    rng = np.random.default_rng(200 + seed)
    P = int(rng.integers(1, 11))
    B = int(rng.integers(0, P + 1))
    # few distinct values so that ties are common
    c = rng.integers(0, 4, size=P).astype(np.float64) / 7.0
    assert O.topk(c, P, B).tolist() == _topk_bruteforce(c, B)


def test_topk_special_cases():
    P = 100
    assert O.topk(np.full(P, 0.01), P, 10).tolist() == list(range(10))
    c = np.full(P, 1e-3)
    c[73] = 0.5
    assert 73 in O.topk(c, P, 1).tolist()
    assert O.topk(np.random.default_rng(0).random(P), P, 500).tolist() == list(range(P))
    assert O.topk(np.random.default_rng(0).random(P), P, 0).tolist() == []
    got = O.topk(np.random.default_rng(1).random(P), P, 30)
    assert np.all(np.diff(got) > 0)


# ------------------------------------------------------------- optional pooling
def _pool_shape(L, H, T, W):
    return O.shape_of(L, H, H, 16, T, W, "f32")


@pytest.mark.parametrize("kernel", [1, 3, 5, 7, 31])
def test_pool_average_equals_normalised_convolution(kernel):
    # average of the in-range neighbours == box convolution of the prefix
    # divided by the box convolution of the prefix's indicator ("same" mode)
    L, H, T, W = 2, 3, 257, 17
    P = T - W
    c = np.random.default_rng(kernel).random((L, H, T)) ** 3
    got = O.pool(_pool_shape(L, H, T, W), c, kernel, 0)
    box = np.ones(kernel)
    count = np.convolve(np.ones(P), box, mode="same")
    for l in range(L):
        for h in range(H):
            want = np.convolve(c[l, h, :P], box, mode="same") / count
            np.testing.assert_allclose(got[l, h, :P], want, rtol=1e-13, atol=0)
            np.testing.assert_array_equal(got[l, h, P:], c[l, h, P:])


@pytest.mark.parametrize("kernel", [1, 3, 9, 63])
def test_pool_max_equals_maximum_filter(kernel):
    from scipy.ndimage import maximum_filter1d
    L, H, T, W = 1, 4, 300, 40
    P = T - W
    c = np.random.default_rng(50 + kernel).random((L, H, T))
    got = O.pool(_pool_shape(L, H, T, W), c, kernel, 1)
    for h in range(H):
        want = maximum_filter1d(c[0, h, :P], size=kernel, mode="constant", cval=-np.inf)
        np.testing.assert_array_equal(got[0, h, :P], want)
        np.testing.assert_array_equal(got[0, h, P:], c[0, h, P:])


def test_pool_special_cases():
    L, H, T, W = 1, 2, 64, 8
    s = _pool_shape(L, H, T, W)
    c = np.random.default_rng(3).random((L, H, T))
    np.testing.assert_array_equal(O.pool(s, c, 1, 0), c)           # kernel 1: identity
    np.testing.assert_array_equal(O.pool(s, c, 1, 1), c)
    flat = np.full((L, H, T), 0.125)
    np.testing.assert_allclose(O.pool(s, flat, 15, 0), flat, rtol=1e-15)   # edges stay flat
    # a kernel wider than the prefix averages the whole prefix everywhere
    s2 = _pool_shape(1, 1, 20, 15)
    c2 = np.random.default_rng(4).random((1, 1, 20))
    np.testing.assert_allclose(O.pool(s2, c2, 31, 0)[0, 0, :5], np.full(5, c2[0, 0, :5].mean()),
                               rtol=1e-14)
    assert (O.pool(s2, c2, 31, 1)[0, 0, :5] == c2[0, 0, :5].max()).all()
    for kernel, mode in [(2, 0), (0, 0), (3, 2)]:
        with pytest.raises(ValueError):
            O.pool(s, c, kernel, mode)


def test_pool_keeps_the_neighbours_of_a_spike():
    # the point of pooling before top-K: a one-hot spike pulls its neighbours
    # into the kept set (average ties resolved to the lower index)
    L, H, T, W = 1, 1, 200, 10
    c = np.full((L, H, T), 1e-6)
    c[0, 0, 80] = 1.0
    pooled = O.pool(_pool_shape(L, H, T, W), c, 5, 0)
    assert O.topk(pooled[0, 0], T - W, 5).tolist() == [78, 79, 80, 81, 82]
    assert O.topk(c[0, 0], T - W, 5).tolist() == [0, 1, 2, 3, 80]


# --------------------------------------------------------------------------- a5
def test_compact_equals_fancy_indexing():
    L, H, D, T, W = 3, 2, 8, 40, 5
    P = T - W
    rng = np.random.default_rng(3)
    x = rng.standard_normal((L, H, T, D)).astype(np.float32)
    bud = np.array([4, 0, 35], dtype=np.int32)
    k_max = 35
    idx = np.full((L, H, k_max), -1, dtype=np.int32)
    for l in range(L):
        for h in range(H):
            idx[l, h, : bud[l]] = np.sort(rng.choice(P, bud[l], replace=False))
    s = O.shape_of(L, H, H, D, T, W, "f32")
    out = O.compact(s, x, idx, bud, k_max)
    want = np.concatenate([
        np.concatenate([x[l, h, idx[l, h, : bud[l]]], x[l, h, P:]])
        for l in range(L) for h in range(H)])
    assert out.shape[0] == H * int((bud + W).sum())
    assert np.array_equal(out, want)


# --------------------------------------------------------------------------- a6
def test_keep_channels_formula():
    # the 128K workload: 40% of 128 key channels pruned keeps floor(76.8) = 76
    assert O.keep_channels(0.4, 128) == 76
    assert O.keep_channels(0.5, 128) == 64
    assert O.keep_channels(0.0, 128) == 128


@pytest.mark.parametrize("seed", range(8))
def test_channel_prune_bruteforce(seed):
    """For D <= 8, the kept channels are the keep-subset with the largest
    total squared norm, lowest channel indices winning ties; norms equal
    numpy's l2 norm squared; pruned rows are the kept rows' chosen columns."""
    rng = np.random.default_rng(300 + seed)
    L, H, D, T, W = 2, 2, 6, 12, 3
    P = T - W
    lam = [0.3, 0.5, 0.17][seed % 3]
    keep = O.keep_channels(lam, D)
    bud = np.array([int(rng.integers(0, P + 1)) for _ in range(L)], dtype=np.int32)
    rows = H * int((bud + W).sum())
    k_out = (rng.integers(-3, 4, size=(rows, D)) / 2.0).astype(np.float32)
    s = O.shape_of(L, H, H, D, T, W, "f32")
    chan, norms, kp = O.channel_prune(s, k_out, bud, lam)
    r0, o0 = 0, 0
    for l in range(L):
        n = int(bud[l])
        for h in range(H):
            blk = k_out[r0: r0 + n]
            np.testing.assert_allclose(norms[l, h], np.linalg.norm(blk.astype(np.float64), axis=0) ** 2,
                                       rtol=1e-15, atol=0)
            fr = [Fraction(float(x)) for x in norms[l, h]]
            best = max(itertools.combinations(range(D), keep),
                       key=lambda sub: (sum((fr[d] for d in sub), Fraction(0)), tuple(-d for d in sub)))
            assert chan[l, h].tolist() == list(best)
            got = kp[o0: o0 + n * keep].reshape(n, keep)
            assert np.array_equal(got, blk[:, list(best)])
            r0 += n + W
            o0 += n * keep


def test_channel_prune_keeps_outlier_channels():
    """Keys with 4 channels scaled x8 (the Llama-shaped generators): those
    channels carry far more magnitude and must be among the kept 76."""
    from eviction_kvc_score_gb300 import workloads as wk
    wl = wk.LLAMA3_8B_LAYER.scaled(n_layers=2, seq_len=1024, n_q_heads=8, n_kv_heads=2)
    x = wk.make_inputs(wl, 17)
    k = x["k"]
    L, H, T, D, W = wl.n_layers, wl.n_kv_heads, wl.seq_len, wl.head_dim, wl.window
    P = T - W
    bud = np.array([300, 500], dtype=np.int32)
    idx = np.zeros((L, H, 500), dtype=np.int32)
    for l in range(L):
        for h in range(H):
            idx[l, h, : bud[l]] = np.arange(bud[l])
    s = O.shape_of(L, 8, H, D, T, W, "bf16")
    k_out = O.compact(s, k, idx, bud, 500)
    chan, _, _ = O.channel_prune(s, k_out, bud, 0.4)
    kf = k.float()
    for l in range(L):
        for h in range(H):
            outl = torch.topk(kf[l, h, :P].abs().mean(0), 4).indices.tolist()
            assert set(outl) <= set(chan[l, h].tolist())


# ------------------------------------------------- optional query-driven ThinK
@pytest.mark.parametrize("seed", range(6))
def test_channel_prune_query_bruteforce(seed):
    """Scores equal the squared Frobenius norm of the explicit outer product of
    the stacked window-query column and the kept-key column (numpy, no product
    of norms); for D <= 8 the kept channels are the keep-subset with the
    largest total score, lowest channel indices winning ties; pruned rows are
    the kept rows' chosen columns."""
    rng = np.random.default_rng(700 + seed)
    L, Hq, H, D, T, W = 2, 4, 2, 6, 12, 3
    G = Hq // H
    P = T - W
    lam = [0.3, 0.5, 0.17][seed % 3]
    keep = O.keep_channels(lam, D)
    bud = np.array([int(rng.integers(0, P + 1)) for _ in range(L)], dtype=np.int32)
    rows = H * int((bud + W).sum())
    k_out = (rng.integers(-3, 4, size=(rows, D)) / 2.0).astype(np.float32)
    q = (rng.integers(-3, 4, size=(L, Hq, W, D)) / 4.0).astype(np.float32)
    s = O.shape_of(L, Hq, H, D, T, W, "f32")
    chan, sc, kp = O.channel_prune_query(s, q, k_out, bud, lam)
    r0, o0 = 0, 0
    for l in range(L):
        n = int(bud[l])
        for h in range(H):
            blk = k_out[r0: r0 + n].astype(np.float64)
            qcol = q[l, h * G:(h + 1) * G].reshape(G * W, D).astype(np.float64)
            for d in range(D):
                outer = np.outer(qcol[:, d], blk[:, d])
                assert sc[l, h, d] == pytest.approx(np.linalg.norm(outer, "fro") ** 2, rel=1e-12,
                                                    abs=1e-300)
            fr = [Fraction(float(x)) for x in sc[l, h]]
            best = max(itertools.combinations(range(D), keep),
                       key=lambda sub: (sum((fr[d] for d in sub), Fraction(0)), tuple(-d for d in sub)))
            assert chan[l, h].tolist() == list(best)
            got = kp[o0: o0 + n * keep].reshape(n, keep)
            assert np.array_equal(got, k_out[r0: r0 + n][:, list(best)])
            r0 += n + W
            o0 += n * keep


def test_channel_prune_query_special_cases():
    """Equal query energy in every channel reduces the criterion to the
    magnitude one; a channel the window queries never use (all-zero query
    column) loses to every channel with a positive score."""
    rng = np.random.default_rng(11)
    L, Hq, H, D, T, W = 1, 2, 1, 16, 40, 4
    P = T - W
    bud = np.array([25], dtype=np.int32)
    k_out = rng.standard_normal((H * (25 + W), D)).astype(np.float32)
    s = O.shape_of(L, Hq, H, D, T, W, "f32")
    signs = np.where(rng.random((L, Hq, W, D)) < 0.5, -1.0, 1.0).astype(np.float32)
    q_flat = 0.5 * signs                       # |q| = 0.5 everywhere
    chan_q, _, kp_q = O.channel_prune_query(s, q_flat, k_out, bud, 0.25)
    chan_m, _, kp_m = O.channel_prune(s, k_out, bud, 0.25)
    assert chan_q.tolist() == chan_m.tolist() and np.array_equal(kp_q, kp_m)
    q = rng.standard_normal((L, Hq, W, D)).astype(np.float32)
    k_big = k_out.copy()
    k_big[:, 5] *= 100.0                       # by far the largest key magnitude ...
    q[..., 5] = 0.0                            # ... but no query weight on it
    chan, sc, _ = O.channel_prune_query(s, q, k_big, bud, 0.25)
    assert sc[0, 0, 5] == 0.0 and 5 not in chan[0, 0].tolist()
    chan_mag, _, _ = O.channel_prune(s, k_big, bud, 0.25)
    assert 5 in chan_mag[0, 0].tolist()


# ------------------------------------------- optional per-head and threshold
@pytest.mark.parametrize("seed", range(8))
def test_head_budget_bruteforce_largest_remainder(seed):
    """Each layer's H_kv * B_l tokens are apportioned over its heads by MBA
    with the largest-remainder rule (checked by enumeration), remainder ties
    to the lower head; no cap binds here."""
    rng = np.random.default_rng(900 + seed)
    L = int(rng.integers(1, 4))
    H = int(rng.integers(1, 4))
    mba = rng.integers(0, 7, size=(L, H)).astype(np.int32)
    bud = rng.integers(0, 4, size=L).astype(np.int32)
    hb = O.head_budget(mba, bud, 10_000)
    for l in range(L):
        R = H * int(bud[l])
        ok, lex_max = _hamilton_ok([int(x) for x in mba[l]], R, [int(x) for x in hb[l]])
        assert ok, (mba[l], R, hb[l])
        assert tuple(int(x) for x in hb[l]) == lex_max


def test_head_budget_invariants_and_caps():
    rng = np.random.default_rng(12)
    for _ in range(200):
        L = int(rng.integers(1, 12))
        H = int(rng.integers(1, 9))
        P = int(rng.integers(1, 300))
        bud = rng.integers(0, P + 1, size=L).astype(np.int32)
        mba = rng.integers(0, 3 * P, size=(L, H)).astype(np.int32)
        hb = O.head_budget(mba, bud, P)
        assert hb.min() >= 0 and hb.max() <= P
        assert np.array_equal(hb.sum(axis=1), H * bud.astype(np.int64))
    # equal MBAs: every head gets the layer budget; all-zero MBAs: equal split
    assert O.head_budget(np.full((2, 4), 5, np.int32), np.array([7, 9], np.int32), 50).tolist() \
        == [[7] * 4, [9] * 4]
    assert O.head_budget(np.zeros((1, 3), np.int32), np.array([4], np.int32), 50).tolist() == [[4, 4, 4]]
    # one dominant head is capped at P and the excess is water-filled
    hb = O.head_budget(np.array([[1000, 1, 1, 2]], np.int32), np.array([10], np.int32), 16)
    assert hb[0, 0] == 16 and hb.sum() == 40 and hb[0, 1:].tolist() == [6, 6, 12]


def test_topk_heads_equals_stable_sort():
    rng = np.random.default_rng(5)
    L, H, T, W = 2, 3, 60, 7
    P = T - W
    sc = (rng.integers(0, 5, size=(L, H, T)) / 7.0)
    hb = rng.integers(0, P + 1, size=(L, H)).astype(np.int32)
    s = O.shape_of(L, H, H, 8, T, W, "f32")
    idx = O.topk_heads(s, sc, hb, P)
    for l in range(L):
        for h in range(H):
            order = np.lexsort((np.arange(P), -sc[l, h, :P]))   # score desc, index asc
            want = np.sort(order[: hb[l, h]])
            assert idx[l, h, : hb[l, h]].tolist() == want.tolist()


def test_threshold_select_equals_nonzero():
    rng = np.random.default_rng(6)
    L, H, T, W = 2, 2, 300, 20
    P = T - W
    sc = rng.random((L, H, T)).astype(np.float32) / 100
    s = O.shape_of(L, H, H, 8, T, W, "f32")
    for tau in [0.0, 0.002, 0.005, 0.0099, 1.0]:
        idx, cnt, over = O.threshold_select(s, sc, tau, P)
        assert not over
        for l in range(L):
            for h in range(H):
                want = np.nonzero(sc[l, h, :P] >= np.float32(tau))[0]
                assert cnt[l, h] == want.size and idx[l, h, : want.size].tolist() == want.tolist()
    idx, cnt, _ = O.threshold_select(s, sc, 0.0, P)
    assert (cnt == P).all()                              # tau = 0 keeps the whole prefix
    idx, cnt, over = O.threshold_select(s, sc, 0.0, 50)   # more than k_max: first k_max kept
    assert over and (cnt == P).all() and idx[0, 0].tolist() == list(range(50))


def test_compact_heads_equals_fancy_indexing():
    rng = np.random.default_rng(8)
    L, H, T, W, D = 2, 3, 40, 5, 4
    P = T - W
    x = rng.standard_normal((L, H, T, D)).astype(np.float32)
    cnt = rng.integers(0, P + 1, size=(L, H)).astype(np.int32)
    k_max = P
    idx = np.full((L, H, k_max), -1, np.int32)
    for l in range(L):
        for h in range(H):
            idx[l, h, : cnt[l, h]] = np.sort(rng.choice(P, cnt[l, h], replace=False))
    s = O.shape_of(L, H, H, D, T, W, "f32")
    got = O.compact_heads(s, x, idx, cnt, k_max)
    want = np.concatenate([np.concatenate([x[l, h, idx[l, h, : cnt[l, h]]], x[l, h, P:]])
                           for l in range(L) for h in range(H)])
    assert np.array_equal(got, want)


# ---------------------------------------------------- optional THINKV (values)
@pytest.mark.parametrize("seed", [0, 1])
def test_value_scores_equal_library_attention_output(seed):
    """THINKV channel scores are the squared column norms of the window
    rows' attention output: torch's own scaled-dot-product attention with the
    real V, the causal window mask and the GQA mapping expanded explicitly,
    then summed over each KV head's G*W rows.  Catches a wrong GQA map, mask
    offset, scale, a missing normalisation, |o| instead of o^2 and a sum over
    the wrong axis."""
    L, Hq, Hkv, D, T, W = 2, 6, 2, 8, 31, 4
    G, P = Hq // Hkv, T - W
    q, k = _rand_inputs(L, Hq, Hkv, D, T, W, seed, scale=1.5)
    v = torch.randn(L, Hkv, T, D, generator=torch.Generator().manual_seed(100 + seed))
    s = O.shape_of(L, Hq, Hkv, D, T, W, "f32")
    got = O.value_scores(s, q, k, v)
    kk = k.double().repeat_interleave(G, dim=1)
    vv = v.double().repeat_interleave(G, dim=1)
    mask = torch.arange(T)[None, :] <= (P + torch.arange(W))[:, None]
    out = torch.nn.functional.scaled_dot_product_attention(q.double(), kk, vv, attn_mask=mask)
    want = (out ** 2).view(L, Hkv, G, W, D).sum(dim=(2, 3)).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-300)


def test_value_scores_equal_keys_closed_form():
    """All keys equal: window row i attends uniformly to keys 0..P+i, so its
    output is the mean of those value rows and score_v[d] is the sum over
    rows of that mean squared."""
    L, H, D, T, W = 1, 2, 5, 17, 3
    q, _ = _rand_inputs(L, H, H, D, T, W, 9)
    k = torch.full((L, H, T, D), 0.25)
    v = torch.randn(L, H, T, D, generator=torch.Generator().manual_seed(4))
    s = O.shape_of(L, H, H, D, T, W, "f32")
    got = O.value_scores(s, q, k, v)
    P = T - W
    for h in range(H):
        vv = v[0, h].double().numpy()
        want = sum(vv[: P + i + 1].mean(axis=0) ** 2 for i in range(W))
        np.testing.assert_allclose(got[0, h], want, rtol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_channel_prune_value_selection_bruteforce(seed):
    """Selection = the keep-subset with the largest scores, ties to the lower
    channel (a stable full sort), written ascending; the pruned bytes are
    those channels of each head's kept prefix rows (numpy fancy indexing)."""
    rng = np.random.default_rng(seed)
    L, H, D, T, W, lam = 2, 2, 6, 12, 3, 0.5
    P = T - W
    keep = O.keep_channels(lam, D)
    sv = rng.integers(0, 4, size=(L, H, D)).astype(np.float64)   # many ties
    bud = np.array([4, 9], dtype=np.int32)
    rows = int(H * sum(min(b, P) + W for b in bud))
    v_out = rng.standard_normal((rows, D)).astype(np.float32)
    s = O.shape_of(L, H, H, D, T, W, "f32")
    chan, vp = O.channel_prune_value(s, sv, v_out, bud, lam)
    r0, parts = 0, []
    for l in range(L):
        n = min(int(bud[l]), P)
        for h in range(H):
            best = max(itertools.combinations(range(D), keep),
                       key=lambda c: (sum(sv[l, h, list(c)]), [-x for x in c]))
            assert chan[l, h].tolist() == list(best)
            parts.append(v_out[r0: r0 + n][:, list(best)].ravel())
            r0 += n + W
    assert np.array_equal(vp, np.concatenate(parts))


def test_value_scores_keep_a_dominant_value_channel():
    """A value channel scaled x8 dominates every output column norm, so it is
    always among the kept channels."""
    L, Hq, H, D, T, W = 1, 4, 2, 16, 64, 8
    q, k = _rand_inputs(L, Hq, H, D, T, W, 5)
    g = torch.Generator().manual_seed(6)
    v = torch.randn(L, H, T, D, generator=g) + 0.5
    v[..., 11] *= 8.0
    s = O.shape_of(L, Hq, H, D, T, W, "f32")
    sv = O.value_scores(s, q, k, v)
    bud = np.array([20], dtype=np.int32)
    rows = H * (20 + W)
    chan, _ = O.channel_prune_value(s, sv, np.zeros((rows, D), np.float32), bud, 0.75)
    for h in range(H):
        assert 11 in chan[0, h].tolist()


# ----------------------------------------------------------- optional Keyformer
def test_philox4x32_10_known_answers():
    """Known-answer vectors published with the Philox4x32-10 generator
    (zero counter and key, all-ones counter and key, and the pi-digits
    counter and key)."""
    cases = [((0, 0, 0, 0), (0, 0), (0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8)),
             ((0xffffffff,) * 4, (0xffffffff,) * 2, (0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd)),
             ((0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344), (0xa4093822, 0x299f31d0),
              (0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1))]
    for ctr, key, want in cases:
        assert O.philox4x32_10(ctr, key) == list(want)


def test_keyformer_uniforms_and_gumbel_moments():
    """The draws are strictly inside (0,1) with the right mean, and
    -ln(-ln u) has the Gumbel mean (Euler's gamma) and variance (pi^2/6)."""
    u = np.array([O.keyformer_uniform(7, unit, row, key)
                  for unit in range(4) for row in range(50) for key in range(500)])
    assert u.min() > 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 0.01
    z = -np.log(-np.log(u))
    assert abs(z.mean() - np.euler_gamma) < 0.02
    assert abs(z.var() - np.pi ** 2 / 6) < 0.05
    assert O.keyformer_uniform(7, 1, 2, 3) != O.keyformer_uniform(8, 1, 2, 3)


def test_keyformer_uniforms_of_a_block_are_its_four_words():
    """Four consecutive keys of a row share one Philox4x32-10 block, one word
    each (the published generator is pinned by its known answers above): the
    draws for keys 4m..4m+3 are the block's four words in order, the four
    differ, and neighbouring keys are uncorrelated."""
    seed, unit, row = 0x1234567890ABCDEF, 5, 17
    key = (seed & 0xFFFFFFFF, seed >> 32)
    for m in (0, 1, 1000):
        words = O.philox4x32_10((m, row, unit, 0), key)
        u = [O.keyformer_uniform(seed, unit, row, 4 * m + i) for i in range(4)]
        assert u == [((w >> 8) + 0.5) / 2 ** 24 for w in words]
        assert len(set(u)) == 4
    x = np.array([O.keyformer_uniform(seed, unit, row, j) for j in range(4000)])
    assert abs(np.corrcoef(x[:-1], x[1:])[0, 1]) < 0.05
    assert abs(np.corrcoef(x[0::4], x[1::4])[0, 1]) < 0.08


@pytest.mark.parametrize("tau", [0.5, 1.0, 3.0])
def test_keyformer_single_row_is_noisy_softmax(tau):
    """W = 1, G = 1: the score is one softmax of (q.k/sqrt(D) + zeta)/tau over
    the visible keys, zeta the Gumbel inverse CDF (scipy) of the uniforms."""
    from scipy.stats import gumbel_r
    L, H, D, T, W = 1, 2, 16, 50, 1
    q, k = _rand_inputs(L, H, H, D, T, W, 3)
    s = O.shape_of(L, H, H, D, T, W, "f32")
    c = O.score_keyformer(s, q, k, 99, tau)
    for h in range(H):
        x = k[0, h].double().numpy() @ q[0, h, 0].double().numpy() / np.sqrt(D)
        zeta = gumbel_r.ppf([O.keyformer_uniform(99, h, 0, j) for j in range(T)])
        want = scipy.special.softmax((x + zeta) / tau)
        np.testing.assert_allclose(c[0, h], want, rtol=1e-9, atol=1e-300)


@pytest.mark.parametrize("tau", [0.5, 2.0])
def test_keyformer_grouped_window_equals_library_attention(tau):
    """G > 1, W > 1, finite tau: the Keyformer score equals torch's own
    scaled-dot-product attention with V = identity (the output IS the
    probability matrix), the logits scaled by 1/(sqrt(D) tau), the noise
    zeta/tau (scipy's Gumbel inverse CDF of the uniforms) as an additive
    float mask with -inf on the causal part, the GQA mapping expanded with
    repeat_interleave and the mean taken over each KV head's G*W rows.
    Catches a wrong query-head -> KV-head map (kv + g*H_kv instead of kv*G + g),
    a wrong row index in the noise counter (w instead of g*W + w), the noise
    not divided by tau, and a wrong causal offset."""
    from scipy.stats import gumbel_r
    L, Hq, Hkv, D, T, W = 2, 6, 2, 8, 29, 4
    G, P = Hq // Hkv, T - W
    q, k = _rand_inputs(L, Hq, Hkv, D, T, W, 11, scale=1.5)
    s = O.shape_of(L, Hq, Hkv, D, T, W, "f32")
    seed = 1234
    c = O.score_keyformer(s, q, k, seed, tau)
    zeta = np.empty((L, Hq, W, T))
    for l in range(L):
        for h in range(Hq):
            kv, g = divmod(h, G)
            unit = l * Hkv + kv
            for w in range(W):
                u = [O.keyformer_uniform(seed, unit, g * W + w, j) for j in range(T)]
                zeta[l, h, w] = gumbel_r.ppf(u)
    visible = np.arange(T)[None, :] <= (P + np.arange(W))[:, None]     # [W][T]
    mask = torch.from_numpy(np.where(visible[None, None], zeta / tau, -np.inf))
    kk = k.double().repeat_interleave(G, dim=1)                          # [L][Hq][T][D]
    eye = torch.eye(T, dtype=torch.float64).expand(L, Hq, T, T)
    probs = torch.nn.functional.scaled_dot_product_attention(
        q.double(), kk, eye, attn_mask=mask, scale=1.0 / (math.sqrt(D) * tau))
    ref = probs.view(L, Hkv, G, W, T).mean(dim=(2, 3)).numpy()
    np.testing.assert_allclose(c, ref, rtol=1e-10, atol=1e-300)


def test_keyformer_rows_sum_to_one_and_hot_temperature_is_uniform():
    L, Hq, H, D, T, W = 2, 4, 2, 8, 40, 5
    q, k = _rand_inputs(L, Hq, H, D, T, W, 4)
    s = O.shape_of(L, Hq, H, D, T, W, "f32")
    c = O.score_keyformer(s, q, k, 5, 1.0)
    np.testing.assert_allclose(c.sum(-1), 1.0, rtol=1e-12)
    # a very hot temperature flattens every row to 1/(visible keys)
    hot = O.score_keyformer(s, q, k, 5, 1e12)
    P = T - W
    want = np.zeros(T)
    for i in range(W):
        want[: P + i + 1] += 1.0 / (P + i + 1) / W
    for l in range(L):
        for h in range(H):
            np.testing.assert_allclose(hot[l, h], want, rtol=1e-9)
    # different seeds give different scores; the same seed the same scores
    assert not np.array_equal(c, O.score_keyformer(s, q, k, 6, 1.0))
    assert np.array_equal(c, O.score_keyformer(s, q, k, 5, 1.0))


# --------------------------------------------------------------------- end to end
def test_tiny_planted_keys_are_selected():
    """The tiny MHA workload plants 4 keys per head equal to 3x the head's mean
    window query; with this seed each lands in its head's top-128.  A much
    stronger plant (logit far above every random one) must always be kept."""
    from eviction_kvc_score_gb300 import workloads as wk
    wl = wk.TINY
    x = wk.make_inputs(wl, wk.seed_for(0))
    s = O.shape_of(wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.seq_len,
                   wl.window, wl.dtype)
    c = O.score(s, x["q"], x["k"])
    P = wl.prefix_len
    for h in range(wl.n_kv_heads):
        sel = set(O.topk(c[0, h, :P], P, wl.per_head_budget).tolist())
        assert set(x["planted"][0, h].tolist()) <= sel
    k2 = x["k"].clone()
    qm = x["q"][0].mean(dim=1)                     # [H][D]
    for h in range(wl.n_kv_heads):
        k2[0, h, 400] = 40.0 * qm[h]
    c2 = O.score(s, x["q"], k2)
    for h in range(wl.n_kv_heads):
        assert 400 in O.topk(c2[0, h, :P], P, 1).tolist()


def test_compress_chains_the_steps():
    from eviction_kvc_score_gb300 import workloads as wk
    wl = wk.ZIGZAG_32K.scaled(n_layers=3, seq_len=300, window=16, n_q_heads=4,
                              n_kv_heads=2, head_dim=16, total_budget=3 * 40,
                              layer_floor=8, think_lambda=0.25)
    x = wk.make_inputs(wl, 21)
    s = O.shape_of(wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.seq_len,
                   wl.window, wl.dtype)
    total, floor = wl.budget_args()
    out = O.compress(s, x["q"], x["k"], x["v"], total, floor, wl.k_max, lam=wl.think_lambda)
    c = O.score(s, x["q"], x["k"])
    assert np.array_equal(out["scores"], c)
    m = O.mba_all(s, c)
    assert np.array_equal(out["mba"], m)
    b = O.budget(m, wl.prefix_len, total, floor)
    assert np.array_equal(out["budget"], b) and b.sum() == total
    idx = O.topk_all(s, c, b, wl.k_max)
    for l in range(wl.n_layers):
        assert np.array_equal(out["idx"][l, :, : b[l]], idx[l, :, : b[l]])
    assert np.array_equal(out["k_out"], O.compact(s, x["k"], idx, b, wl.k_max))
    assert np.array_equal(out["v_out"], O.compact(s, x["v"], idx, b, wl.k_max))
    chan, _, kp = O.channel_prune(s, out["k_out"], b, wl.think_lambda)
    assert np.array_equal(out["chan"], chan) and np.array_equal(out["k_pruned"], kp)

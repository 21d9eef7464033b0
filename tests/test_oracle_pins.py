"""Pins of the fp64 oracle against what the MagicPIG pages and the mathematics fix.

None of these retypes an oracle formula and compares it with itself. Each check comes from
somewhere else: Monte-Carlo over fresh hyperplanes, exact rational arithmetic, brute-force loops
on tiny inputs, textbook attention special cases, invariances, and the pages' own numbers.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))


def _pair_at_angle(theta, d=3):
    x = np.zeros(d)
    y = np.zeros(d)
    x[0] = 1.0
    y[0], y[1] = math.cos(theta), math.sin(theta)
    return x, y


def _brute_attention(q, keys, values, scale):
    """Softmax attention written as scalar loops (independent of numpy's vector forms)."""
    s = [scale * sum(qe * ke for qe, ke in zip(q, k)) for k in keys]
    m = max(s)
    w = [math.exp(si - m) for si in s]
    z = sum(w)
    d = len(values[0])
    return np.array([sum(w[i] * values[i][e] for i in range(len(keys))) / z for e in range(d)])


# ------------------------------------------------------------------------------------------------
# SimHash: one hyperplane separates two vectors with probability theta/pi
# ("LSH Sampling..." background, LSH basics; "don't pick the tallest" section 5)
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("deg", [10, 45, 90, 135, 170])
def test_simhash_bit_agreement_is_one_minus_theta_over_pi(deg):
    rng = np.random.default_rng(1000 + deg)
    theta = math.radians(deg)
    x, y = _pair_at_angle(theta, d=5)
    N = 100_000
    W = rng.standard_normal((5, N))
    bx = O.sign_bits(O.simhash_projections(x[None], W))[0]
    by = O.sign_bits(O.simhash_projections(y[None], W))[0]
    freq = float(np.mean(bx == by))
    p = 1 - theta / math.pi
    sigma = math.sqrt(p * (1 - p) / N)
    assert abs(freq - p) < 4.5 * sigma, (freq, p, sigma)


# ------------------------------------------------------------------------------------------------
# u(p): the chance that a key collides in at least 2 of L tables of K bits
# ("LSH Sampling..." hash-function choice and the u_i formula; "don't pick the tallest" section 5)
# ------------------------------------------------------------------------------------------------
def _exact_tail(p: Fraction, K: int, L: int) -> Fraction:
    x = p ** K
    return sum(Fraction(math.comb(L, j)) * x ** j * (1 - x) ** (L - j) for j in range(2, L + 1))


@pytest.mark.parametrize("K,L", [(2, 3), (3, 5), (8, 75), (9, 120), (10, 150), (11, 300)])
@pytest.mark.parametrize("p", [Fraction(1, 8), Fraction(1, 4), Fraction(1, 2), Fraction(5, 8),
                               Fraction(3, 4), Fraction(7, 8), Fraction(15, 16),
                               Fraction(99, 100)])
def test_log_u_matches_exact_rational_binomial_tail(K, L, p):
    exact = _exact_tail(p, K, L)
    assert exact > 0
    got = float(O.log_inclusion_probability(float(p), K, L)[0])
    want = math.log(exact.numerator) - math.log(exact.denominator)
    assert abs(got - want) < 1e-11 * max(1.0, abs(want)), (got, want)


def test_log_u_both_branches_near_the_switch():
    # L p^K = 1/2 is where the evaluation switches branch; check either side against exact tails
    K, L = 10, 150
    p_switch = (0.5 / L) ** (1 / K)
    for f in (0.97, 0.999, 1.0, 1.001, 1.03):
        p = Fraction(p_switch * f).limit_denominator(10**9)
        exact = _exact_tail(p, K, L)
        got = float(O.log_inclusion_probability(float(p), K, L)[0])
        want = math.log(exact.numerator) - math.log(exact.denominator)
        assert abs(got - want) < 1e-11 * abs(want)


def test_log_u_special_values():
    assert O.log_inclusion_probability(1.0, 10, 150)[0] == 0.0          # u(1) = 1
    assert O.log_inclusion_probability(0.7, 0, 150)[0] == 0.0           # K = 0: p^0 = 1, u = 1
    assert O.log_inclusion_probability(0.0, 10, 150)[0] == O.LOG_DBL_MIN  # clamped u(0) = 0
    for p in (0.0, 0.3, 1.0):
        assert O.log_inclusion_probability(p, 10, 1)[0] == -math.inf    # L = 1: never 2 hits
    ps = np.linspace(0.01, 1.0, 400)
    lu = O.log_inclusion_probability(ps, 10, 150)
    assert np.all(np.diff(lu) >= 0)                                   # monotone in p,
    assert np.all(np.diff(lu)[lu[1:] < -1e-9] > 0)                    # strictly below u = 1


@pytest.mark.parametrize("K,L,target_u,trials", [(2, 3, 0.5, 6000), (3, 5, 0.35, 6000),
                                                 (8, 75, 0.5, 3000), (10, 150, 0.3, 2000),
                                                 (10, 150, 0.7, 2000)])
def test_u_matches_monte_carlo_collision_frequency(K, L, target_u, trials):
    # pick the angle whose u is target_u, then count >= 2 collisions over fresh hyperplanes
    lo, hi = 0.0, 1.0
    for _ in range(60):
        mid = (lo + hi) / 2
        if O.inclusion_probability(mid, K, L)[0] < target_u:
            lo = mid
        else:
            hi = mid
    p = (lo + hi) / 2
    theta = (1 - p) * math.pi
    q, k = _pair_at_angle(theta, d=3)
    rng = np.random.default_rng(7 * K + L)
    W = rng.standard_normal((3, trials * K * L))
    kc = O.encode_keys(k[None], np.zeros(3), W, K, trials * L)[0].reshape(trials, L)
    qc = O.encode_query(q, W, K, trials * L)[0].reshape(trials, L)
    hits = np.array([O.collision_counts(kc[t][None], qc[t])[0] >= 2 for t in range(trials)])
    freq = float(hits.mean())
    u = float(O.inclusion_probability(p, K, L)[0])
    sigma = math.sqrt(u * (1 - u) / trials)
    assert abs(freq - u) < 4.5 * sigma, (freq, u, sigma)


# ------------------------------------------------------------------------------------------------
# Codes, counts and the sample set, by brute force on tiny inputs
# ------------------------------------------------------------------------------------------------
def _brute_codes(keys, centre, W, K, L):
    n, d = len(keys), len(centre)
    out = []
    for i in range(n):
        row = []
        for t in range(L):
            code = 0
            for b in range(K):
                col = t * K + b
                proj = sum(W[e][col] * (keys[i][e] - centre[e]) for e in range(d))
                if proj > 0:
                    code += 2 ** b
            row.append(code)
        out.append(row)
    return out


def test_key_centre_is_the_mean_over_all_n_keys_by_scalar_loops():
    # "LSH Sampling..." data preprocessing: mu = (1/n) sum_{i=1..n} k_i; integer-valued keys
    # make every partial sum exact, so a divide by n - 1 or a dropped row cannot pass
    rng = np.random.default_rng(31)
    for n, d in ((1, 3), (7, 5), (64, 4)):
        keys = rng.integers(-40, 41, size=(n, d)).astype(np.float64)
        want = [Fraction(sum(int(keys[i][e]) for i in range(n)), n) for e in range(d)]
        got = O.key_centre(keys)
        assert [Fraction(float(x)).limit_denominator(10 ** 6) for x in got] == want


def _band_offset(c: float, rest_norm2: float) -> float:
    """delta with delta = c * 1e-5 * sqrt(delta^2 + rest_norm2): a vector (delta, rest) whose
    projection delta * |w| on w = |w| e_0 sits at c times the band 1e-5 |w| |x|."""
    t = c * 1e-5
    return t * math.sqrt(rest_norm2) / math.sqrt(1.0 - t * t)


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_key_near_tie_band_edges(sign):
    # the band is |w_j . (k_i - mu)| < 1e-5 |w_j| |k_i| with the RAW key norm: the key
    # (delta, 0, 8, 4) has centred part (delta, 0, 3, 4) for mu = (0, 0, 5, 0); w_0 = 7 e_0
    mu = np.array([0.0, 0.0, 5.0, 0.0])
    W = np.zeros((4, 2))
    W[0, 0] = 7.0
    W[:, 1] = [0.0, 3.0, 0.0, 4.0]
    for c, inside in ((0.999, True), (1.001, False), (0.5, True), (2.0, False)):
        delta = sign * _band_offset(c, 8.0 ** 2 + 4.0 ** 2)
        key = np.array([[delta, 0.0, 8.0, 4.0]])
        _, bits, near = O.encode_keys(key, mu, W, 1, 2)
        assert bool(near[0, 0]) is inside, (c, sign)
        assert bool(bits[0, 0]) is (sign > 0)
        assert not near[0, 1]                      # projection 16, far from the band


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_query_near_tie_band_edges(sign):
    # the query is not centred: |w_j . q| < 1e-5 |w_j| |q|, here q = (delta, 0, 3, 4), w_0 = 7 e_0
    W = np.zeros((4, 1))
    W[0, 0] = 7.0
    for c, inside in ((0.999, True), (1.001, False)):
        q = np.array([sign * _band_offset(c, 25.0), 0.0, 3.0, 4.0])
        _, bits, near = O.encode_query(q, W, 1, 1)
        assert bool(near[0, 0]) is inside, (c, sign)
        assert bool(bits[0, 0]) is (sign > 0)


def test_replay_takes_every_flip_inside_the_band_and_rejects_any_outside():
    rng = np.random.default_rng(32)
    ob = rng.random((6, 40)) < 0.5
    near = rng.random((6, 40)) < 0.3
    other = ob.copy()
    flips = near & (rng.random((6, 40)) < 0.5)
    other[flips] = ~other[flips]
    got, count = O.replay_bits(ob, near, other)
    assert count == int(flips.sum()) > 0
    assert np.array_equal(got, other)              # every flip in the band is taken
    assert np.array_equal(O.replay_bits(ob, near, ob)[0], ob) and O.replay_bits(ob, near, ob)[1] == 0
    i, j = np.argwhere(~near)[0]
    bad = other.copy()
    bad[i, j] = ~bad[i, j]                          # one flip outside the band
    with pytest.raises(AssertionError):
        O.replay_bits(ob, near, bad)


def test_estimate_is_the_weighted_ratio_by_scalar_loops():
    # o = (sum_S e^{s_i}/u_i v_i + sum_T e^{s_i} v_i) / (sum_S e^{s_i}/u_i + sum_T e^{s_i}),
    # evaluated with 60-digit arithmetic; the sampled scores sit 700 above the exact ones in the
    # second case (plain exponentials of either would overflow a double)
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 60
    rng = np.random.default_rng(33)
    d = 6
    for shift in (0.0, 700.0):
        KS = rng.standard_normal((4, d))
        VS = rng.standard_normal((4, d))
        KT = rng.standard_normal((3, d))
        VT = rng.standard_normal((3, d))
        q = rng.standard_normal(d)
        u = rng.uniform(0.01, 1.0, size=4)
        scale = 0.9
        sS = [mpmath.mpf(scale * float(KS[i] @ q)) + shift for i in range(4)]
        sT = [mpmath.mpf(scale * float(KT[i] @ q)) for i in range(3)]
        wS = [mpmath.exp(sS[i]) / mpmath.mpf(u[i]) for i in range(4)]
        wT = [mpmath.exp(x) for x in sT]
        den = sum(wS) + sum(wT)
        want = [float((sum(wS[i] * VS[i][e] for i in range(4)) +
                       sum(wT[i] * VT[i][e] for i in range(3))) / den) for e in range(d)]
        KS_shift = KS + (shift / scale) * q / float(q @ q)   # raises each sampled score by shift
        got = O.snis_attention(q, KS_shift, VS, np.log(u), KT, VT, scale)
        assert np.allclose(got, want, rtol=0, atol=1e-9)
    # only one of the two parts present
    assert np.allclose(O.snis_attention(q, KS[:0], VS[:0], np.zeros(0), KT, VT, scale),
                       _brute_attention(q.tolist(), KT.tolist(), VT.tolist(), scale), atol=1e-13)


def test_codes_counts_and_set_by_brute_force():
    rng = np.random.default_rng(3)
    d, n, K, L = 3, 9, 2, 3
    keys = rng.standard_normal((n, d)) + np.array([2.0, -1.0, 0.5])
    W = rng.standard_normal((d, K * L))
    centre = keys.mean(axis=0)
    q = rng.standard_normal(d)
    codes, _, _ = O.encode_keys(keys, centre, W, K, L)
    assert codes.tolist() == _brute_codes(keys.tolist(), centre.tolist(), W.tolist(), K, L)
    qcode = O.encode_query(q, W, K, L)[0][0]
    want_q = _brute_codes([q.tolist()], [0.0] * d, W.tolist(), K, L)[0]
    assert qcode.tolist() == want_q
    cnt = O.collision_counts(codes, qcode)
    brute_cnt = [sum(1 for t in range(L) if codes[i][t] == want_q[t]) for i in range(n)]
    assert cnt.tolist() == brute_cnt
    T = O.exact_set_mask(n, 1, 2)
    assert T.tolist() == [True] + [False] * (n - 3) + [True, True]
    S = O.sampled_set(cnt, T)
    assert S.tolist() == [i for i in range(n) if brute_cnt[i] >= 2 and not T[i]]


def test_bucket_tables_by_brute_force():
    """Buckets hold exactly the keys of their code, ascending; the query's buckets count each
    key once per table it shares ("LSH Sampling..." system co-design item 3; "don't pick the
    tallest" section 6). The counts are checked against scalar loops over the codes."""
    rng = np.random.default_rng(21)
    n, K, L = 37, 3, 5
    codes = rng.integers(0, 1 << K, size=(n, L))
    offsets, members = O.bucket_tables(codes, K, L)
    for t in range(L):
        assert offsets[t, 0] == 0 and offsets[t, -1] == n
        for c in range(1 << K):
            got = members[t, offsets[t, c]:offsets[t, c + 1]].tolist()
            assert got == [i for i in range(n) if codes[i][t] == c]
    for _ in range(5):
        qc = rng.integers(0, 1 << K, size=L)
        brute = [sum(1 for t in range(L) if codes[i][t] == qc[t]) for i in range(n)]
        assert O.bucket_collision_counts(offsets, members, qc, n).tolist() == brute


def test_scanned_entries_average_the_pages_figure():
    """With evenly filled buckets a query scans L n / 2^K entries: 14,400 at n = 98,304 and
    (10, 150) ("don't pick the tallest", section 6). Uniform random codes stand in for evenly
    filled buckets; the mean over random queries must sit within a few standard errors."""
    g = json.load(open(os.path.join(HERE, "golden", "page_arithmetic.json")))
    n, K, L = 98304, 10, 150
    rng = np.random.default_rng(22)
    codes = rng.integers(0, 1 << K, size=(n, L))
    offsets, _ = O.bucket_tables(codes, K, L)
    sizes = np.diff(offsets, axis=1)                       # [L, 2^K]
    scanned = [int(sizes[np.arange(L), rng.integers(0, 1 << K, size=L)].sum()) for _ in range(64)]
    se = math.sqrt(L * n * 2.0 ** -K) / math.sqrt(len(scanned))   # binomial bucket sizes
    assert abs(np.mean(scanned) - g["entries_scanned_per_query"]["value"]) < 5 * se
    assert 4 * L * n // (1 << K) == g["index_bytes_scanned_per_query"]["value"]


def test_key_along_query_collides_in_every_table():
    rng = np.random.default_rng(4)
    d, K, L = 16, 10, 150
    W = rng.standard_normal((d, K * L))
    q = rng.standard_normal(d)
    mu = rng.standard_normal(d) * 3
    keys = np.stack([mu + s * q for s in (0.01, 1.0, 250.0)])
    codes, _, _ = O.encode_keys(keys, mu, W, K, L)
    qcode = O.encode_query(q, W, K, L)[0][0]
    assert O.collision_counts(codes, qcode).tolist() == [L, L, L]


def test_negated_centred_key_flips_every_bit():
    rng = np.random.default_rng(5)
    d, K, L = 32, 8, 75
    W = rng.standard_normal((d, K * L))
    mu = rng.standard_normal(d)
    k = rng.standard_normal((20, d)) + mu
    _, bits, _ = O.encode_keys(k, mu, W, K, L)
    _, bits_neg, _ = O.encode_keys(2 * mu - k, mu, W, K, L)
    assert np.array_equal(bits, ~bits_neg)


def test_zero_length_vectors():
    rng = np.random.default_rng(6)
    d, K, L = 8, 4, 6
    W = rng.standard_normal((d, K * L))
    _, qbits, _ = O.encode_query(np.zeros(d), W, K, L)
    assert not qbits.any()                               # strict > 0
    p = O.collision_probability(np.zeros(d), rng.standard_normal((3, d)))
    assert np.all(p == 0.5)
    p = O.collision_probability(rng.standard_normal(d), np.zeros((2, d)))
    assert np.all(p == 0.5)


# ------------------------------------------------------------------------------------------------
# The estimator
# ------------------------------------------------------------------------------------------------
def test_full_attention_textbook_cases():
    rng = np.random.default_rng(8)
    keys = np.zeros((5, 4))
    vals = rng.standard_normal((5, 3))
    q = rng.standard_normal(4)
    assert np.allclose(O.full_attention(q, keys, vals, 1.0), vals.mean(axis=0), atol=1e-15)
    keys2 = rng.standard_normal((5, 4)) * 0.01
    keys2[2] = q * 1000
    assert np.allclose(O.full_attention(q, keys2, vals, 1.0), vals[2], atol=1e-12)
    keys3 = rng.standard_normal((7, 4))
    vals3 = rng.standard_normal((7, 4))
    assert np.allclose(O.full_attention(q, keys3, vals3, 0.5),
                       _brute_attention(q.tolist(), keys3.tolist(), vals3.tolist(), 0.5),
                       atol=1e-13)


def test_K0_reduces_to_full_softmax_attention():
    # K = 0: empty codes always agree, every key collides in all L >= 2 tables, u = 1
    rng = np.random.default_rng(9)
    d, n = 16, 50
    keys = rng.standard_normal((n, d)) + 1.5
    vals = rng.standard_normal((n, d))
    q = rng.standard_normal(d)
    W = np.zeros((d, 0))
    mu = O.key_centre(keys)
    kc, _, _ = O.encode_keys(keys, mu, W, 0, 4)
    qc = O.encode_query(q, W, 0, 4)[0][0]
    r = O.decode_head(q, keys, vals, mu, kc, qc, 0, 4, n_sink=2, n_local=5)
    assert r["S"].tolist() == list(range(2, n - 5))
    assert np.all(r["logu"] == 0.0)
    want = _brute_attention(q.tolist(), keys.tolist(), vals.tolist(), 1 / math.sqrt(d))
    assert np.allclose(r["o"], want, rtol=0, atol=1e-13)


def test_half_inclusion_probability_equals_a_duplicated_key():
    # weight exp(s - log u) with u = 1/2 counts the key twice: same as attention over a multiset
    rng = np.random.default_rng(10)
    d = 8
    KS = rng.standard_normal((3, d))
    VS = rng.standard_normal((3, d))
    KT = rng.standard_normal((2, d))
    VT = rng.standard_normal((2, d))
    q = rng.standard_normal(d)
    got = O.snis_attention(q, KS, VS, np.array([math.log(0.5), 0.0, math.log(0.25)]), KT, VT,
                           0.7)
    mk = [KS[0], KS[0], KS[1], KS[2], KS[2], KS[2], KS[2], KT[0], KT[1]]
    mv = [VS[0], VS[0], VS[1], VS[2], VS[2], VS[2], VS[2], VT[0], VT[1]]
    want = _brute_attention(q.tolist(), [k.tolist() for k in mk], [v.tolist() for v in mv], 0.7)
    assert np.allclose(got, want, atol=1e-13)


def test_single_table_leaves_only_the_exact_set():
    # L = 1: no key can collide in two tables, S is empty, o = exact attention over T
    rng = np.random.default_rng(11)
    d, n = 16, 40
    keys = rng.standard_normal((n, d))
    vals = rng.standard_normal((n, d))
    q = rng.standard_normal(d)
    W = rng.standard_normal((d, 3))
    mu = O.key_centre(keys)
    kc, _, _ = O.encode_keys(keys, mu, W, 3, 1)
    qc = O.encode_query(q, W, 3, 1)[0][0]
    r = O.decode_head(q, keys, vals, mu, kc, qc, 3, 1, n_sink=3, n_local=4)
    assert r["S"].size == 0
    T = list(range(3)) + list(range(n - 4, n))
    want = _brute_attention(q.tolist(), keys[T].tolist(), vals[T].tolist(), 1 / math.sqrt(d))
    assert np.allclose(r["o"], want, atol=1e-13)


def test_empty_sample_and_exact_sets_give_zero():
    d = 4
    o = O.snis_attention(np.ones(d), np.zeros((0, d)), np.zeros((0, d)), np.zeros(0),
                         np.zeros((0, d)), np.zeros((0, d)), 1.0)
    assert np.array_equal(o, np.zeros(d))


def test_centring_leaves_the_output_unchanged():
    # every score shifts by q.mu, which the softmax ignores ("don't pick the tallest" section 5)
    rng = np.random.default_rng(12)
    d, n, K, L = 32, 300, 4, 12
    mu = rng.standard_normal(d) * 4
    keys = rng.standard_normal((n, d)) + mu
    vals = rng.standard_normal((n, d))
    q = -mu / np.linalg.norm(mu) + 0.3 * rng.standard_normal(d)
    W = rng.standard_normal((d, K * L))
    c = O.key_centre(keys)
    kc, _, _ = O.encode_keys(keys, c, W, K, L)
    qc = O.encode_query(q, W, K, L)[0][0]
    a = O.decode_head(q, keys, vals, c, kc, qc, K, L, 2, 8)
    b = O.decode_head(q, keys, vals, c, kc, qc, K, L, 2, 8, centred_scores=True)
    assert a["S"].size > 10
    assert np.allclose(a["o"], b["o"], rtol=0, atol=1e-12)


def test_importance_weights_are_unbiased_over_hyperplane_draws():
    # Horvitz-Thompson: E[sum_{i in S} f_i / u_i] = sum_i f_i exactly when u_i = P[i in S].
    # This fails for a wrong u, a wrong sign of log u, or a wrong ">= 2 tables" rule.
    rng = np.random.default_rng(13)
    d, n, K, L, M = 6, 40, 2, 6, 20000
    keys = rng.standard_normal((n, d))
    vals = rng.standard_normal((n, d))
    q = rng.standard_normal(d)
    mu = O.key_centre(keys)
    scale = 1 / math.sqrt(d)
    s = keys @ q * scale
    logu = O.log_inclusion_probability(O.collision_probability(q, keys - mu), K, L)
    W = rng.standard_normal((d, M * K * L))
    kc = O.encode_keys(keys, mu, W, K, M * L)[0].reshape(n, M, L)
    qc = O.encode_query(q, W, K, M * L)[0][0].reshape(M, L)
    T = O.exact_set_mask(n, 0, 0)
    num = np.zeros((M, d))
    den = np.zeros(M)
    for m in range(M):
        S = O.sampled_set(O.collision_counts(kc[:, m, :], qc[m]), T)
        wS = np.exp(s[S] - logu[S])
        num[m] = wS @ vals[S]
        den[m] = wS.sum()
    want_num = np.exp(s) @ vals
    want_den = np.exp(s).sum()
    se_den = den.std(ddof=1) / math.sqrt(M)
    assert abs(den.mean() - want_den) < 4.5 * se_den, (den.mean(), want_den, se_den)
    se_num = num.std(axis=0, ddof=1) / math.sqrt(M)
    assert np.all(np.abs(num.mean(axis=0) - want_num) < 4.5 * se_num + 1e-12)


def test_expected_sample_size_is_the_sum_of_inclusion_probabilities():
    rng = np.random.default_rng(14)
    d, n, K, L, M = 128, 1024, 8, 75, 60
    mu = rng.standard_normal(d)
    mu *= 8 / np.linalg.norm(mu)
    keys = rng.standard_normal((n, d)) + mu
    q = -4 * mu / 8 + 0.5 * rng.standard_normal(d)
    c = O.key_centre(keys)
    T = O.exact_set_mask(n, 4, 64)
    u = O.inclusion_probability(O.collision_probability(q, keys - c), K, L)
    want = u[~T].sum()
    sizes = []
    for m in range(M):
        W = rng.standard_normal((d, K * L))
        kc, _, _ = O.encode_keys(keys, c, W, K, L)
        qc = O.encode_query(q, W, K, L)[0][0]
        sizes.append(O.sampled_set(O.collision_counts(kc, qc), T).size)
    sizes = np.array(sizes, dtype=float)
    se = sizes.std(ddof=1) / math.sqrt(M)
    assert abs(sizes.mean() - want) < 4.5 * se + 0.5, (sizes.mean(), want, se)


def test_without_centring_almost_no_key_is_sampled():
    # "don't pick the tallest" section 5 / "LSH Sampling..." ablation: raw keys sit in one cone
    # away from the query, so they rarely share its buckets; centring brings them back
    import torch
    from workloads import WORKLOADS, make_hyperplanes, make_layer
    wl = WORKLOADS["tiny_f32_n4096"]
    x = make_layer(wl, 0)
    W = make_hyperplanes(wl)
    keys = x["keys"][0, 0]
    q = x["q"][0, 0]
    T = O.exact_set_mask(wl.n, wl.n_sink, wl.n_local)
    qc = O.encode_query(q, W, wl.K, wl.L)[0][0]
    frac = {}
    for name, c in (("centred", O.key_centre(keys)), ("raw", np.zeros(wl.d))):
        kc, _, _ = O.encode_keys(keys, c, W, wl.K, wl.L)
        frac[name] = O.sampled_set(O.collision_counts(kc, qc), T).size / (~T).sum()
    assert frac["raw"] < 0.005 and frac["centred"] > 0.01, frac
    assert frac["raw"] < 0.25 * frac["centred"], frac
    del torch


# ------------------------------------------------------------------------------------------------
# The pages' own arithmetic, re-derived from the workload shapes
# ------------------------------------------------------------------------------------------------
def test_page_arithmetic_matches_the_96k_workload():
    from workloads import WORKLOADS
    g = json.load(open(os.path.join(HERE, "golden", "page_arithmetic.json")))
    wl = WORKLOADS["llama8b_n96k_32layers"]
    per_token = wl.layers * wl.Hkv * wl.d * 2 * 2
    assert per_token == g["kv_bytes_per_token"]["value"]
    assert per_token * wl.n == g["kv_bytes_96k_context"]["value"]
    assert 4 * wl.L == g["table_entry_bytes_per_key"]["value"]
    tables = 4 * wl.L * wl.n * wl.layers * wl.Hkv
    assert abs(tables / 2**30 - g["table_bytes_96k_gib"]["value"]) < 0.05
    entries = wl.L * wl.n // 2**wl.K
    assert entries == g["entries_scanned_per_query"]["value"]
    assert 4 * entries == g["index_bytes_scanned_per_query"]["value"]
    key_bytes = wl.n * wl.d * 2
    assert key_bytes == g["key_bytes_one_head_one_layer"]["value"]
    assert abs(100 * 4 * entries / key_bytes - g["scan_fraction_percent"]["value"]) < 0.005
    projector = wl.d * wl.C * 2                    # bf16 projector
    assert abs(projector / 1000 - g["projector_kb"]["value"]) < 0.05 * g["projector_kb"]["value"]


# ------------------------------------------------------------------------------------------------
# MIPS -> cosine variant ("LSH Sampling..." method details, variance reduction with LSH: keys
# extended by sqrt(r^2 - |k|^2), the query by 0, r the longest key; here the centred keys)
# ------------------------------------------------------------------------------------------------
def _mips_case(seed, n=12, d=5):
    rng = np.random.default_rng(seed)
    keys = rng.standard_normal((n, d)) * rng.uniform(0.3, 2.0, size=(n, 1))
    q = rng.standard_normal(d)
    return keys, q, O.key_centre(keys)


def test_mips_radius_and_extended_lengths():
    keys, q, mu = _mips_case(21)
    want_r = max(math.sqrt(sum((k[e] - mu[e]) ** 2 for e in range(len(mu)))) for k in keys)
    r = O.mips_radius(keys, mu)
    assert abs(r - want_r) < 1e-12
    khat = O.mips_augment_keys(keys, mu, r)
    assert np.allclose(np.linalg.norm(khat, axis=1), r, rtol=0, atol=1e-12)
    assert np.allclose(khat[:, :-1], keys - mu, rtol=0, atol=0)
    assert np.all(khat[:, -1] >= 0)
    assert O.mips_augment_query(q).tolist() == [list(q) + [0.0]]


def test_mips_probability_is_the_plain_cosine_of_the_extended_pair():
    keys, q, mu = _mips_case(22)
    r = O.mips_radius(keys, mu)
    plain = O.collision_probability(O.mips_augment_query(q)[0], O.mips_augment_keys(keys, mu, r))
    assert np.allclose(O.collision_probability_mips(q, keys - mu, r), plain, rtol=0, atol=1e-12)


def test_mips_bit_agreement_monte_carlo():
    # each extended key agrees with the query on one hyperplane of d + 1 rows with probability
    # p_mips; the query's bits come from the first d rows only
    keys, q, mu = _mips_case(23, n=4)
    r = O.mips_radius(keys, mu)
    rng = np.random.default_rng(24)
    N = 100_000
    W = rng.standard_normal((keys.shape[1] + 1, N))
    _, kbits, _ = O.encode_keys_mips(keys, mu, W, r, 1, N)
    _, qbits, _ = O.encode_query(q, W[:-1], 1, N)
    p = O.collision_probability_mips(q, keys - mu, r)
    for i in range(keys.shape[0]):
        freq = float(np.mean(kbits[i] == qbits[0]))
        sigma = math.sqrt(p[i] * (1 - p[i]) / N)
        assert abs(freq - p[i]) < 4.5 * sigma, (i, freq, p[i], sigma)


def test_mips_probability_follows_the_inner_product():
    # a short key along q has the larger cosine, a long key at an angle the larger inner
    # product: the plain probability ranks the short key first, the MIPS variant the long one
    q = np.array([1.0, 0.0, 0.0])
    mu = np.zeros(3)
    keys = np.array([[0.5, 0.05, 0.0], [3.0, 2.0, 0.0], [0.0, 0.0, 1.0]])
    r = O.mips_radius(keys, mu)
    plain = O.collision_probability(q, keys)
    mips = O.collision_probability_mips(q, keys, r)
    assert plain[0] > plain[1] and mips[1] > mips[0]
    order = np.argsort(keys @ q)
    assert np.all(np.diff(mips[order]) > 0)


def test_mips_codes_by_brute_force():
    keys, q, mu = _mips_case(25, n=6, d=3)
    K, L = 2, 3
    rng = np.random.default_rng(26)
    W = rng.standard_normal((4, K * L))
    r = O.mips_radius(keys, mu)
    codes, _, _ = O.encode_keys_mips(keys, mu, W, r, K, L)
    for i, k in enumerate(keys):
        kb = [k[e] - mu[e] for e in range(3)]
        a = math.sqrt(max(0.0, r * r - sum(x * x for x in kb)))
        for t in range(L):
            c = 0
            for b in range(K):
                j = t * K + b
                P = sum(W[e][j] * kb[e] for e in range(3)) + W[3][j] * a
                c |= (1 if P > 0 else 0) << b
            assert codes[i, t] == c


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_mips_near_tie_band_edges(sign):
    # MIPS keys: near iff |P| < 1e-5 |w_j| (|k_i| + r), the raw key's norm plus the radius. Key
    # (delta, 3, 9), centre (0, 0, 5), r = 6: the centred part (delta, 3, 4), the extra coordinate
    # sqrt(11 - delta^2); column 0 of W_aug is 7 e_0, so P = 7 delta
    mu = np.array([0.0, 0.0, 5.0])
    W = np.zeros((4, 2))
    W[0, 0] = 7.0
    W[:, 1] = [0.0, 1.0, 1.0, 1.0]
    r = 6.0
    for c, inside in ((0.999, True), (1.001, False), (0.5, True), (2.0, False)):
        delta = 0.0
        for _ in range(60):
            delta = c * 1e-5 * (math.sqrt(delta * delta + 90.0) + r)
        key = np.array([[sign * delta, 3.0, 9.0]])
        _, bits, near = O.encode_keys_mips(key, mu, W, r, 1, 2)
        assert bool(near[0, 0]) is inside, (c, sign)
        assert bool(bits[0, 0]) is (sign > 0)
        assert not near[0, 1]


def test_mips_importance_weights_are_unbiased_over_hyperplane_draws():
    # Horvitz-Thompson with the variant's inclusion probability: fails if p ignored the radius
    # or the query took the extra row
    rng = np.random.default_rng(27)
    d, n, K, L, M = 6, 40, 2, 6, 20000
    keys = rng.standard_normal((n, d)) * rng.uniform(0.5, 1.5, size=(n, 1))
    vals = rng.standard_normal((n, d))
    q = rng.standard_normal(d)
    mu = O.key_centre(keys)
    r = O.mips_radius(keys, mu)
    s = keys @ q / math.sqrt(d)
    logu = O.log_inclusion_probability(O.collision_probability_mips(q, keys - mu, r), K, L)
    W = rng.standard_normal((d + 1, M * K * L))
    kc = O.encode_keys_mips(keys, mu, W, r, K, M * L)[0].reshape(n, M, L)
    qc = O.encode_query(q, W[:d], K, M * L)[0][0].reshape(M, L)
    T = O.exact_set_mask(n, 0, 0)
    den = np.zeros(M)
    for m in range(M):
        S = O.sampled_set(O.collision_counts(kc[:, m, :], qc[m]), T)
        den[m] = np.exp(s[S] - logu[S]).sum()
    se = den.std(ddof=1) / math.sqrt(M)
    assert abs(den.mean() - np.exp(s).sum()) < 4.5 * se, (den.mean(), np.exp(s).sum(), se)


# ------------------------------------------------------------------------------------------------
# Cross-polytope hashing (named by "LSH Sampling..." conclusion as the hash to shrink the tables):
# code = signed argmax of |G x|, G Gaussian d x d
# ------------------------------------------------------------------------------------------------
def test_cp_probability_closed_forms():
    for d in (8, 128):
        p = O.cp_collision_probability([0.0, 1.0, -1.0], d)
        assert abs(p[0] - 1.0 / (2 * d)) < 1e-10 / d      # independent: same index and sign
        assert p[1] == 1.0 and p[2] == 0.0
    # d = 1: the code is the sign alone, so p is SimHash's 1 - arccos(rho)/pi
    rho = np.array([-0.8, -0.3, 0.0, 0.4, 0.9])
    assert np.allclose(O.cp_collision_probability(rho, 1), 1 - np.arccos(rho) / math.pi,
                       rtol=0, atol=1e-9)
    grid = np.linspace(-0.95, 0.99, 40)
    assert np.all(np.diff(O.cp_collision_probability(grid, 16)) > 0)


@pytest.mark.parametrize("rho", [-0.4, 0.0, 0.3, 0.7, 0.95])
def test_cp_collision_frequency_monte_carlo(rho):
    d, N = 16, 40_000
    rng = np.random.default_rng(int(1000 * rho) + 5000)
    x, y = _pair_at_angle(math.acos(rho), d=d)
    G = rng.standard_normal((N, d, d))
    yx, yy = G @ x, G @ y
    ix, iy = np.argmax(np.abs(yx), axis=1), np.argmax(np.abs(yy), axis=1)
    r = np.arange(N)
    same = (ix == iy) & (np.sign(yx[r, ix]) == np.sign(yy[r, iy]))
    p = float(O.cp_collision_probability([rho], d)[0])
    sigma = math.sqrt(p * (1 - p) / N)
    assert abs(float(np.mean(same)) - p) < 4.5 * sigma + 1e-12, (rho, float(np.mean(same)), p)


def test_cp_codes_by_brute_force():
    rng = np.random.default_rng(31)
    d, L, n = 4, 3, 7
    G = rng.standard_normal((L, d, d))
    keys = rng.standard_normal((n, d))
    mu = O.key_centre(keys)
    codes, _, _ = O.encode_keys_cp(keys, mu, G)
    for i in range(n):
        kb = [keys[i][e] - mu[e] for e in range(d)]
        for t in range(L):
            y = [sum(G[t][j][e] * kb[e] for e in range(d)) for j in range(d)]
            j = max(range(d), key=lambda jj: abs(y[jj]))
            assert codes[i, t] == 2 * j + (1 if y[j] < 0 else 0)
    qc, _, _ = O.encode_query_cp(keys[:2], G)             # the query is hashed as given
    assert np.array_equal(qc[0], O.encode_keys_cp(keys[:1], np.zeros(d), G)[0][0])


def test_cp_code_replay_accepts_only_runner_up_near_ties():
    oc = np.array([[4, 7]])
    alt = np.array([[5, 2]])
    near = np.array([[True, False]])
    out, flips = O.replay_codes(oc, alt, near, np.array([[5, 7]]))
    assert flips == 1 and out.tolist() == [[5, 7]]
    with pytest.raises(AssertionError):
        O.replay_codes(oc, alt, near, np.array([[6, 7]]))     # not the runner-up
    with pytest.raises(AssertionError):
        O.replay_codes(oc, alt, near, np.array([[4, 2]]))     # not a near tie


def _cp_gap_offset(c, rest_norm2):
    """delta with 7 delta = c * 1e-5 * 7 * sqrt((1 + delta)^2 + rest_norm2): the two largest
    |(G x)_i| = 7 (1 + delta) and 7 sit c times the band 1e-5 |g|max |x| apart (G rows 7 e_0,
    7 e_1, e_2, e_3, so |g|max = 7 and x = (1 + delta, 1, ...))."""
    delta = 0.0
    for _ in range(60):
        delta = c * 1e-5 * math.sqrt((1.0 + delta) ** 2 + rest_norm2)
    return delta


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_cp_near_tie_band_edges(sign):
    # cross-polytope: near iff the two largest |G x| differ by less than 1e-5 |g|max |x|; the
    # code is 2 i + [(G x)_i < 0] of the largest, the runner-up code that of the second
    G = np.diag([7.0, 7.0, 1.0, 1.0])
    for c, inside in ((0.999, True), (1.001, False), (0.5, True), (2.0, False)):
        delta = _cp_gap_offset(c, 1.0 + 0.02)
        x = np.array([[sign * (1.0 + delta), 1.0, 0.1, 0.1]])
        code, alt, near = O.cp_hash(x, G)
        assert bool(near[0]) is inside, (c, sign)
        assert code[0] == (0 if sign > 0 else 1) and alt[0] == 2


def test_cp_key_band_uses_the_raw_key_norm():
    # keys are hashed centred, but the band scales with the raw key's norm (as for SimHash):
    # key (1 + delta, 1, 0.1, 5.1) with centre (0, 0, 0, 5) hashes x = (1 + delta, 1, 0.1, 0.1)
    G = np.diag([7.0, 7.0, 1.0, 1.0])[None]
    mu = np.array([0.0, 0.0, 0.0, 5.0])
    for c, inside in ((0.999, True), (1.001, False)):
        delta = _cp_gap_offset(c, 1.0 + 0.01 + 5.1 ** 2)
        key = np.array([[1.0 + delta, 1.0, 0.1, 5.1]])
        code, alt, near = O.encode_keys_cp(key, mu, G)
        assert bool(near[0, 0]) is inside, c
        assert code[0, 0] == 0 and alt[0, 0] == 2


def test_cp_importance_weights_are_unbiased_over_rotation_draws():
    # Horvitz-Thompson with the cross-polytope inclusion probability (one hash per table)
    rng = np.random.default_rng(33)
    d, n, L, M = 6, 30, 5, 8000
    keys = rng.standard_normal((n, d))
    q = rng.standard_normal(d)
    mu = O.key_centre(keys)
    kbar = keys - mu
    cos = (kbar @ q) / (np.linalg.norm(kbar, axis=1) * np.linalg.norm(q))
    logu = O.log_inclusion_probability(O.cp_collision_probability(cos, d), 1, L)
    s = keys @ q / math.sqrt(d)
    T = O.exact_set_mask(n, 0, 0)
    den = np.zeros(M)
    for m in range(M):
        G = rng.standard_normal((L, d, d))
        kc = O.encode_keys_cp(keys, mu, G)[0]
        qc = O.encode_query_cp(q, G)[0][0]
        S = O.sampled_set(O.collision_counts(kc, qc), T)
        den[m] = np.exp(s[S] - logu[S]).sum()
    se = den.std(ddof=1) / math.sqrt(M)
    assert abs(den.mean() - np.exp(s).sum()) < 4.5 * se, (den.mean(), np.exp(s).sum(), se)

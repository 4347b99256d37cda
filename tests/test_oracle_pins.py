"""Pins for the fp64 oracle against what the pages and mathematics fix.

Each test ties one oracle function to something other than itself: values
printed on the pages (tests/golden/), closed forms, exact rational
enumeration, chi-square tests over seeded draws, and finite differences.
"""

import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import spec_oracle as so

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def _rand_dist(rng, V, spiky=1.0):
    z = rng.standard_normal(V) * spiky
    return so.softmax_t(z, 1.0)


# ---------------------------------------------------------------------------
# softmax
# ---------------------------------------------------------------------------

def test_softmax_sums_to_one_and_is_shift_invariant():
    rng = np.random.default_rng(1)
    for V in (1, 2, 7, 1000):
        z = rng.standard_normal(V) * 3
        for T in (0.3, 1.0, 2.5):
            p = so.softmax_t(z, T)
            assert abs(p.sum() - 1.0) < 1e-12
            assert np.all(p >= 0)
            assert np.allclose(so.softmax_t(z + 17.25, T), p, rtol=1e-12, atol=0)


def test_softmax_closed_form_two_tokens():
    # p(0) = 1 / (1 + exp((z1 - z0)/T)) (logistic function)
    for d, T in ((0.0, 1.0), (1.5, 0.7), (-3.0, 2.0)):
        p = so.softmax_t(np.array([0.0, d]), T)
        assert abs(p[0] - 1.0 / (1.0 + math.exp(d / T))) < 1e-15


def test_softmax_rejects_zero_temperature():
    with pytest.raises(ValueError):
        so.softmax_t(np.zeros(3), 0.0)


# ---------------------------------------------------------------------------
# overlap / TV
# ---------------------------------------------------------------------------

def test_overlap_equals_one_minus_tv():
    rng = np.random.default_rng(2)
    for V in (2, 5, 300):
        for _ in range(20):
            p, q = _rand_dist(rng, V, 2.0), _rand_dist(rng, V, 2.0)
            a = so.overlap(p, q)
            assert abs(a - (1.0 - so.tv_distance(p, q))) < 1e-12
            assert 0.0 <= a <= 1.0 + 1e-15
            assert abs(a - so.overlap(q, p)) < 1e-15


def test_overlap_one_iff_equal_and_zero_for_disjoint():
    p = np.array([0.25, 0.25, 0.5, 0.0])
    assert so.overlap(p, p) == pytest.approx(1.0, abs=1e-15)
    assert so.overlap(np.array([1.0, 0.0]), np.array([0.0, 1.0])) == 0.0
    q = np.array([0.25, 0.25, 0.25, 0.25])
    assert so.overlap(p, q) == pytest.approx(0.75, abs=1e-15)


def test_overlap_is_expected_acceptance_exact():
    # alpha_RS = E_{y~q}[min(1, p(y)/q(y))] = sum min(p, q), in exact rationals
    p = np.array([Fraction(1, 2), Fraction(1, 3), Fraction(1, 6), Fraction(0)], dtype=object)
    q = np.array([Fraction(1, 5), Fraction(1, 5), Fraction(1, 5), Fraction(2, 5)], dtype=object)
    e = sum(q[y] * min(Fraction(1), p[y] / q[y]) for y in range(4))
    assert so.overlap(p, q) == e == Fraction(1, 5) + Fraction(1, 5) + Fraction(1, 6)
    assert so.tv_distance(p, q) == 1 - e


def test_residual_decomposition_recovers_target():
    # accepted path min(p,q) plus rejected path (1-alpha) * residual equals p
    rng = np.random.default_rng(3)
    for V in (3, 50, 4000):
        p, q = _rand_dist(rng, V, 1.5), _rand_dist(rng, V, 1.5)
        a = so.overlap(p, q)
        rho = so.residual(p, q)
        assert abs(rho.sum() - (1.0 - a)) < 1e-12
        assert np.allclose(np.minimum(p, q) + (1.0 - a) * rho / rho.sum(), p, rtol=0, atol=1e-15)
    pf = np.array([Fraction(3, 10), Fraction(3, 10), Fraction(2, 5)], dtype=object)
    qf = np.array([Fraction(1, 2), Fraction(1, 4), Fraction(1, 4)], dtype=object)
    rf = so.residual(pf, qf)
    af = so.overlap(pf, qf)
    assert list(np.minimum(pf, qf) + (1 - af) * rf / rf.sum()) == list(pf)


# ---------------------------------------------------------------------------
# inverse CDF
# ---------------------------------------------------------------------------

def test_inverse_cdf_uniform_weights_closed_form():
    # equal weights: index floor(u * V)
    V = 7
    for u in (0.0, 0.01, 0.2, 0.5, 0.86, 0.999):
        v, _ = so.inverse_cdf(np.ones(V), u)
        assert v == math.floor(u * V)


def test_inverse_cdf_skips_zero_weights_and_one_hot():
    w = np.array([0.0, 0.0, 2.0, 0.0, 1.0, 0.0])
    for u in np.linspace(0, 0.999, 50):
        v, _ = so.inverse_cdf(w, u)
        assert w[v] > 0
        assert v == (2 if u < 2.0 / 3.0 else 4)
    assert so.inverse_cdf(np.array([0.0, 5.0, 0.0]), 0.9999)[0] == 1


def test_inverse_cdf_near_flag():
    w = np.array([1.0, 1.0])
    assert so.inverse_cdf(w, 0.5 - 1e-7)[1]
    assert not so.inverse_cdf(w, 0.25)[1]


def _near_case(u0, u1=0.0):
    """Two drafted positions over two tokens, every ratio exact in binary:
    p_k = (1/4, 3/4), q_k = (1/2, 1/2), token 0 drafted at both, so
    p(y)/q(y) = 1/2 exactly (q/p = 2, p(y) = 1/4)."""
    p = [np.array([0.25, 0.75])] * 3
    q = [np.array([0.5, 0.5])] * 2
    return so.accept_and_correct(p, q, [0, 0], [u0, u1], 0.3)


def test_accept_near_flag_threshold_and_operand():
    # the acceptance test (Speculative Decoding 与 MTP, sections 2 and 3)
    # compares u with p(y)/q(y) = 1/2;
    # the oracle flags |u - p/q| < 1e-6 at every evaluated position
    for du in (5e-7, -5e-7):
        _, n, near, _, _ = _near_case(0.5 + du)
        assert near, du
        assert n == (2 if du < 0 else 0)  # u <= p/q accepts (u = 0 accepts the second)
    for du in (5e-6, -5e-6):
        assert not _near_case(0.5 + du)[2], du
    # equality is a near tie and accepts (u <= p/q)
    _, n, near, _, _ = _near_case(0.5, 0.9)
    assert near and n == 1
    # the operand is p/q: u near p(y) = 1/4 or near 1 (q/p = 2 is out of reach) raises no flag
    for u in (0.25, 0.25 + 1e-7, 1.0 - 1e-7):
        assert not _near_case(u)[2], u
    # positions after the first rejection are not evaluated: no flag there
    _, n, near, _, _ = _near_case(0.9, 0.5)
    assert n == 0 and not near
    # an evaluated later position does flag
    _, n, near, _, _ = _near_case(0.1, 0.5 + 2e-7)
    assert n == 1 and near


# ---------------------------------------------------------------------------
# worked examples printed on the pages
# ---------------------------------------------------------------------------

def test_worked_examples_expected_emitted():
    g = json.load(open(GOLDEN))
    for ex in g["expected_emitted"]:
        assert np.allclose(so.prefix_survival(ex["alpha"]), ex["prefix_survival"], atol=1e-12), ex["cite"]
        assert abs(so.expected_emitted(ex["alpha"]) - ex["value"]) < 1e-12, ex["cite"]
        assert abs(so.expected_accepted(ex["alpha"]) - (ex["value"] - 1)) < 1e-12


def test_worked_examples_speedup():
    g = json.load(open(GOLDEN))
    for ex in g["speedup"]:
        s = so.speedup_estimate(ex["alpha"], ex["t_ar"], ex["t_draft"], ex["t_verify"], ex["t_overhead"])
        assert abs(s - ex["value"]) < ex["tol"], ex["cite"]


# ---------------------------------------------------------------------------
# exact rational enumeration of the verify sampler
# ---------------------------------------------------------------------------

def _enumerate_outputs(p, q):
    """Exact output distribution of oracle.accept_and_correct, by evaluating it
    at one representative uniform inside every interval on which its decisions
    are constant, weighted by the interval's length and by prod q_k(y_k)."""
    K = len(q)
    V = len(q[0])
    dist = {}
    for ys in itertools.product(range(V), repeat=K):
        py = Fraction(1)
        for k in range(K):
            py *= q[k][ys[k]]
        if py == 0:
            continue
        # acceptance uniform: accept on [0, r], reject on (r, 1)
        choices = []
        for k in range(K):
            r = p[k][ys[k]] / q[k][ys[k]]
            opts = []
            if r > 0:
                m = min(r, Fraction(1))
                opts.append((m / 2, m))
            if r < 1:
                opts.append(((r + 1) / 2, 1 - r))
            choices.append(opts)
        for combo in itertools.product(*choices):
            us = [c[0] for c in combo]
            wu = Fraction(1)
            for c in combo:
                wu *= c[1]
            # final uniform: midpoints of the 4V intervals between every CDF
            # boundary that any draw could use (fine enough for all of them)
            bounds = set([Fraction(0), Fraction(1)])
            for k in range(K + 1):
                w = p[k] if k == K else so.residual(p[k], q[k])
                tot = w.sum()
                if tot > 0:
                    c = Fraction(0)
                    for x in w:
                        c += x
                        bounds.add(c / tot)
            bl = sorted(bounds)
            for lo, hi in zip(bl[:-1], bl[1:]):
                if hi == lo:
                    continue
                uf = (lo + hi) / 2
                toks, n, *_ = so.accept_and_correct(p, q, list(ys), us, uf)
                key = (tuple(toks), n)
                dist[key] = dist.get(key, Fraction(0)) + py * wu * (hi - lo)
    return dist


def _frac_dist(vals):
    vals = [int(v) for v in vals]
    s = sum(vals)
    return np.array([Fraction(v, s) for v in vals], dtype=object)


@pytest.mark.parametrize("K", [1, 2, 3])
def test_exact_enumeration_matches_target(K):
    V = 3 if K == 3 else 4
    rng = np.random.default_rng(10 + K)
    p = [_frac_dist(list(rng.integers(0, 6, V) + (np.arange(V) == k))) for k in range(K + 1)]
    q = [_frac_dist(list(rng.integers(1, 6, V))) for k in range(K)]
    dist = _enumerate_outputs(p, q)
    assert sum(dist.values()) == 1
    alpha = [so.overlap(p[k], q[k]) for k in range(K)]
    # P(n >= j) = prod_{k<=j} alpha_k exactly (positions independent here)
    for j in range(K + 1):
        pj = sum(w for (toks, n), w in dist.items() if n >= j)
        want = Fraction(1)
        for k in range(j):
            want *= alpha[k]
        assert pj == want
    # the token emitted at position j, given the cycle reaches j, follows p_j
    for j in range(K + 1):
        reach = sum(w for (toks, n), w in dist.items() if n >= j)
        for v in range(V):
            pv = sum(w for (toks, n), w in dist.items() if n >= j and toks[j] == v)
            assert pv == reach * p[j][v]


def test_exact_enumeration_detects_full_p_resample(monkeypatch):
    # planted mistake: resample the correction from the full target p
    p = [_frac_dist([1, 2, 3]), _frac_dist([3, 2, 1])]
    q = [_frac_dist([3, 2, 1])]
    monkeypatch.setattr(so, "residual", lambda pp, qq: pp.copy())
    dist = _enumerate_outputs(p, q)
    p0 = sum(w for (toks, n), w in dist.items() if toks[0] == 2)
    assert p0 != p[0][2]


# ---------------------------------------------------------------------------
# chi-square over 1e6 seeded draws
# ---------------------------------------------------------------------------

N_DRAWS = 1_000_000


def _draws(p, q, n, seed):
    rng = np.random.default_rng(seed)
    K = len(q)
    cq = [np.cumsum(qk) for qk in q]
    ys = np.stack([np.minimum(np.searchsorted(cq[k], rng.random(n), side="right"), len(q[k]) - 1)
                   for k in range(K)], axis=1)
    ua = rng.random((n, K))
    uf = rng.random(n)
    toks = np.full((n, K + 1), -1, dtype=np.int64)
    ns = np.zeros(n, dtype=np.int64)
    for i in range(n):
        t, m, *_ = so.accept_and_correct(p, q, ys[i], ua[i], uf[i])
        toks[i] = t
        ns[i] = m
    return toks, ns


@pytest.fixture(scope="module")
def chi_case():
    rng = np.random.default_rng(42)
    V, K = 4, 2
    p = [_rand_dist(rng, V, 1.0) for _ in range(K + 1)]
    q = [_rand_dist(rng, V, 1.0) for _ in range(K)]
    toks, ns = _draws(p, q, N_DRAWS, seed=2024)
    return p, q, toks, ns


def _chi2_pvalue(counts, probs):
    from scipy.stats import chisquare
    counts = np.asarray(counts, dtype=np.float64)
    exp = np.asarray(probs, dtype=np.float64) * counts.sum()
    keep = exp > 0
    assert counts[~keep].sum() == 0
    return chisquare(counts[keep], exp[keep]).pvalue


@pytest.mark.slow
def test_chi_square_output_distribution(chi_case):
    p, q, toks, ns = chi_case
    K = len(q)
    V = len(p[0])
    alpha = [so.overlap(p[k], q[k]) for k in range(K)]
    # first emitted token ~ p_1
    assert _chi2_pvalue(np.bincount(toks[:, 0], minlength=V), p[0]) > 1e-3
    # emitted token at position j given the cycle reaches j ~ p_j
    for j in range(1, K + 1):
        sel = ns >= j
        assert _chi2_pvalue(np.bincount(toks[sel, j], minlength=V), p[j]) > 1e-3
    # number accepted: P(n = j) = prod_{k<=j} alpha_k * (1 - alpha_{j+1})
    surv = [1.0] + so.prefix_survival(alpha)
    pn = [surv[j] - (surv[j + 1] if j < K else 0.0) for j in range(K + 1)]
    assert _chi2_pvalue(np.bincount(ns, minlength=K + 1), pn) > 1e-3
    # mean emitted length matches 1 + sum prod alpha within 3 sigma
    emitted = ns + 1
    se = emitted.std() / math.sqrt(len(emitted))
    assert abs(emitted.mean() - so.expected_emitted(alpha)) < 3 * se


@pytest.mark.slow
def test_chi_square_rejects_full_p_resample(monkeypatch):
    # planted mistake in the oracle: after a rejection, resample from full p
    rng = np.random.default_rng(7)
    V, K = 4, 1
    p = [_rand_dist(rng, V, 1.5) for _ in range(K + 1)]
    q = [_rand_dist(rng, V, 1.5) for _ in range(K)]
    monkeypatch.setattr(so, "residual", lambda pp, qq: pp.copy())
    toks, ns = _draws(p, q, 200_000, seed=5)
    assert _chi2_pvalue(np.bincount(toks[:, 0], minlength=V), p[0]) < 1e-6


# ---------------------------------------------------------------------------
# greedy
# ---------------------------------------------------------------------------

def test_greedy_equals_argmax_and_first_mismatch():
    rng = np.random.default_rng(4)
    K, V = 4, 50
    zt = rng.standard_normal((1, K + 1, V))
    am = zt[0].argmax(axis=1)
    draft = am[:K].copy()
    draft[2] = (am[2] + 1) % V
    r = oracle.verify(zt, None, draft[None], np.zeros((1, K)), np.zeros(1), 0.0)
    assert r.n_accepted[0] == 2
    assert list(r.tokens[0]) == [am[0], am[1], am[2], -1, -1]
    r2 = oracle.verify(zt, None, am[None, :K], np.zeros((1, K)), np.zeros(1), 0.0)
    assert r2.n_accepted[0] == K and list(r2.tokens[0]) == list(am)


def test_greedy_ties_take_smallest_index():
    z = np.array([[[1.0, 3.0, 3.0, 0.0], [2.0, 2.0, 1.0, 2.0]]])
    r = oracle.verify(z, None, np.array([[2]]), np.zeros((1, 1)), np.zeros(1), 0.0)
    assert list(r.tokens[0]) == [1, -1] and r.n_accepted[0] == 0
    r = oracle.verify(z, None, np.array([[1]]), np.zeros((1, 1)), np.zeros(1), 0.0)
    assert list(r.tokens[0]) == [1, 0]


def test_greedy_is_zero_temperature_limit():
    rng = np.random.default_rng(5)
    B, K, V = 20, 3, 12
    # well separated logits: at T=0.01 every distribution is one-hot to 1e-40
    zt = np.stack([np.stack([rng.permutation(V).astype(np.float64) for _ in range(K + 1)])
                   for _ in range(B)])
    zd = np.where(rng.random((B, K, 1)) < 0.5, zt[:, :K], zt[:, :K][:, :, ::-1])
    draft = zd.argmax(axis=2)
    ua = rng.random((B, K)).astype(np.float32)
    uf = rng.random(B).astype(np.float32)
    g = oracle.verify(zt, zd, draft, ua, uf, 0.0)
    s = oracle.verify(zt, zd, draft, ua, uf, 0.01)
    assert (g.tokens == s.tokens).all() and (g.n_accepted == s.n_accepted).all()
    assert np.allclose(g.alpha, s.alpha, atol=1e-12)


def test_identical_logits_accept_everything():
    rng = np.random.default_rng(6)
    B, K, V = 8, 5, 30
    zt = rng.standard_normal((B, K + 1, V)) * 2
    zd = zt[:, :K].copy()
    draft = rng.integers(0, V, (B, K))
    ua = rng.random((B, K)).astype(np.float32)
    uf = rng.random(B).astype(np.float32)
    r = oracle.verify(zt, zd, draft, ua, uf, 0.8)
    assert (r.n_accepted == K).all()
    assert (r.tokens[:, :K] == draft).all()
    assert np.allclose(r.alpha, 1.0, atol=1e-12)
    # the bonus follows p_{K+1}'s inverse CDF at u'
    for b in range(B):
        v, _ = so.inverse_cdf(so.softmax_t(zt[b, K], 0.8), float(uf[b]))
        assert r.tokens[b, K] == v


def test_zero_draft_probability_always_accepts():
    p = [np.array([0.5, 0.5]), np.array([1.0, 0.0])]
    q = [np.array([1.0, 0.0])]
    toks, n, *_ = so.accept_and_correct(p, q, [1], [0.999], 0.3)
    assert n == 1 and toks[0] == 1


def test_K_zero_is_plain_sampling():
    z = np.log(np.array([[[0.1, 0.2, 0.7]]]))
    # CDF of p = (0.1, 0.3, 1.0): u' = 0.25 -> index 1, u' = 0.35 -> index 2
    for uf, want in ((0.05, 0), (0.25, 1), (0.35, 2)):
        r = oracle.verify(z, np.zeros((1, 0, 3)), np.zeros((1, 0), dtype=np.int64),
                          np.zeros((1, 0)), np.array([uf]), 1.0)
        assert r.n_accepted[0] == 0 and list(r.tokens[0]) == [want]


# ---------------------------------------------------------------------------
# overlap statistics
# ---------------------------------------------------------------------------

def test_overlap_stats_prefix_products():
    rng = np.random.default_rng(8)
    zt = rng.standard_normal((3, 4, 20))
    zd = zt + rng.standard_normal((3, 4, 20)) * 0.5
    o = oracle.overlap_stats(zt, zd, 1.0)
    assert np.allclose(o.alpha, 1 - o.tv, atol=1e-12)
    assert np.allclose(o.prefix_survival, np.cumprod(o.alpha, axis=1), atol=1e-15)
    assert np.allclose(o.expected_accepted, o.prefix_survival.sum(axis=1), atol=1e-15)


# ---------------------------------------------------------------------------
# E2E-TV loss and gradient
# ---------------------------------------------------------------------------

def test_e2e_loss_single_position_is_alpha():
    rng = np.random.default_rng(9)
    zt = rng.standard_normal((5, 1, 40))
    zd = rng.standard_normal((5, 1, 40))
    L, a = oracle.e2e_tv_loss(zt, zd, 1.3)
    assert abs(L - a[:, 0].mean()) < 1e-15
    for b in range(5):
        p, q = so.softmax_t(zt[b, 0], 1.3), so.softmax_t(zd[b, 0], 1.3)
        assert abs(a[b, 0] - (1 - so.tv_distance(p, q))) < 1e-12


def test_e2e_loss_worked_example_structure():
    # with constant alpha the loss is sum_j alpha^j (page's prefix-product form)
    zt = np.zeros((2, 4, 6))
    zd = np.zeros((2, 4, 6))
    L, a = oracle.e2e_tv_loss(zt, zd, 1.0)
    assert np.allclose(a, 1.0) and abs(L - 4.0) < 1e-12


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_e2e_grad_matches_finite_differences(T):
    rng = np.random.default_rng(11)
    B, K, V = 2, 3, 6
    zt = rng.standard_normal((B, K, V)) * 1.5
    zd = zt + rng.standard_normal((B, K, V)) * 0.8
    g, amb = oracle.e2e_tv_grad(zt, zd, T, grad_scale=-1.0)
    assert not amb.any()
    h = 1e-6
    num = np.zeros_like(zd)
    for idx in np.ndindex(*zd.shape):
        zp = zd.copy()
        zp[idx] += h
        zm = zd.copy()
        zm[idx] -= h
        num[idx] = -(oracle.e2e_tv_loss(zt, zp, T)[0] - oracle.e2e_tv_loss(zt, zm, T)[0]) / (2 * h)
    assert np.allclose(g, num, rtol=1e-6, atol=1e-9)


def test_e2e_grad_rows_sum_to_zero_and_subset():
    rng = np.random.default_rng(12)
    zt = rng.standard_normal((3, 4, 50))
    zd = zt + rng.standard_normal((3, 4, 50)) * 0.3
    g, _ = oracle.e2e_tv_grad(zt, zd, 0.9)
    assert np.allclose(g.sum(axis=2), 0.0, atol=1e-15)
    g1, _ = oracle.e2e_tv_grad(zt, zd, 0.9, rows=[2])
    assert np.array_equal(g1[0], g[2])


def test_inverse_cdf_strict_boundary_reading():
    # reading: the chosen index is the first whose running sum is strictly
    # above u * total, so u landing exactly on a boundary moves to the next
    # token (u in [0, 1) never selects past the last positive weight)
    assert so.inverse_cdf(np.array([1.0, 1.0]), 0.5)[0] == 1
    assert so.inverse_cdf(np.array([1.0, 1.0]), 0.0)[0] == 0
    assert so.inverse_cdf(np.array([0.0, 1.0, 1.0]), 0.0)[0] == 1


# ---------------------------------------------------------------------------
# entropy, cross-entropy, KL and target-only acceptance
# ---------------------------------------------------------------------------

def test_entropy_closed_forms():
    # uniform over V tokens: ln V; a point mass: 0
    for V in (1, 2, 7, 1024):
        assert abs(so.entropy(np.full(V, 1.0 / V)) - math.log(V)) < 1e-12
    assert so.entropy(np.array([0.0, 1.0, 0.0])) == 0.0
    # infinite temperature flattens any logits to the uniform distribution
    z = np.random.default_rng(3).normal(size=50) * 3
    assert abs(so.entropy(so.softmax_t(z, 1e9)) - math.log(50)) < 1e-6


def test_two_token_worked_example():
    # p = (1/2, 1/2), q = (1/4, 3/4), worked by hand:
    #   H = ln 2 = 0.6931471805599453
    #   KL = 1/2 ln 2 + 1/2 ln(2/3) = 1/2 ln(4/3) = 0.14384103622589045
    #   CE = -1/2 ln(1/4) - 1/2 ln(3/4) = 0.8369882167858358
    #   alpha_TO = p(argmax q) = p(1) = 1/2
    p, q = np.array([0.5, 0.5]), np.array([0.25, 0.75])
    assert abs(so.entropy(p) - 0.6931471805599453) < 1e-15
    assert abs(so.kl_divergence(p, q) - 0.14384103622589045) < 1e-15
    assert abs(so.cross_entropy(p, q) - 0.8369882167858358) < 1e-15
    assert so.alpha_target_only(p, q) == 0.5


def test_entropy_and_kl_match_scipy():
    from scipy.stats import entropy as sp_entropy
    rng = np.random.default_rng(5)
    for _ in range(20):
        V = int(rng.integers(2, 300))
        p = so.softmax_t(rng.normal(size=V) * 2, 1.0)
        q = so.softmax_t(rng.normal(size=V) * 2, 0.7)
        assert abs(so.entropy(p) - sp_entropy(p)) < 1e-12
        assert abs(so.kl_divergence(p, q) - sp_entropy(p, q)) < 1e-12


def test_cross_entropy_is_entropy_plus_kl_and_inequalities():
    rng = np.random.default_rng(6)
    for _ in range(50):
        V = int(rng.integers(2, 200))
        p = so.softmax_t(rng.normal(size=V) * 3, 1.0)
        q = so.softmax_t(rng.normal(size=V) * 3, 1.0)
        h, ce, kl = so.entropy(p), so.cross_entropy(p, q), so.kl_divergence(p, q)
        assert abs(ce - (h + kl)) < 1e-10
        assert kl >= 0.0 and 0.0 <= h <= math.log(V) + 1e-12
        # Pinsker: d_TV <= sqrt(KL / 2)
        assert so.tv_distance(p, q) <= math.sqrt(kl / 2) + 1e-12
        assert abs(so.kl_divergence(p, p)) < 1e-15


def test_point_mass_drafter_acceptance_is_target_only():
    # a greedy drafter is a point mass at y_hat: the rejection-sampling
    # acceptance sum min(p, q) then equals the target-only p(y_hat)
    rng = np.random.default_rng(7)
    p = so.softmax_t(rng.normal(size=40) * 2, 1.0)
    for y in (0, 13, 39):
        q = np.zeros(40)
        q[y] = 1.0
        assert so.overlap(p, q) == so.alpha_target_only(p, q) == p[y]


def test_diagnostics_shift_invariant_and_batched():
    rng = np.random.default_rng(8)
    zt = rng.normal(size=(2, 3, 64)) * 2
    zd = zt + rng.normal(size=(2, 3, 64)) * 0.5
    a = so.diagnostics(zt, zd, 0.8)
    b = so.diagnostics(zt + 7.0, zd - 3.0, 0.8)
    for f in ("alpha", "entropy", "cross_entropy", "kl", "alpha_to"):
        np.testing.assert_allclose(getattr(a, f), getattr(b, f), rtol=0, atol=1e-12)
    p = so.softmax_t(zt[1, 2], 0.8)
    q = so.softmax_t(zd[1, 2], 0.8)
    assert a.alpha_to[1, 2] == p[np.argmax(q)]
    np.testing.assert_allclose(a.cross_entropy, a.entropy + a.kl, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# top-k / top-p truncation
# ---------------------------------------------------------------------------

def _kept(z_out):
    return [int(v) for v in np.nonzero(np.isfinite(z_out))[0]]


def test_truncation_worked_example():
    # z = (2, 1, 0, 1) at T = 1: p = (e^2, e, 1, e) / (e^2 + 2e + 1)
    #   = (0.534447, 0.196612, 0.072329, 0.196612); ranking 0, 1, 3, 2
    #   (tokens 1 and 3 tie: smaller index first); preceding masses in that
    #   order 0, 0.534447, 0.731059, 0.927671.
    z = np.array([2.0, 1.0, 0.0, 1.0])
    cases = [
        (2, 1.0, 1.0, [0, 1]),     # top-k: the tie at 1 keeps the smaller index
        (0, 0.6, 1.0, [0, 1]),     # 0.534 < 0.6 <= 0.731
        (0, 0.5, 1.0, [0]),        # 0.534 >= 0.5
        (0, 0.8, 1.0, [0, 1, 3]),  # 0.731 < 0.8 <= 0.928
        (3, 0.9, 1.0, [0, 1, 3]),  # top-3 renormalised: preceding 0, 0.576, 0.788
        (1, 1.0, 1.0, [0]),
        # T = 0.5: p = (e^4, e^2, 1, e^2) / (e^4 + 2e^2 + 1) = (0.7758, 0.1050, 0.0142, 0.1050)
        (0, 0.8, 0.5, [0, 1]),     # 0.776 < 0.8 <= 0.881
    ]
    for k, tp, T, want in cases:
        out, near = so.truncate_logits(z, T, k, tp)
        assert _kept(out) == want, (k, tp, T)
        assert not near
        assert (out[want] == z[want]).all() and np.isneginf(np.delete(out, want)).all()
    # a cut exactly at a preceding mass is a near tie, and the token is dropped
    p0 = math.exp(2) / (math.exp(2) + 2 * math.e + 1)
    out, near = so.truncate_logits(z, 1.0, 0, p0)
    assert near and _kept(out) in ([0], [0, 1])


def test_truncation_masked_logits():
    # z = (1, -inf, 0, -inf, 2) at T = 1: masked tokens have p = 0, so
    # p = (e, 0, 1, 0, e^2) / (e^2 + e + 1) = (0.244728, 0, 0.090031, 0, 0.665241);
    # ranking 4, 0, 2, then the masked tokens 1, 3 by index; preceding masses
    # along it 0, 0.665241, 0.909969, 1, 1.
    z = np.array([1.0, -np.inf, 0.0, -np.inf, 2.0])
    cases = [
        (2, 1.0, [0, 4]),
        (0, 0.5, [4]),          # 0.665 >= 0.5
        (0, 0.7, [0, 4]),       # 0.665 < 0.7 <= 0.910
        (0, 0.95, [0, 2, 4]),   # 0.910 < 0.95; the masked tokens add no mass
        (4, 0.95, [0, 2, 4]),   # top-4 takes masked token 1 too; it stays -inf
    ]
    for k, tp, want in cases:
        out, near = so.truncate_logits(z, 1.0, k, tp)
        assert _kept(out) == want, (k, tp)
        assert not near
        assert (out[want] == z[want]).all() and np.isneginf(np.delete(out, want)).all()


def test_truncation_closed_forms():
    z = np.zeros(10)  # uniform: the preceding mass of rank i is i / 10
    for tp, n in ((0.35, 4), (0.05, 1), (0.5, 5), (0.95, 10)):
        out, _ = so.truncate_logits(z, 1.3, 0, tp)
        assert _kept(out) == list(range(n))  # ties rank by index
    out, _ = so.truncate_logits(z, 1.0, 3, 1.0)
    assert _kept(out) == [0, 1, 2]
    rng = np.random.default_rng(11)
    z = rng.normal(size=50) * 2
    assert _kept(so.truncate_logits(z, 1.0, 1, 1.0)[0]) == [so.argmax_first(z)]
    assert _kept(so.truncate_logits(z, 1.0, 0, 1e-9)[0]) == [so.argmax_first(z)]
    for k in (0, 50, 80):
        out, _ = so.truncate_logits(z, 0.7, k, 1.0)
        assert (out == z).all()


def test_truncation_brute_force_tiny():
    """The kept set is the smallest subset of the top-k set whose
    renormalised mass reaches top_p, with the largest mass among subsets of
    that size (unique here: no equal masses)."""
    rng = np.random.default_rng(12)
    for trial in range(300):
        V = int(rng.integers(1, 7))
        z = rng.normal(size=V) * 1.5
        T = float(rng.choice([0.5, 1.0, 2.0]))
        k = int(rng.integers(0, V + 2))
        tp = float(rng.uniform(0.05, 1.0))
        out, near = so.truncate_logits(z, T, k, tp)
        if near:
            continue
        kept = set(_kept(out))
        cand = list(range(V)) if not (0 < k < V) else sorted(np.argsort(-z, kind="stable")[:k].tolist())
        p = so.softmax_t(z[cand], T)
        mass = dict(zip(cand, p))
        best = None
        for size in range(1, len(cand) + 1):
            sets = [s for s in itertools.combinations(cand, size) if sum(mass[v] for v in s) >= tp]
            if sets:
                best = max(sets, key=lambda s: sum(mass[v] for v in s))
                break
        if tp >= 1.0:
            best = tuple(cand)
        assert kept == set(best), (trial, z, T, k, tp)


def test_truncation_invariants_random_rows():
    rng = np.random.default_rng(13)
    for trial in range(40):
        V = 500
        z = np.round(rng.normal(size=V) * 3, 1)  # rounded: many ties
        T = float(rng.uniform(0.3, 2.0))
        k = int(rng.integers(0, 600))
        tp = float(rng.uniform(0.1, 1.0))
        out, near = so.truncate_logits(z, T, k, tp)
        kept = np.isfinite(out)
        n = int(kept.sum())
        assert n >= 1 and (n <= k or not 0 < k < V)
        # upward closed in the ranking (logit descending, index ascending)
        rank = sorted(range(V), key=lambda v: (-z[v], v))
        flags = [bool(kept[v]) for v in rank]
        assert flags == sorted(flags, reverse=True)
        if tp < 1.0 and not near:
            top = rank[: (k if 0 < k < V else V)]
            p = so.softmax_t(z[top], T)
            m = dict(zip(top, p))
            ranked_kept = [v for v in rank if kept[v]]
            assert sum(m[v] for v in ranked_kept) >= tp
            assert sum(m[v] for v in ranked_kept[:-1]) < tp


# ---------------------------------------------------------------------------
# verify-length scheduling
# ---------------------------------------------------------------------------

def test_schedule_hand_example():
    # R = 2, L = 2, a = [[0.9, 0.5], [0.6, 0.1]], SPS(2..6) = 100, 95, 80, 78, 60.
    # Taking the largest survivals first: B = 2 -> 2 * 100 = 200; B = 3 -> 2.9 * 95 = 275.5;
    # B = 4 -> 3.5 * 80 = 280; B = 5 -> 4.0 * 78 = 312; B = 6 -> 4.1 * 60 = 246.
    r = so.schedule_lengths([[0.9, 0.5], [0.6, 0.1]], [0, 0, 100, 95, 80, 78, 60])
    assert r.lengths.tolist() == [2, 1]
    assert r.theta == pytest.approx(312.0, rel=1e-15) and r.tau == pytest.approx(4.0) and r.batch == 5
    assert not r.near


def test_schedule_tie_rules():
    # Equal survivals are taken in (row, position) order: R = 2, L = 1,
    # a = [[0.5], [0.5]], SPS(2..4) = 1, 1, 0.5: B = 2 -> 2, B = 3 -> 2.5,
    # B = 4 -> 1.5, so one survival is taken, and it is row 0's.
    r = so.schedule_lengths([[0.5], [0.5]], [0, 0, 1.0, 1.0, 0.5])
    assert r.lengths.tolist() == [1, 0] and r.batch == 3 and r.theta == 2.5
    # Equal throughputs keep the smaller batch: SPS(2..4) = 1.25, 1, 0.5 gives
    # B = 2 -> 2.5 and B = 3 -> 2.5 exactly (binary fractions), so B = 2.
    r = so.schedule_lengths([[0.5], [0.5]], [0, 0, 1.25, 1.0, 0.5])
    assert r.lengths.tolist() == [0, 0] and r.batch == 2 and r.theta == 2.5
    assert r.near  # another B reaches the same throughput


def _survivals(rng, R, L):
    c = rng.uniform(0.3, 1.0, size=(R, L))
    return np.cumprod(c, axis=1)


def _step_sps(rng, n):
    # a decreasing throughput curve with cliffs at random batch sizes
    base = 1000.0 / (1.0 + np.arange(n) / rng.uniform(2.0, 8.0))
    cliffs = rng.choice(np.arange(1, n), size=min(3, n - 1), replace=False)
    for c in cliffs:
        base[c:] *= rng.uniform(0.6, 0.95)
    return base


def test_schedule_brute_force_tiny():
    rng = np.random.default_rng(21)
    for trial in range(200):
        R = int(rng.integers(1, 4))
        L = int(rng.integers(1, 4))
        a = _survivals(rng, R, L)
        sps = _step_sps(rng, R * (1 + L) + 1)
        r = so.schedule_lengths(a, sps)
        best, best_b = -1.0, None
        for ls in itertools.product(range(L + 1), repeat=R):
            B = sum(1 + l for l in ls)
            tau = sum(1 + a[i, :l].sum() for i, l in enumerate(ls))
            th = tau * sps[B]
            if th > best * (1 + 1e-12):
                best, best_b = th, B
            elif abs(th - best) <= 1e-12 * best and B < best_b:
                best_b = B
        assert r.theta == pytest.approx(best, rel=1e-12)
        ls = r.lengths
        B = int(sum(1 + l for l in ls))
        tau = sum(1 + a[i, :l].sum() for i, l in enumerate(ls))
        assert B == r.batch and tau * sps[B] == pytest.approx(best, rel=1e-12)
        if not r.near:
            assert B == best_b


def test_schedule_closed_forms():
    rng = np.random.default_rng(22)
    a = _survivals(rng, 5, 4)
    flat = np.full(5 * 5 + 1, 7.0)  # constant SPS: every positive survival pays
    r = so.schedule_lengths(a, flat)
    assert r.lengths.tolist() == [4] * 5 and r.batch == 25
    assert r.tau == pytest.approx(5 + a.sum())
    cliff = np.zeros(26)
    cliff[: 5 + 1] = 10.0  # nothing beyond one token per request runs
    r = so.schedule_lengths(a, cliff)
    assert r.lengths.tolist() == [0] * 5 and r.batch == 5 and r.theta == 50.0
    # non-monotone input: the running minimum is what counts
    r1 = so.schedule_lengths([[0.5, 0.9]], [0, 10, 9, 8])
    r2 = so.schedule_lengths([[0.5, 0.5]], [0, 10, 9, 8])
    assert r1.lengths.tolist() == r2.lengths.tolist() and r1.theta == r2.theta


# ---------------------------------------------------------------------------
# relaxed (lossy) acceptance
# ---------------------------------------------------------------------------

def test_relaxed_accept_hand_example():
    # z = (2, 1, 0, 1), T = 1, y = 3: two logits rank above or tie before it
    # (2, and the tied 1 at index 1), so its rank is 2; log p(3) - log p_max = -1.
    z = [2.0, 1.0, 0.0, 1.0]
    inf = float("inf")
    assert so.relaxed_accept(z, 3, 1.0, 2, inf) == (False, False)
    assert so.relaxed_accept(z, 3, 1.0, 3, inf) == (True, False)
    assert so.relaxed_accept(z, 3, 1.0, 0, 0.5) == (False, False)
    assert so.relaxed_accept(z, 3, 1.0, 0, 1.5) == (True, False)
    assert so.relaxed_accept(z, 3, 2.0, 0, 0.6) == (True, False)  # gap -1/2 at T = 2
    acc, near = so.relaxed_accept(z, 3, 1.0, 0, 1.0)  # gap exactly -delta
    assert acc and near
    assert so.relaxed_accept(z, 1, 1.0, 2, inf) == (True, False)  # the tie at index 1 ranks first
    assert so.relaxed_accept(z, 7, 1.0, 0, inf)[0] is False        # a token outside the vocabulary


def test_relaxed_limits():
    rng = np.random.default_rng(31)
    B, K, V = 6, 4, 40
    zt = rng.normal(size=(B, K + 1, V)) * 2
    y = rng.integers(0, V, size=(B, K))
    uf = rng.uniform(size=B)
    r = so.verify_relaxed(zt, None, y, uf, 1.0, 0, float("inf"))  # no condition: everything accepted
    assert (r.n_accepted == K).all()
    for b in range(B):
        assert r.tokens[b, :K].tolist() == y[b].tolist()
        assert r.tokens[b, K] == so.inverse_cdf(so.softmax_t(zt[b, K], 1.0), uf[b])[0]
    r = so.verify_relaxed(zt, None, y, uf, 1.0, 1, float("inf"))  # top-1: the greedy test
    for b in range(B):
        n = next((k for k in range(K) if y[b, k] != so.argmax_first(zt[b, k])), K)
        assert r.n_accepted[b] == n


def test_relaxed_is_lossy_exact_enumeration():
    """With the draft drawn from q, the first emitted token of the exact
    verify has distribution p; the relaxed rule does not."""
    z = np.array([1.0, 0.8, -1.0])
    p = so.softmax_t(z, 1.0)
    q = np.array([0.05, 0.9, 0.05])
    # relaxed, top-2: a rejected draft (token 2) emits a draw from p
    dist = np.zeros(3)
    for y in range(3):
        if so.relaxed_accept(z, y, 1.0, 2, float("inf"))[0]:
            dist[y] += q[y]
        else:
            dist += q[y] * p
    assert abs(dist.sum() - 1.0) < 1e-12
    assert np.max(np.abs(dist - p)) > 0.2
    # the exact rule on the same pair: accepted mass min(p, q), residual the rest
    exact = np.minimum(p, q) + (1 - so.overlap(p, q)) * so.residual(p, q) / so.residual(p, q).sum()
    np.testing.assert_allclose(exact, p, atol=1e-12)


# ---------------------------------------------------------------------------
# candidate trees
# ---------------------------------------------------------------------------

def test_tree_mask_closed_forms_and_brute_force():
    M, depth = so.tree_mask([-1, 0, 1, 2])  # a chain: lower-triangular, depth = index
    assert (M == np.tril(np.ones((4, 4), dtype=bool))).all() and depth.tolist() == [0, 1, 2, 3]
    M, depth = so.tree_mask([-1, -1, -1])   # siblings on the prefix: each sees itself
    assert (M == np.eye(3, dtype=bool)).all() and depth.tolist() == [0, 0, 0]
    # the example tree of two branches: 0 -> {1, 2}, 1 -> {3}, 2 -> {4, 5}
    M, depth = so.tree_mask([-1, 0, 0, 1, 2, 2])
    assert M[3].nonzero()[0].tolist() == [0, 1, 3] and M[5].nonzero()[0].tolist() == [0, 2, 5]
    assert not M[4, 5] and not M[3, 2] and depth.tolist() == [0, 1, 1, 2, 2, 2]
    rng = np.random.default_rng(41)
    for _ in range(50):
        N = int(rng.integers(1, 12))
        par = [-1] + [int(rng.integers(-1, i)) for i in range(1, N)]
        M, depth = so.tree_mask(par)
        for u in range(N):
            anc = set()
            v = par[u]
            while v >= 0:
                anc.add(v)
                v = par[v]
            assert set(M[u].nonzero()[0].tolist()) == anc | {u}
            assert depth[u] == len(anc)


def test_tree_greedy_chain_is_the_linear_greedy_verify():
    rng = np.random.default_rng(42)
    B, K, V = 8, 5, 30
    zt = rng.normal(size=(B, K + 1, V))
    zt = np.round(zt * 2) / 2  # ties
    y = np.array([[so.argmax_first(zt[b, k]) if rng.uniform() < 0.7 else int(rng.integers(0, V))
                   for k in range(K)] for b in range(B)])
    lin = so.verify(zt, None, y, np.zeros((B, K)), np.zeros(B), 0.0)
    tr = so.tree_verify_greedy(zt, np.tile(np.arange(-1, K - 1), (B, 1)), y)
    assert tr.n_accepted.tolist() == lin.n_accepted.tolist()
    assert tr.tokens.tolist() == lin.tokens.tolist()
    for b in range(B):
        assert tr.path[b, : tr.n_accepted[b]].tolist() == list(range(tr.n_accepted[b]))


def test_tree_greedy_branches_by_hand():
    # two branches on the prefix: node 0 (token 3) and node 1 (token 5); node 1 has a child,
    # node 2 (token 7).  The prefix slot's argmax is 5, node 1's slot argmax is 7, node 2's is 9.
    V = 10
    zt = np.zeros((1, 4, V))
    zt[0, 0, 5] = 2.0   # after the prefix
    zt[0, 1, 0] = 2.0   # after node 0 (not taken)
    zt[0, 2, 7] = 2.0   # after node 1
    zt[0, 3, 9] = 2.0   # after node 2
    r = so.tree_verify_greedy(zt, [[-1, -1, 1]], [[3, 5, 7]])
    assert r.path.tolist() == [[1, 2, -1]] and r.n_accepted.tolist() == [2]
    assert r.tokens.tolist() == [[5, 7, 9, -1]]
    # duplicate sibling tokens: the first in node order is taken
    r = so.tree_verify_greedy(zt, [[-1, -1, 0]], [[5, 5, 7]])
    assert r.path[0, 0] == 0 and r.n_accepted[0] == 1 and r.tokens[0].tolist() == [5, 0, -1, -1]

"""Pins for the CPU oracle: each checks it against something other than
itself (published values, closed forms, exact enumeration over the 2^-24
lattice of uniforms, statistics, limits and special cases).

Each pin is written as a function returning an error so the mutation tests at
the bottom can plant a plausible mistake in the oracle and show the pin
catches it.
"""
import itertools
import json
import math
from pathlib import Path

import numpy as np
import pytest
from scipy import stats

from oracle import spec_oracle as O

GOLDEN = Path(__file__).parent / "golden"
L = 1 << 24
LSB = 2.0 ** -24


# ---------------------------------------------------------------- helpers
def lattice_accept_fraction(a):
    """Fraction of the 2^24 lattice uniforms the oracle's coin accepts at
    acceptance probability a (the predicate is monotone in u: bisect it)."""
    lo, hi = 0, L
    while lo < hi:
        mid = (lo + hi) // 2
        if O.coin_accepts(mid * LSB, a):
            lo = mid + 1
        else:
            hi = mid
    return lo / L


def lattice_law(draw, V):
    """Exact law over tokens of a draw u -> token that is non-decreasing in u,
    counted over the 2^24 lattice by bisecting the first u reaching each
    token."""
    firsts = []
    for y in range(V + 1):
        lo, hi = 0, L
        while lo < hi:
            mid = (lo + hi) // 2
            if draw(mid * LSB) >= y:
                hi = mid
            else:
                lo = mid + 1
        firsts.append(lo)
    law = np.diff(np.asarray(firsts)) / L
    # spot-check that the draw really is the step function the bisection saw
    rng = np.random.default_rng(7)
    for k in rng.integers(0, L, 64):
        y = draw(k * LSB)
        assert firsts[y] <= k < firsts[y + 1]
    return law


def rand_pair(rng, V, scale=1.5):
    zp = scale * rng.normal(size=V)
    zq = zp + scale * rng.normal(size=V)
    return O.softmax_T(zp, 1.0), O.softmax_T(zq, 1.0)


def exact_first_token_law(p, q):
    """Law of the first emitted token for K=1: draft x ~ q, accepted with the
    oracle's coin, otherwise the oracle's correction draw."""
    V = p.size
    A = np.array([lattice_accept_fraction(O.acceptance_prob(p[x], q[x]))
                  for x in range(V)])
    acc_mass = float(np.sum(q * A))
    R = lattice_law(lambda u: O.sample_residual_or_p(p, q, u)[0], V)
    return q * A + (1.0 - acc_mass) * R, acc_mass


def lossless_error(seed=0, trials=6, V=12):
    rng = np.random.default_rng(seed)
    worst = 0.0
    for _ in range(trials):
        p, q = rand_pair(rng, V)
        law, _ = exact_first_token_law(p, q)
        worst = max(worst, float(np.max(np.abs(law - p))))
    return worst


def acceptance_mass_error(seed=1, trials=6, V=12):
    rng = np.random.default_rng(seed)
    worst = 0.0
    for _ in range(trials):
        p, q = rand_pair(rng, V)
        _, acc = exact_first_token_law(p, q)
        worst = max(worst, abs(acc - float(np.sum(np.minimum(p, q)))))
    return worst


def iid_batch(rng, N, K, V, p, q):
    """N requests with the same target law p at all K+1 positions and draft
    law q at all K positions, drafts drawn from q."""
    zp, zq = np.log(p), np.log(q)
    target = np.tile(zp[None], (N * (K + 1), 1))
    draft = np.tile(zq[None], (N * K, 1))
    toks = rng.choice(V, size=N * K, p=q)
    cu = np.arange(0, N * K + 1, K)
    return target, draft, toks, cu


def accepted_length_zscore(seed=3, N=100_000, K=4, V=10):
    rng = np.random.default_rng(seed)
    p, q = rand_pair(rng, V, scale=1.0)
    target, draft, toks, cu = iid_batch(rng, N, K, V, p, q)
    out = O.verify_linear(target, draft, toks, cu, np.ones(N), seed=99 + seed)
    alpha = float(np.sum(np.minimum(p, q)))
    # P(n = k) = alpha^k (1 - alpha) for k < K, alpha^K for k = K
    pk = np.array([alpha ** k * (1 - alpha) for k in range(K)] + [alpha ** K])
    ks = np.arange(K + 1)
    mean = float(np.sum(ks * pk))
    assert abs(mean - alpha * (1 - alpha ** K) / (1 - alpha)) < 1e-12
    sd = math.sqrt(float(np.sum((ks - mean) ** 2 * pk)))
    return (float(np.mean(out["accepted"])) - mean) / (sd / math.sqrt(N))


def chi2_first_token_pvalue(seed=5, N=1_000_000, V=8):
    rng = np.random.default_rng(seed)
    p, q = rand_pair(rng, V, scale=1.0)
    p2, _ = rand_pair(rng, V, scale=1.0)
    zp, zp2, zq = np.log(p), np.log(p2), np.log(q)
    target = np.empty((2 * N, V))
    target[0::2], target[1::2] = zp, zp2
    draft = np.tile(zq[None], (N, 1))
    toks = rng.choice(V, size=N, p=q)
    out = O.verify_linear(target, draft, toks, np.arange(N + 1), np.ones(N),
                          seed=1000 + seed)
    counts = np.bincount(out["tokens"][:, 0], minlength=V)
    return stats.chisquare(counts, N * p).pvalue


# ------------------------------------------------------------- the hash
def test_splitmix64_matches_published_sequence():
    data = json.loads((GOLDEN / "splitmix64_seed0.json").read_text())
    state = 0
    for want in data["outputs"]:
        assert O.splitmix64(state) == int(want, 16)
        state = (state + O.GOLDEN_GAMMA) & O.MASK64


def test_uniform_lattice_and_uniformity():
    us = np.array([O.uniform(0xABCDEF, b, pos, s)
                   for b in range(200) for pos in range(1, 26) for s in range(3)])
    assert np.all(us >= 0.0) and np.all(us < 1.0)
    assert np.all(us * L == np.floor(us * L))          # on the 2^-24 lattice
    assert stats.kstest(us, "uniform").pvalue > 1e-3
    # keys are distinct for distinct (b, pos, stream); streams decorrelated
    keys = {O.hash_key(b, pos, s) for b in range(50) for pos in range(300)
            for s in range(3)}
    assert len(keys) == 50 * 300 * 3
    a = np.array([O.uniform(7, b, 1, 0) for b in range(5000)])
    c = np.array([O.uniform(7, b, 1, 1) for b in range(5000)])
    assert abs(np.corrcoef(a, c)[0, 1]) < 0.06


# ------------------------------------------------------ softmax / greedy
def test_softmax_closed_forms():
    z = np.array([0.3, -1.2])
    for T in (0.5, 1.0, 2.0):
        p = O.softmax_T(z, T)
        assert abs(p[0] - 1.0 / (1.0 + math.exp((z[1] - z[0]) / T))) < 1e-15
    assert np.allclose(O.softmax_T(np.full(7, 3.0), 0.7), 1.0 / 7, atol=1e-16)
    zz = np.random.default_rng(0).normal(size=50)
    ref = np.array([math.exp(v / 0.8) for v in zz])
    assert np.allclose(O.softmax_T(zz, 0.8), ref / ref.sum(), rtol=1e-13)


def test_greedy_worked_example_status_vector():
    ex = json.loads((GOLDEN / "greedy_status_ok_ok_reject_unused.json").read_text())
    target = np.array(ex["target_logits"])
    toks = np.array(ex["draft_tokens"])
    out = O.verify_linear(target, np.zeros((4, ex["V"])), toks, [0, 4],
                          [ex["temperature"]], seed=1)
    assert out["tokens"][0].tolist() == ex["expected_tokens"]
    assert out["accepted"][0] == ex["expected_accepted"]


def test_greedy_is_the_zero_temperature_limit_of_the_strict_rule():
    """At T -> 0 the strict rule degenerates into argmax prefix matching: run
    the stochastic machinery on logits scaled by 1e4 at T = 1 and the greedy
    branch at T = 0; the committed tokens must agree."""
    rng = np.random.default_rng(11)
    B, K, V = 40, 5, 300
    zt = rng.normal(size=(B * (K + 1), V)) * 2.0
    zd = np.repeat(zt.reshape(B, K + 1, V)[:, :K], 1, axis=0).reshape(B * K, V)
    zd = zd + rng.normal(size=zd.shape) * 0.8
    toks = np.argmax(zd, axis=1)            # greedy drafts
    cu = np.arange(0, B * K + 1, K)
    g = O.verify_linear(zt, zd, toks, cu, np.zeros(B), seed=5)
    s = O.verify_linear(zt * 1e4, zd * 1e4, toks, cu, np.ones(B), seed=5)
    assert np.array_equal(g["tokens"], s["tokens"])
    assert np.array_equal(g["accepted"], s["accepted"])
    assert 0 < g["accepted"].mean() < K     # both accept and reject occur


# --------------------------------------------------- losslessness (exact)
def test_lossless_exact_enumeration():
    assert lossless_error() <= 12 * 2.0 ** -23


def test_acceptance_probability_is_sum_of_min():
    assert acceptance_mass_error() <= 12 * 2.0 ** -24


def test_bonus_draw_law_is_p():
    rng = np.random.default_rng(2)
    for _ in range(4):
        p, _ = rand_pair(rng, 16)
        law = lattice_law(lambda u: O.inverse_cdf(p, u)[0], 16)
        assert np.max(np.abs(law - p)) <= 2.0 ** -23


def test_chi_square_first_token_million_draws():
    assert chi2_first_token_pvalue() > 1e-3


def test_accepted_length_closed_form():
    assert abs(accepted_length_zscore()) < 4.0


# ----------------------------------------------------------- special cases
def test_q_equal_p_accepts_everything():
    rng = np.random.default_rng(4)
    N, K, V = 2000, 3, 9
    p, _ = rand_pair(rng, V)
    target, draft, toks, cu = iid_batch(rng, N, K, V, p, p)
    out = O.verify_linear(target, draft, toks, cu, np.ones(N), seed=3)
    assert np.all(out["accepted"] == K)


def test_one_hot_draft_on_zero_target_mass_rejects_and_draws_from_p():
    V = 10
    zp = np.log(np.array([0.0, 1, 2, 3, 4, 0, 1, 2, 3, 4]) + 1e-300)
    zp[0] = -np.inf                     # p(0) = 0 exactly
    zq = np.full(V, -np.inf)
    zq[0] = 0.0                         # q one-hot at token 0
    N = 3000
    target = np.tile(zp[None], (2 * N, 1))
    draft = np.tile(zq[None], (N, 1))
    out = O.verify_linear(target, draft, np.zeros(N, int), np.arange(N + 1),
                          np.ones(N), seed=8)
    assert np.all(out["accepted"] == 0)
    p = O.softmax_T(zp, 1.0)
    law = lattice_law(lambda u: O.sample_residual_or_p(
        p, O.softmax_T(zq, 1.0), u)[0], V)
    assert np.max(np.abs(law - p)) <= 2.0 ** -23
    assert stats.chisquare(np.bincount(out["tokens"][:, 0], minlength=V)[1:],
                           N * p[1:]).pvalue > 1e-3


# ---------------------------------------------------------------- top-128
def test_top128_against_full_sort_with_ties():
    rng = np.random.default_rng(6)
    for V in (100, 128, 129, 1000, 5000):
        z = np.round(rng.normal(size=V) * 4) / 4      # many exact ties
        want = sorted(range(V), key=lambda i: (-z[i], i))[:128]
        assert O.top128_select(z).tolist() == sorted(want)
    assert O.top128_select(np.zeros(1000)).tolist() == list(range(128))
    ids, probs = O.top128_softmax(np.arange(300.0) % 7, 0.9)
    ref = np.array([math.exp((v % 7) / 0.9) for v in ids])
    assert np.allclose(probs, ref / ref.sum(), rtol=1e-13)
    assert abs(probs.sum() - 1.0) < 1e-12


def test_top128_equals_dense_when_vocab_fits():
    lb_rng = np.random.default_rng(9)
    B, K, V = 30, 3, 96
    zt = lb_rng.normal(size=(B * (K + 1), V)) * 2
    zd = lb_rng.normal(size=(B * K, V)) * 2
    toks = lb_rng.integers(0, V, B * K)
    cu = np.arange(0, B * K + 1, K)
    a = O.verify_linear(zt, zd, toks, cu, np.full(B, 0.9), seed=4)
    b = O.verify_linear(zt, zd, toks, cu, np.full(B, 0.9), seed=4,
                        rule=O.RULE_STRICT_TOP128)
    assert np.array_equal(a["tokens"], b["tokens"])
    assert np.allclose(a["pq"], b["pq"], rtol=1e-13)


# ------------------------------------------------------------------- trees
def chain_from_linear(zt, zd, toks, K):
    """Rewrite a linear batch as chain trees: node i holds d_i, target row of
    node i is p_{i+1}, draft row of node i is q_{i+1} (the leaf's unused)."""
    B = zt.shape[0] // (K + 1)
    V = zt.shape[1]
    t = zt.reshape(B, K + 1, V)
    d = np.concatenate([zd.reshape(B, K, V), np.zeros((B, 1, V))], axis=1)
    node_tok = np.concatenate([-np.ones((B, 1), int), toks.reshape(B, K)], 1)
    parent = np.tile(np.arange(-1, K)[None], (B, 1))
    return (t.reshape(-1, V), d.reshape(-1, V), node_tok.reshape(-1),
            parent.reshape(-1), np.arange(0, B * (K + 1) + 1, K + 1))


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_chain_tree_is_the_linear_verifier(T):
    rng = np.random.default_rng(12)
    B, K, V = 300, 4, 40
    zt = rng.normal(size=(B * (K + 1), V)) * 1.5
    zd = zt.reshape(B, K + 1, V)[:, :K].reshape(B * K, V) + rng.normal(size=(B * K, V))
    q = np.stack([O.softmax_T(r, 1.0) for r in zd])
    toks = np.array([rng.choice(V, p=r) for r in q]) if T > 0 else np.argmax(zd, 1)
    cu = np.arange(0, B * K + 1, K)
    lin = O.verify_linear(zt, zd, toks, cu, np.full(B, T), seed=21)
    tree = O.verify_tree(*chain_from_linear(zt, zd, toks, K), np.full(B, T),
                         seed=21, max_depth=K)
    assert np.array_equal(lin["tokens"], tree["tokens"])
    assert np.array_equal(lin["accepted"], tree["accepted"])
    assert 0 < lin["accepted"].mean() < K


def exact_rrsw_law(p, q, m):
    """Exact law of the token a depth-1 tree with m children emits: sum over
    the ordered without-replacement draws of the children and over the
    lattice of coins, using the oracle's node step and inverse CDF."""
    V = p.size
    law = np.zeros(V)
    reject_all = [1.0 - LSB] * m          # read each child's a by rejecting
    for tup in itertools.permutations(range(V), m):
        pr, left = 1.0, 1.0
        for x in tup:
            pr *= q[x] / left
            left -= q[x]
        _, final_law, tested = O.rrsw_node(p, q, list(tup), reject_all)
        reach = 1.0
        for j, (_, a) in enumerate(tested):
            A = lattice_accept_fraction(a)
            law[tup[j]] += pr * reach * A
            reach *= 1.0 - A
        if reach > 0.0:
            law += pr * reach * lattice_law(
                lambda u: O.inverse_cdf(final_law, u)[0], V)
    return law


def rrsw_error(seed=13, V=6, m=3, trials=2):
    rng = np.random.default_rng(seed)
    worst = 0.0
    for _ in range(trials):
        p, q = rand_pair(rng, V, scale=1.2)
        worst = max(worst, float(np.max(np.abs(exact_rrsw_law(p, q, m) - p))))
    return worst


def test_rrsw_depth1_exact_enumeration():
    assert rrsw_error() <= 2.0 ** -20


def test_rrsw_depth1_four_siblings_exact():
    assert rrsw_error(seed=14, V=7, m=4, trials=1) <= 2.0 ** -20


def test_rrsw_chi_square_over_trees():
    rng = np.random.default_rng(15)
    N, V, m = 100_000, 8, 3
    p, q = rand_pair(rng, V, scale=1.2)
    zp, zq = np.log(p), np.log(q)
    target = np.tile(zp[None], (N * (m + 1), 1))
    draft = np.tile(zq[None], (N * (m + 1), 1))
    g = rng.gumbel(size=(N, V)) + zq
    kids = np.argsort(-g, axis=1)[:, :m]     # ordered, without replacement
    node_tok = np.concatenate([-np.ones((N, 1), int), kids], 1).reshape(-1)
    parent = np.tile(np.array([-1] + [0] * m)[None], (N, 1)).reshape(-1)
    out = O.verify_tree(target, draft, node_tok, parent,
                        np.arange(0, N * (m + 1) + 1, m + 1), np.ones(N),
                        seed=77, max_depth=1)
    counts = np.bincount(out["tokens"][:, 0], minlength=V)
    assert stats.chisquare(counts, N * p).pvalue > 1e-3


# ------------------------------------------- pins catch planted mistakes
def test_pins_catch_swapped_residual(monkeypatch):
    monkeypatch.setattr(O, "residual", lambda p, q: np.maximum(0.0, q - p))
    assert lossless_error(trials=2) > 1e-3


def test_pins_catch_inverted_ratio(monkeypatch):
    monkeypatch.setattr(O, "acceptance_prob",
                        lambda p, q: 1.0 if p <= q else q / p)
    assert acceptance_mass_error(trials=2) > 1e-3


def test_pins_catch_off_by_one_cdf(monkeypatch):
    real = O.inverse_cdf

    def shifted(w, u):
        x, f = real(w, u)
        return min(x + 1, w.size - 1), f
    monkeypatch.setattr(O, "inverse_cdf", shifted)
    rng = np.random.default_rng(2)
    p, _ = rand_pair(rng, 16)
    law = lattice_law(lambda u: O.inverse_cdf(p, u)[0], 16)
    assert np.max(np.abs(law - p)) > 1e-3


def test_pins_catch_shared_coin(monkeypatch):
    real = O.uniform
    monkeypatch.setattr(O, "uniform",
                        lambda seed, b, pos, s: real(seed, b, 1, s))
    assert abs(accepted_length_zscore(N=20_000)) > 6.0


def test_pins_catch_missing_without_replacement(monkeypatch):
    """Keeping the rejected token in the draft law (no renormalisation)
    breaks losslessness of the sibling walk."""
    def with_replacement(p, q, child_tokens, coins):
        p_j = np.asarray(p, float)
        tested = []
        for j, x in enumerate(child_tokens):
            a = O.acceptance_prob(p_j[x], q[x])
            tested.append((coins[j], a))
            if O.coin_accepts(coins[j], a):
                return j, None, tested
            r = O.residual(p_j, q)
            p_j = r / r.sum()
        return -1, p_j, tested
    monkeypatch.setattr(O, "rrsw_node", with_replacement)
    assert rrsw_error(trials=1) > 1e-3

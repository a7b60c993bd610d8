"""Pins for the oracle's relaxed CACTUS rule and its low-support guard
("Acceptance Is Not Speed (arXiv:2610.23818)", §6 RULE 1-3 and §7 item 3).

Each pin checks the oracle against something other than itself: hand-worked
values, a library ranking routine, the strict and greedy rules (pinned in
test_oracle_pins.py) as limiting cases, and the law of the first emitted token
derived in closed form. Planted mistakes at the bottom show the pins bite.
"""
import math

import numpy as np
from scipy import stats

from oracle import spec_oracle as O


def rand_pair(rng, V, scale=1.5):
    zp = scale * rng.normal(size=V)
    zq = zp + scale * rng.normal(size=V)
    return O.softmax_T(zp, 1.0), O.softmax_T(zq, 1.0)


def iid_batch(rng, N, K, V, p, q):
    target = np.tile(np.log(p)[None], (N * (K + 1), 1))
    draft = np.tile(np.log(q)[None], (N * K, 1))
    toks = rng.choice(V, size=N * K, p=q)
    return target, draft, toks, np.arange(0, N * K + 1, K)


# ----------------------------------------------------------- closed forms
def test_gamma_hand_values():
    # p + sqrt(2 alpha p (1 - p)) worked by hand
    assert O.cactus_gamma(0.5, 0.125) == 0.75            # 0.5 + sqrt(0.0625)
    assert abs(O.cactus_gamma(0.1, 0.5) - 0.4) < 1e-15   # 0.1 + sqrt(0.09)
    assert O.cactus_gamma(0.9, 1.0) == 1.0               # 0.9 + 0.424 clipped
    assert O.cactus_gamma(0.0, 3.0) == 0.0               # no mass, no boost
    assert O.cactus_gamma(1.0, 3.0) == 1.0
    assert O.cactus_gamma(0.37, 0.0) == 0.37             # alpha = 0: gamma = p


def test_target_rank_hand_example_and_scipy():
    z = np.array([3.0, 1.0, 3.0, 2.0])
    assert [O.target_rank(z, d) for d in range(4)] == [1, 4, 1, 3]
    rng = np.random.default_rng(0)
    for V in (7, 50, 1000):
        z = np.round(rng.normal(size=V) * 2) / 2          # many ties
        want = stats.rankdata(-z, method="min")          # 1 + #greater
        got = [O.target_rank(z, d) for d in range(V)]
        assert np.array_equal(got, want)


def test_guard_predicate():
    assert O.low_support(0.05, 1, 10, 0.10)              # p below threshold
    assert O.low_support(0.5, 11, 10, 0.10)              # outside top 10
    assert not O.low_support(0.5, 10, 10, 0.10)
    assert not O.low_support(0.10, 3, 10, 0.10)          # p == threshold passes
    assert not O.low_support(1e-9, 10 ** 6, 0, 0.0)      # guard off


# ------------------------------------------------------ limiting cases
def test_alpha_zero_without_guard_is_the_strict_rule():
    rng = np.random.default_rng(1)
    N, K, V = 400, 5, 40
    target = 1.3 * rng.normal(size=(N * (K + 1), V))
    draft = target[np.repeat(np.arange(N) * (K + 1), K) + np.tile(np.arange(K), N)] \
        + 1.3 * rng.normal(size=(N * K, V))
    toks = np.array([rng.choice(V, p=O.softmax_T(r, 1.0)) for r in draft])
    cu = np.arange(0, N * K + 1, K)
    T = rng.choice([0.0, 0.5, 1.0], size=N)
    s = O.verify_linear(target, draft, toks, cu, T, seed=5)
    c = O.verify_linear(target, draft, toks, cu, T, seed=5, rule=O.RULE_CACTUS, alpha=0.0)
    assert np.array_equal(s["tokens"], c["tokens"])
    assert np.array_equal(s["accepted"], c["accepted"])
    assert 0 < s["accepted"].mean() < K


def test_rank_one_guard_with_saturated_gamma_is_greedy_matching():
    """alpha large makes gamma = 1 for every 0 < p < 1, so every draft passes
    the coin; max_rank = 1 then accepts exactly the target argmax, i.e. the
    accepted length is the greedy prefix (continuous logits: no ties)."""
    rng = np.random.default_rng(2)
    N, K, V = 300, 4, 6
    target = rng.normal(size=(N * (K + 1), V))
    draft = rng.normal(size=(N * K, V))
    toks = rng.integers(0, V, N * K)
    cu = np.arange(0, N * K + 1, K)
    c = O.verify_linear(target, draft, toks, cu, np.ones(N), seed=8,
                        rule=O.RULE_CACTUS, alpha=1e9, max_rank=1)
    g = O.verify_linear(target, draft, toks, cu, np.ones(N), seed=8, rule=O.RULE_GREEDY)
    assert np.array_equal(c["accepted"], g["accepted"])
    assert 0 < g["accepted"].mean() < K


def test_probability_floor_of_one_rejects_every_sampled_draft():
    rng = np.random.default_rng(3)
    p, q = rand_pair(rng, 9)
    target, draft, toks, cu = iid_batch(rng, 500, 3, 9, p, q)
    T = np.where(np.arange(500) % 5 == 0, 0.0, 1.0)       # every 5th greedy
    c = O.verify_linear(target, draft, toks, cu, T, seed=4, rule=O.RULE_CACTUS,
                        alpha=2.0, min_prob=1.0)
    assert np.all(c["accepted"][T > 0] == 0)
    g = O.verify_linear(target, draft, toks, cu, T, seed=4, rule=O.RULE_GREEDY)
    assert np.array_equal(c["accepted"][T == 0], g["accepted"][T == 0])


# ------------------------------------------ law of the first token (K=1)
def first_token_law(p, q, alpha):
    """Draft x ~ q accepted with probability min(1, gamma(x)/q(x)); on
    rejection a draw from norm(max(0, p - q))."""
    g = np.array([O.cactus_gamma(v, alpha) for v in p])
    acc = np.minimum(q, g)                     # q(x) * min(1, gamma/q)
    r = np.maximum(0.0, p - q)
    return acc + (1.0 - acc.sum()) * r / r.sum(), float(acc.sum())


def cactus_acceptance_zscore(alpha=0.05, seed=6, N=100_000, V=10):
    rng = np.random.default_rng(seed)
    p, q = rand_pair(rng, V, scale=1.0)
    target, draft, toks, cu = iid_batch(rng, N, 1, V, p, q)
    out = O.verify_linear(target, draft, toks, cu, np.ones(N), seed=11,
                          rule=O.RULE_CACTUS, alpha=alpha)
    _, acc = first_token_law(p, q, alpha)
    assert acc > float(np.minimum(p, q).sum()) + 0.02   # lossy: accepts more
    return (float(np.mean(out["accepted"])) - acc) / math.sqrt(acc * (1 - acc) / N)


def cactus_first_token_pvalue(alpha=0.05, seed=7, N=300_000, V=8):
    rng = np.random.default_rng(seed)
    p, q = rand_pair(rng, V, scale=1.5)
    target, draft, toks, cu = iid_batch(rng, N, 1, V, p, q)
    out = O.verify_linear(target, draft, toks, cu, np.ones(N), seed=12,
                          rule=O.RULE_CACTUS, alpha=alpha)
    law, _ = first_token_law(p, q, alpha)
    counts = np.bincount(out["tokens"][:, 0], minlength=V)
    return stats.chisquare(counts, N * law).pvalue


def test_cactus_acceptance_rate_closed_form():
    assert abs(cactus_acceptance_zscore()) < 4.0


def test_cactus_first_token_law_chi_square():
    assert cactus_first_token_pvalue() > 1e-3


# ------------------------------------------- pins catch planted mistakes
def test_pins_catch_gamma_ignoring_alpha(monkeypatch):
    monkeypatch.setattr(O, "cactus_gamma", lambda p, alpha: p)
    rng = np.random.default_rng(6)
    p, q = rand_pair(rng, 10, scale=1.0)
    target, draft, toks, cu = iid_batch(rng, 20_000, 1, 10, p, q)
    out = O.verify_linear(target, draft, toks, cu, np.ones(20_000), seed=11,
                          rule=O.RULE_CACTUS, alpha=0.05)
    monkeypatch.undo()
    _, acc = first_token_law(p, q, 0.05)
    z = (out["accepted"].mean() - acc) / math.sqrt(acc * (1 - acc) / 20_000)
    assert abs(z) > 6.0


def test_pins_catch_rank_guard_off_by_one(monkeypatch):
    monkeypatch.setattr(O, "low_support",
                        lambda p, rank, k, pmin: (k > 0 and rank >= k) or p < pmin)
    rng = np.random.default_rng(2)
    N, K, V = 300, 4, 6
    target = rng.normal(size=(N * (K + 1), V))
    draft = rng.normal(size=(N * K, V))
    toks = rng.integers(0, V, N * K)
    cu = np.arange(0, N * K + 1, K)
    c = O.verify_linear(target, draft, toks, cu, np.ones(N), seed=8,
                        rule=O.RULE_CACTUS, alpha=1e9, max_rank=1)
    monkeypatch.undo()
    g = O.verify_linear(target, draft, toks, cu, np.ones(N), seed=8, rule=O.RULE_GREEDY)
    assert not np.array_equal(c["accepted"], g["accepted"])


def test_pins_catch_residual_against_relaxed_law(monkeypatch):
    """Drawing the correction from max(0, gamma - q) instead of the plain
    residual changes the first-token law."""
    real = O.sample_residual_or_p
    monkeypatch.setattr(O, "sample_residual_or_p",
                        lambda p, q, u: real(np.minimum(p + np.sqrt(0.1 * p * (1 - p)), 1.0),
                                             q, u))
    assert cactus_first_token_pvalue(N=100_000) < 1e-6

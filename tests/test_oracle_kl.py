"""Pins for the oracle's per-position KL(p || q) (R13; "Test-Time
Speculation", §2 step 3): closed forms, invariances and scipy's relative
entropy, on single rows and through the verifier."""
import math

import numpy as np
from scipy import special

from oracle import spec_oracle as O


def test_two_point_closed_form():
    for a, b in ((0.3, 0.6), (0.9, 0.1), (0.5, 0.5)):
        want = a * math.log(a / b) + (1 - a) * math.log((1 - a) / (1 - b))
        assert abs(O.kl_divergence([a, 1 - a], [b, 1 - b]) - want) < 1e-15


def test_zero_for_equal_laws_and_shifted_logits():
    rng = np.random.default_rng(0)
    z = rng.normal(size=500) * 3
    p = O.softmax_T(z, 0.7)
    assert O.kl_divergence(p, p) == 0.0
    assert abs(O.kl_divergence(p, O.softmax_T(z + 4.25, 0.7))) < 1e-13


def test_support_rules():
    assert O.kl_divergence([0.5, 0.5, 0.0], [0.25, 0.75, 0.0]) == \
        O.kl_divergence([0.5, 0.5], [0.25, 0.75])        # p = 0 terms vanish
    assert O.kl_divergence([0.5, 0.5], [1.0, 0.0]) == float("inf")


def test_matches_scipy_relative_entropy():
    rng = np.random.default_rng(1)
    for V in (3, 40, 5000):
        for T in (0.3, 1.0, 2.0):
            zt, zd = rng.normal(size=V) * 2, rng.normal(size=V) * 2
            p, q = special.softmax(zt / T), special.softmax(zd / T)
            want = float(np.sum(special.rel_entr(p, q)))
            got = O.kl_divergence(O.softmax_T(zt, T), O.softmax_T(zd, T))
            assert abs(got - want) <= 1e-12 * max(1.0, want)


def test_verifier_reports_kl_of_every_draft_position():
    rng = np.random.default_rng(2)
    N, K, V = 30, 4, 60
    target = rng.normal(size=(N * (K + 1), V)) * 2
    t_of_d = np.repeat(np.arange(N) * (K + 1), K) + np.tile(np.arange(K), N)
    draft = target[t_of_d] + rng.normal(size=(N * K, V))
    toks = rng.integers(0, V, N * K)
    cu = np.arange(0, N * K + 1, K)
    T = np.where(np.arange(N) % 3 == 0, 0.0, 0.8)
    out = O.verify_linear(target, draft, toks, cu, T, seed=1)
    for r in range(N * K):
        b = r // K
        if T[b] < O.GREEDY_T:
            assert np.isnan(out["kl"][r])
            continue
        p = special.softmax(target[t_of_d[r]] / T[b])
        q = special.softmax(draft[r] / T[b])
        assert abs(out["kl"][r] - np.sum(special.rel_entr(p, q))) < 1e-12


def test_truncated_draft_law_gives_infinite_kl():
    """Under the top-128 rule q is 0 outside 128 ids while p is positive
    everywhere, so KL(p || q) is +inf; with V <= 128 nothing is cut."""
    rng = np.random.default_rng(3)
    for V, finite in ((300, False), (100, True)):
        target = rng.normal(size=(2, V))
        draft = target[:1] + rng.normal(size=(1, V))
        out = O.verify_linear(target, draft, [0], [0, 1], [1.0], seed=1,
                              rule=O.RULE_STRICT_TOP128)
        assert np.isfinite(out["kl"][0]) == finite


def test_pins_catch_swapped_arguments(monkeypatch):
    real = O.kl_divergence
    monkeypatch.setattr(O, "kl_divergence", lambda p, q: real(q, p))
    rng = np.random.default_rng(1)
    zt, zd = rng.normal(size=40) * 2, rng.normal(size=40) * 2
    p, q = special.softmax(zt), special.softmax(zd)
    assert abs(O.kl_divergence(O.softmax_T(zt, 1.0), O.softmax_T(zd, 1.0))
               - np.sum(special.rel_entr(p, q))) > 1e-3

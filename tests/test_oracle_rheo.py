"""Pins of the oracle's RheoSampling tree construction ("RheoSampling 2026",
§2 dual identities, §3 the rheostat m and the top-128 cut, §7 no temperature
in construction). Each check rests on a hand-worked case, a library routine
(scipy's softmax, Python's sorted) or an invariant the page states, not on
the oracle's own formulas."""
import math

import numpy as np
import pytest
from scipy import special, stats

from oracle import spec_oracle as O

EPS = 1e-6


def expand_one(z, T=1.0, K=3, m=1, eps=EPS, level=0, seed=11, score=0.0,
               n_keep=None):
    z = np.asarray(z, dtype=np.float64)[None, :]
    return O.rheo_expand(z, [0, 1], [score], [T], seed, level, K, m, eps,
                         n_keep or K)


# ------------------------------------------------------ hand-worked example
# z over V = 6 ids: best first the order is 3 (z=3), 0 (2), 2 (1), 1 (0),
# 5 (0, tie with 1: lower id first), 4 (-1).
Z6 = [2.0, 0.0, 1.0, 3.0, -1.0, 0.0]
SUM6 = math.exp(2) + 1 + math.e + math.exp(3) + math.exp(-1) + 1
Q6 = {0: math.exp(2) / SUM6, 1: 1 / SUM6, 2: math.e / SUM6,
      3: math.exp(3) / SUM6, 4: math.exp(-1) / SUM6, 5: 1 / SUM6}
# children (K = 3, m = 1) for every possible probe, worked by hand:
# lead = best token other than the probe, then the probe, then the next one
HAND_SLOTS_K3_M1 = {3: [0, 3, 2], 0: [3, 0, 2], 2: [3, 2, 0], 1: [3, 1, 0],
                    5: [3, 5, 0], 4: [3, 4, 0]}


# the true sampling law at T = 4: exp(z/4) / sum exp(z/4)
SUM6_T4 = sum(math.exp(v / 4) for v in Z6)
QT6_T4 = {x: math.exp(Z6[x] / 4) / SUM6_T4 for x in range(6)}
HAND_LEVELS = range(40)


@pytest.mark.parametrize("level", HAND_LEVELS)
def test_hand_worked_children_and_proxies(level):
    r = expand_one(Z6, T=4.0, K=3, m=1, level=level)
    tok = r["child_token"][0].tolist()
    probe = tok[1]                       # m = 1: the probe sits in slot 2
    assert tok == HAND_SLOTS_K3_M1[probe]
    # proxies: deterministic children their own unscaled q; the probe
    # q(x_2) + eps, x_2 = token 0 (the second best)
    want = [Q6[t] for t in tok]
    want[1] = Q6[0] + EPS
    np.testing.assert_allclose(r["child_qproxy"][0], want, rtol=1e-13)
    np.testing.assert_allclose(r["child_score"][0], np.log(want), rtol=1e-13)
    np.testing.assert_allclose(r["child_qtrue"][0], [QT6_T4[t] for t in tok],
                               rtol=1e-13)


def test_hand_worked_levels_reach_every_probe():
    probes = {int(expand_one(Z6, T=4.0, K=3, m=1, level=l)["child_token"][0, 1])
              for l in HAND_LEVELS}
    assert probes == set(range(6))


def test_hand_worked_m0_puts_the_probe_first():
    for level in range(8):
        r = expand_one(Z6, K=4, m=0, level=level)
        tok = r["child_token"][0].tolist()
        probe = tok[0]
        rest = [t for t in [3, 0, 2, 1, 5, 4] if t != probe][:3]
        assert tok == [probe] + rest
        assert r["child_qproxy"][0, 0] == pytest.approx(Q6[3] + EPS, rel=1e-13)


# ------------------------------------------------------------- invariants
def zipf_rows(n, V, seed, scale=2.0):
    rng = np.random.default_rng(seed)
    rank = np.stack([rng.permutation(V) + 1 for _ in range(n)])
    return scale * rng.standard_normal((n, V)) - 1.1 * np.log(rank)


@pytest.mark.parametrize("m", [0, 1, 3])
def test_probe_ranks_after_at_most_m_siblings(m):
    z = zipf_rows(40, 500, seed=1)
    cu = [0, 20, 40]
    r = O.rheo_expand(z, cu, np.zeros(40), [1.0, 0.7], 5, 2, 8, m, EPS, 8)
    for f in range(40):
        sc = r["child_score"][f]
        above = int(np.sum(sc > sc[m]))
        assert above <= m                 # the probe holds slot m+1 or better
        order = sorted(range(500), key=lambda x: (-z[f, x], x))
        if r["child_token"][f, m] not in order[: m + 1]:
            assert above == m             # behind exactly the m leads


def test_deterministic_children_are_the_best_tokens_except_the_probe():
    z = np.round(zipf_rows(16, 300, seed=2), 1)   # rounding makes ties
    r = O.rheo_expand(z, [0, 16], np.zeros(16), [0.9], 3, 0, 6, 2, EPS, 4)
    for f in range(16):
        tok = r["child_token"][f].tolist()
        probe = tok[2]
        det = tok[:2] + tok[3:]
        assert len(set(tok)) == 6 and probe not in det
        # sorted() by (-z, id) over the whole row, not the oracle's lexsort
        best = [x for x in sorted(range(300), key=lambda x: (-z[f, x], x))
                if x != probe][:5]
        assert det == best


def test_construction_ignores_temperature():
    z = zipf_rows(1, 400, seed=3)
    top = np.sort(np.argpartition(-z[0], 128)[:128])
    q = dict(zip(top.tolist(), special.softmax(z[0, top]).tolist()))
    for T in (0.2, 1.0, 3.0):
        r = expand_one(z[0], T=T, K=10, m=1, level=7)
        for s, t in enumerate(r["child_token"][0]):
            if s != 1:
                assert r["child_qproxy"][0, s] == pytest.approx(q[int(t)], rel=1e-12)


def test_true_sampling_probability_is_the_tempered_top128_law():
    z = zipf_rows(1, 400, seed=4)
    top = np.sort(np.argpartition(-z[0], 128)[:128])
    for T in (0.4, 1.3):
        qt = dict(zip(top.tolist(), special.softmax(z[0, top] / T).tolist()))
        r = expand_one(z[0], T=T, K=10, m=1, level=3)
        for s, t in enumerate(r["child_token"][0]):
            assert r["child_qtrue"][0, s] == pytest.approx(qt[int(t)], rel=1e-12)


def test_probe_law_chi_square():
    """The probe is a draw from q~ = softmax(z/T) over the top 128 (§2)."""
    z = zipf_rows(1, 300, seed=5, scale=0.5)[0]
    T = 0.8
    top = np.sort(np.argpartition(-z, 128)[:128])
    qt = special.softmax(z[top] / T)
    n = 20000
    zz = np.repeat(z[None, :], 50, axis=0)
    counts = dict.fromkeys(top.tolist(), 0)
    for lvl in range(n // 50):
        r = O.rheo_expand(zz, [0, 50], np.zeros(50), [T], 99, lvl, 1, 0, EPS, 1)
        for t in r["child_token"][:, 0]:
            counts[int(t)] += 1
    obs = np.array([counts[t] for t in top.tolist()], dtype=np.float64)
    exp = qt * n
    big = exp >= 5
    chi = np.sum((obs[big] - exp[big]) ** 2 / exp[big])
    rest_o, rest_e = obs[~big].sum(), exp[~big].sum()
    if rest_e > 0:
        chi += (rest_o - rest_e) ** 2 / rest_e
    dof = int(big.sum()) - (0 if rest_e > 0 else 1)
    assert stats.chi2.sf(chi, dof) > 1e-4
    assert obs[~np.isin(np.arange(top.size), np.nonzero(qt > 0)[0])].sum() == 0


def test_greedy_probe_is_the_argmax():
    z = zipf_rows(6, 256, seed=6)
    r = O.rheo_expand(z, [0, 6], np.zeros(6), [0.01], 1, 0, 4, 1, EPS, 4)
    for f in range(6):
        assert r["child_token"][f, 1] == int(np.argmax(z[f]))
        assert r["child_qtrue"][f, 1] == 1.0
        assert (r["child_qtrue"][f, [0, 2, 3]] == 0.0).all()


def test_small_vocabulary_uses_every_token():
    z = zipf_rows(3, 9, seed=7)
    r = O.rheo_expand(z, [0, 3], np.zeros(3), [1.0], 2, 0, 9, 4, EPS, 27)
    for f in range(3):
        assert sorted(r["child_token"][f].tolist()) == list(range(9))
    assert sorted(r["keep"][0].tolist()) == list(range(27))


def test_scores_multiply_along_a_path():
    """exp(score) of a child = parent's path score x its proxy (§2: proxies
    rank candidates through path scores)."""
    z = zipf_rows(4, 300, seed=8)
    parent_scores = np.log([1.0, 0.5, 0.25, 0.01])
    r = O.rheo_expand(z, [0, 4], parent_scores, [1.0], 4, 1, 5, 1, EPS, 20)
    for f in range(4):
        np.testing.assert_allclose(np.exp(r["child_score"][f]),
                                   np.exp(parent_scores[f]) * r["child_qproxy"][f],
                                   rtol=1e-12)


def test_selection_keeps_the_best_scores_per_tree():
    z = np.round(zipf_rows(12, 200, seed=9), 0)
    cu = [0, 5, 5, 12]                     # the middle tree has no frontier
    fs = np.round(np.random.default_rng(1).uniform(-3, 0, 12), 0)
    K, n_keep = 4, 7
    r = O.rheo_expand(z, cu, fs, [1.0, 1.0, 0.6], 8, 0, K, 1, 0.0, n_keep)
    flat = r["child_score"].reshape(-1)
    for b in range(3):
        cand = list(range(cu[b] * K, cu[b + 1] * K))
        want = sorted(cand, key=lambda c: (-flat[c], c))[:n_keep]
        got = [c for c in r["keep"][b].tolist() if c >= 0]
        assert got == want
        assert (r["keep"][b][len(want):] == -1).all()
    assert (r["keep"][1] == -1).all()


# --------------------------------------------- pins catch planted mistakes
def _run_pins():
    test_hand_worked_children_and_proxies(0)
    test_hand_worked_children_and_proxies(5)
    test_hand_worked_m0_puts_the_probe_first()
    test_probe_ranks_after_at_most_m_siblings(1)
    test_deterministic_children_are_the_best_tokens_except_the_probe()
    test_construction_ignores_temperature()
    test_greedy_probe_is_the_argmax()
    test_selection_keeps_the_best_scores_per_tree()


def test_pins_catch_proxy_off_by_one(monkeypatch):
    monkeypatch.setattr(O, "rheo_probe_proxy",
                        lambda qr, m, eps: float(qr[max(m - 1, 0)]) + eps)
    with pytest.raises(AssertionError):
        _run_pins()


def test_pins_catch_tempered_ranking(monkeypatch):
    real = O.rheo_expand

    def tempered(draft, cu, fs, temps, *a):
        saved = O.rheo_ranking_law
        T = float(np.asarray(temps)[0])
        O.rheo_ranking_law = lambda z, ids: special.softmax(np.asarray(z)[ids] / T)
        try:
            return real(draft, cu, fs, temps, *a)
        finally:
            O.rheo_ranking_law = saved
    monkeypatch.setattr(O, "rheo_expand", tempered)
    with pytest.raises(AssertionError):
        _run_pins()


def test_pins_catch_duplicate_probe(monkeypatch):
    def keep_probe_token(order, probe, K, m):
        det = [int(x) for x in order][: K - 1]
        return det[:m] + [probe] + det[m:]
    monkeypatch.setattr(O, "rheo_slots", keep_probe_token)
    with pytest.raises(AssertionError):
        _run_pins()


def test_pins_catch_probe_after_every_lead(monkeypatch):
    def probe_last(order, probe, K, m):
        det = [int(x) for x in order if int(x) != probe][: K - 1]
        return det + [probe]
    monkeypatch.setattr(O, "rheo_slots", probe_last)
    with pytest.raises(AssertionError):
        _run_pins()


def test_pins_catch_ascending_selection(monkeypatch):
    def worst_first(scores, n_keep):
        scores = np.asarray(scores, dtype=np.float64)
        order = np.lexsort((np.arange(scores.size), scores))
        out = np.full(n_keep, -1, dtype=np.int64)
        out[: min(n_keep, scores.size)] = order[:n_keep]
        return out
    monkeypatch.setattr(O, "rheo_select", worst_first)
    with pytest.raises(AssertionError):
        _run_pins()


# ------------------------- verifying built trees: point-mass children (R19)
def _node_output_law(p, qt, kids, fixed):
    """Exact law of the token one node emits: every accept / reject branch
    of the oracle's rrsw_node, weighted by its acceptance probabilities
    (coin 0 accepts whenever a > 0; a coin just below 1 rejects unless
    a = 1), plus the final draw's law when every child is rejected."""
    V = p.size
    out = np.zeros(V)
    for k in range(len(kids) + 1):            # children 0..k-1 rejected, k accepted
        coins = [1.0 - 2.0 ** -40] * k + ([0.0] if k < len(kids) else [])
        coins += [0.0] * (len(kids) - len(coins))
        acc, law, tested = O.rrsw_node(p, qt, kids, coins, fixed)
        if acc != (k if k < len(kids) else -1):
            continue                          # this branch has probability 0
        w = 1.0
        for j in range(min(k, len(tested))):
            w *= 1.0 - tested[j][1]
        if k < len(kids):
            out[kids[k]] += w * tested[k][1]
        elif w > 0.0:
            out += w * law / law.sum()
    return out


def _rheo_node_law(zd, zt, T, K, m, probe_first=True):
    """Output law of one node built by construction and verified with the
    probe drawn from q~ (enumerated exactly) and point-mass leads."""
    ids = np.arange(zd.size)
    qt = special.softmax(zd / T)               # V <= 128: the top-128 law is dense
    p = special.softmax(zt / T)
    order = sorted(ids.tolist(), key=lambda x: (-zd[x], x))
    out = np.zeros(zd.size)
    for u in ids:
        slots = O.rheo_slots(np.array(order), int(u), K, m)
        det = [x for x in slots if x != u]
        if probe_first:
            kids, fixed = [int(u)] + det, [False] + [True] * len(det)
        else:
            kids, fixed = slots, [x != u for x in slots]
        out += qt[u] * _node_output_law(p, qt, kids, fixed)
    return out, p


@pytest.mark.parametrize("K,m,T,seed", [(3, 1, 1.0, 0), (4, 0, 0.7, 1), (5, 2, 1.3, 2),
                                        (6, 5, 0.9, 3), (2, 1, 2.0, 4)])
def test_built_node_verified_probe_first_is_lossless(K, m, T, seed):
    """"RheoSampling 2026" §6 Teorema 1 for one built node: the emitted
    token's law equals p exactly."""
    rng = np.random.default_rng(seed)
    zd = rng.standard_normal(6) * 1.5
    zt = zd + rng.standard_normal(6)
    law, p = _rheo_node_law(zd, zt, T, K, m)
    np.testing.assert_allclose(law, p, atol=1e-12)


def test_leads_tested_before_the_probe_are_not_lossless():
    """The reading behind R18: the leads depend on the probe's token, so
    testing them first distorts the law; probe first restores it."""
    rng = np.random.default_rng(7)
    zd = rng.standard_normal(6) * 1.5
    zt = zd + rng.standard_normal(6) * 1.5
    bad, p = _rheo_node_law(zd, zt, 1.0, 3, 2, probe_first=False)
    good, _ = _rheo_node_law(zd, zt, 1.0, 3, 2)
    assert np.abs(bad - p).max() > 1e-3
    np.testing.assert_allclose(good, p, atol=1e-12)


def test_fixed_children_alone_are_lossless():
    rng = np.random.default_rng(8)
    zt = rng.standard_normal(5)
    p = special.softmax(zt)
    qt = special.softmax(rng.standard_normal(5))
    law = _node_output_law(p, qt, [3, 0, 4], [True, True, True])
    np.testing.assert_allclose(law, p, atol=1e-12)
    # a single fixed child x is accepted with probability p(x)
    _, _, tested = O.rrsw_node(p, qt, [2], [0.5], [True])
    assert tested[0][1] == pytest.approx(p[2], rel=1e-14)


def test_verify_tree_with_point_mass_children_chain_and_greedy():
    """Through verify_tree: a chain tree of fixed children emits the token
    of each accepted node; greedy trees ignore the flags."""
    rng = np.random.default_rng(9)
    V = 7
    zt = rng.standard_normal((3, V))
    zd = rng.standard_normal((3, V))
    parent = [-1, 0, 1]
    tokens = [-1, int(np.argmax(zt[0])), int(np.argmax(zt[1]))]
    for T in (0.01, 1.0):
        r = O.verify_tree(zt, zd, tokens, parent, [0, 3], [T], 5, 2, node_fixed=[0, 1, 1])
        assert 0 <= r["accepted"][0] <= 2
        n = int(r["accepted"][0])
        assert r["tokens"][0, :n].tolist() == tokens[1:1 + n]
        if T < 0.05:
            assert n == 2                      # argmax children are accepted greedily


def _pins_rheo_verify():
    test_built_node_verified_probe_first_is_lossless(3, 1, 1.0, 0)
    test_built_node_verified_probe_first_is_lossless(5, 2, 1.3, 2)
    test_fixed_children_alone_are_lossless()


def test_pins_catch_fixed_child_tested_against_q(monkeypatch):
    real = O.rrsw_node
    monkeypatch.setattr(O, "rrsw_node",
                        lambda p, q, kids, coins, fixed=None: real(p, q, kids, coins, None))
    with pytest.raises(AssertionError):
        _pins_rheo_verify()


def test_pins_catch_fixed_child_accepted_with_its_draft_ratio(monkeypatch):
    real_acc = O.acceptance_prob
    # a point mass mistaken for a draw from q: min(1, p / q(x)) instead of p
    monkeypatch.setattr(O, "acceptance_prob",
                        lambda p_d, q_d: real_acc(p_d, 0.5 if q_d == 1.0 else q_d))
    with pytest.raises(AssertionError):
        _pins_rheo_verify()

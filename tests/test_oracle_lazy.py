"""Pins for the position-lazy reading (R12 of the oracle): the verifier's
result does not depend on any row after position n+1 ("Penolakan
memendekkan pekerjaan speculative", nalar.dev), so a schedule that never
reads those rows returns the same tokens."""
import numpy as np

from oracle import spec_oracle as O


def batch(rng, N=200, K=5, V=30):
    target = 1.5 * rng.normal(size=(N * (K + 1), V))
    t_of_d = np.repeat(np.arange(N) * (K + 1), K) + np.tile(np.arange(K), N)
    draft = target[t_of_d] + 1.2 * rng.normal(size=(N * K, V))
    toks = np.array([rng.choice(V, p=O.softmax_T(r, 1.0)) for r in draft])
    cu = np.arange(0, N * K + 1, K)
    T = rng.choice([0.0, 0.6, 1.0, 1.5], size=N)
    return target, draft, toks, cu, T


def unread_mask(cu, n, K):
    """Target and draft rows a lazy verifier skips (after position n+1)."""
    N = cu.size - 1
    tmask = np.zeros(N * (K + 1), bool)
    dmask = np.zeros(N * K, bool)
    for b in range(N):
        m = min(int(n[b]) + 1, K)
        tmask[b * (K + 1) + int(n[b]) + 1:(b + 1) * (K + 1)] = True
        dmask[b * K + m:(b + 1) * K] = True
    return tmask, dmask


def test_rows_after_the_first_rejection_are_never_used():
    rng = np.random.default_rng(0)
    target, draft, toks, cu, T = batch(rng)
    K = 5
    for rule, kw in ((O.RULE_STRICT, {}), (O.RULE_CACTUS, dict(alpha=0.3, max_rank=4))):
        ref = O.verify_linear(target, draft, toks, cu, T, seed=3, rule=rule, **kw)
        n = ref["accepted"]
        assert 0 < n.mean() < K and np.any(n == K) and np.any(n == 0)
        tmask, dmask = unread_mask(cu, n, K)
        t2, d2 = target.copy(), draft.copy()
        t2[tmask] = rng.normal(size=(tmask.sum(), target.shape[1])) * 5.0
        d2[dmask] = rng.normal(size=(dmask.sum(), draft.shape[1])) * 5.0
        got = O.verify_linear(t2, d2, toks, cu, T, seed=3, rule=rule, **kw)
        assert np.array_equal(got["tokens"], ref["tokens"])
        assert np.array_equal(got["accepted"], ref["accepted"])
        # and the positions a lazy verifier reads keep their p(d), q(d)
        lz = O.lazy_view(ref, cu)
        keep = ~np.isnan(lz["pq"][:, 0])
        assert np.array_equal(got["pq"][keep], ref["pq"][keep])
        # while a row that is read does matter
        t3 = target.copy()
        b = int(np.nonzero((n > 0) & (n < K) & (T >= 0.05))[0][0])
        t3[b * (K + 1)] = t3[b * (K + 1)][::-1]
        moved = O.verify_linear(t3, draft, toks, cu, T, seed=3, rule=rule, **kw)
        assert not np.array_equal(moved["pq"][b * K], ref["pq"][b * K])


def test_lazy_positions_count():
    cu = np.array([0, 3, 3, 7])
    assert list(O.lazy_positions(cu, [0, 0, 4])) == [1, 0, 4]
    assert list(O.lazy_positions(cu, [3, 0, 2])) == [3, 0, 3]

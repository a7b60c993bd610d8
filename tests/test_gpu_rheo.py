"""Parity of the CUDA RheoSampling tree expansion (spec_rheo_expand, through
the C ABI) with the oracle.

Children, proxies and true sampling probabilities are compared per frontier
row: tokens bit for bit, probabilities within 1e-5 relative, scores within
1e-5 (1 + |score|). Rows whose probe draw the oracle flags (R8: within 1e-6
of a CDF boundary) are checked for validity instead: given the GPU's probe,
the deterministic children must be the oracle's. The kept candidates must
carry the oracle's scores in the oracle's order; candidates whose scores
differ by less than the tolerance may trade places."""
import numpy as np
import pytest
import torch

import speculative_decoding_rejection_gb300 as sv
from oracle import spec_oracle as O
from speculative_decoding_rejection_gb300 import synthetic as S

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
RTOL = 1e-5


def gpu_rheo(rb, **kw):
    args = dict(K=rb.K, m=rb.m, eps=rb.eps, n_keep=rb.n_keep)
    args.update(kw)
    tok, qp, qt, sc, keep, ws = sv.spec_rheo_expand(
        rb.draft, rb.cu_frontier, rb.frontier_score, rb.temperature, rb.seed, rb.level, **args)
    return dict(child_token=tok.cpu().numpy(), child_qproxy=qp.cpu().numpy().astype(np.float64),
                child_qtrue=qt.cpu().numpy().astype(np.float64),
                child_score=sc.cpu().numpy().astype(np.float64),
                keep=keep.cpu().numpy(), status=sv.spec_get_status(ws))


def oracle_rheo(rb, trees=None, **kw):
    """The oracle on the whole batch, or on its first `trees` trees (a
    prefix keeps every frontier row's index, which keys its probe draw)."""
    args = dict(K=rb.K, m=rb.m, eps=rb.eps, n_keep=rb.n_keep)
    args.update(kw)
    cu = rb.cu_frontier.cpu().numpy()
    nb = cu.size - 1 if trees is None else trees
    F = int(cu[nb])
    return O.rheo_expand(rb.draft[:F].cpu(), cu[: nb + 1], rb.frontier_score[:F].cpu().numpy(),
                         rb.temperature[:nb].cpu().numpy(), rb.seed, rb.level, args["K"],
                         args["m"], args["eps"], args["n_keep"])


def close(g, o, tol):
    g, o = np.asarray(g, np.float64), np.asarray(o, np.float64)
    same_inf = np.isinf(g) & np.isinf(o) & (np.sign(g) == np.sign(o))
    return same_inf | (np.abs(g - o) <= tol)


def assert_rheo_parity(rb, g, r, m):
    assert g["status"] == sv.SPEC_OK
    F, K = r["child_token"].shape
    draft = rb.draft.cpu()
    flagged = set(np.nonzero(r["probe_flag"])[0].tolist())
    for f in range(F):
        if f in flagged:
            order = O.rheo_ranking_order(O.as_f64(draft[f]))
            probe = int(g["child_token"][f, m])
            assert probe in set(order.tolist())
            assert g["child_token"][f].tolist() == O.rheo_slots(order, probe, K, m), f
            continue
        assert np.array_equal(g["child_token"][f], r["child_token"][f]), (
            f, g["child_token"][f], r["child_token"][f])
        for key in ("child_qproxy", "child_qtrue"):
            ok = close(g[key][f], r[key][f], RTOL * np.abs(r[key][f]))
            assert ok.all(), (f, key, g[key][f], r[key][f])
        ok = close(g["child_score"][f], r["child_score"][f],
                   RTOL * (1 + np.abs(r["child_score"][f])))
        assert ok.all(), (f, g["child_score"][f], r["child_score"][f])
    cu = rb.cu_frontier.cpu().numpy()
    so = r["child_score"].reshape(-1)
    for b in range(r["keep"].shape[0]):
        kg, ko = g["keep"][b], r["keep"][b]
        assert np.array_equal(kg < 0, ko < 0), (b, kg, ko)
        n = int((ko >= 0).sum())
        lo, hi = int(cu[b]) * K, int(cu[b + 1]) * K
        assert ((kg[:n] >= lo) & (kg[:n] < hi)).all() and len(set(kg[:n].tolist())) == n
        rows = set((kg[:n] // K).tolist()) | set((ko[:n] // K).tolist())
        if rows & flagged:
            continue                       # the candidates themselves differ
        tol = RTOL * (1 + np.abs(so[ko[:n]]))
        ok = close(so[kg[:n]], so[ko[:n]], tol)
        assert ok.all(), (b, kg[:n], ko[:n], so[kg[:n]], so[ko[:n]])


CASES = [
    dict(B=5, W=(0, 6), V=1000, K=8, m=1, n_keep=9, dtype="f32", T=1.0, level=0),
    dict(B=6, W=(1, 5), V=4097, K=10, m=0, n_keep=12, dtype="bf16", T=("uniform", 0.0, 1.2),
         level=2),
    dict(B=4, W=3, V=20011, K=16, m=3, n_keep=40, dtype="bf16", T=0.7, level=5),
    dict(B=3, W=(2, 4), V=50, K=50, m=2, n_keep=7, dtype="f32", T=1.3, level=1),
    dict(B=2, W=4, V=77, K=7, m=6, n_keep=28, dtype="bf16", T=0.01, level=1),
    dict(B=3, W=(1, 3), V=128, K=128, m=1, n_keep=3, dtype="bf16", T=0.9, level=4),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_rheo_expand_matches_oracle(case):
    w = CASES[case]
    rb = S.make_rheo(device=DEV, input_seed=7000 + case, **w)
    assert_rheo_parity(rb, gpu_rheo(rb), oracle_rheo(rb), w["m"])


def test_rheo_ties_and_minus_inf_logits():
    rb = S.make_rheo(device=DEV, input_seed=7101, B=3, W=3, V=300, K=128, m=1, n_keep=20,
                     dtype="bf16", T=0.8, level=1)
    z = rb.draft.float()
    z = torch.round(z * 2) / 2                      # many ties
    z[:, 100:] = -float("inf")                      # 100 finite logits per row
    z[1, 3] = z[1, 4] = 5.0                         # a tie at the top
    rb.draft = z.to(torch.bfloat16).contiguous()
    g, r = gpu_rheo(rb), oracle_rheo(rb)
    assert np.isneginf(r["child_score"]).any()      # q = 0 children exist
    assert_rheo_parity(rb, g, r, 1)


def test_rheo_full_size_workload():
    """64 trees x 10 frontier rows, V = 128256, K = 10, m = 1 (the bench's
    launch). The oracle takes the first 16 trees (160 rows); every row and
    tree is checked for validity."""
    rb = S.make_rheo(device=DEV)
    g, r = gpu_rheo(rb), oracle_rheo(rb, trees=16)
    assert_rheo_parity(rb, g, r, rb.m)
    assert r["probe_flag"].sum() <= 3
    K = rb.K
    for f in range(g["child_token"].shape[0]):
        assert len(set(g["child_token"][f].tolist())) == K
    sc = g["child_score"].reshape(-1)
    cu = rb.cu_frontier.cpu().numpy()
    for b in range(rb.B):
        kb = g["keep"][b]
        assert ((kb >= cu[b] * K) & (kb < cu[b + 1] * K)).all()
        assert (np.diff(sc[kb]) <= 0).all()


def test_rheo_largest_tree_and_empty_trees():
    n = sv.SPEC_RHEO_MAX_CANDIDATES // 8
    rb = S.make_rheo(device=DEV, input_seed=7202, B=1, W=n, V=256, K=8, m=1, n_keep=300,
                     dtype="bf16", T=1.0, level=2)
    assert_rheo_parity(rb, gpu_rheo(rb), oracle_rheo(rb), 1)
    rb = S.make_rheo(device=DEV, input_seed=7203, B=4, W=0, V=256, K=8, m=1, n_keep=5,
                     dtype="bf16", T=1.0, level=0)
    g = gpu_rheo(rb)
    assert g["status"] == sv.SPEC_OK and (g["keep"] == -1).all()


def test_rheo_is_deterministic_and_level_keys_the_probe():
    rb = S.make_rheo(device=DEV, input_seed=7204, B=8, W=4, V=5000, K=6, m=1, n_keep=6,
                     dtype="bf16", T=1.5, level=3)
    a, b = gpu_rheo(rb), gpu_rheo(rb)
    for k in ("child_token", "child_qproxy", "child_qtrue", "child_score", "keep"):
        assert np.array_equal(a[k], b[k]), k
    rb.level = 4
    c = gpu_rheo(rb)
    assert not np.array_equal(a["child_token"][:, 1], c["child_token"][:, 1])


def test_rheo_invalid_inputs_set_the_status():
    rb = S.make_rheo(device=DEV, input_seed=7205, B=3, W=2, V=256, K=4, m=1, n_keep=4,
                     dtype="bf16", T=1.0, level=1)
    bad = rb.frontier_score.clone()
    bad[2] = float("nan")
    tok, _, _, sc, keep, ws = sv.spec_rheo_expand(rb.draft, rb.cu_frontier, bad,
                                                  rb.temperature, 1, 1, K=4, m=1, n_keep=4)
    assert sv.spec_get_status(ws) == sv.SPEC_ERR_INVALID_ARG
    assert (keep.cpu() == -1).all()
    temp = rb.temperature.clone()
    temp[1] = -1.0
    *_, ws = sv.spec_rheo_expand(rb.draft, rb.cu_frontier, rb.frontier_score, temp, 1, 1,
                                 K=4, m=1, n_keep=4)
    assert sv.spec_get_status(ws) == sv.SPEC_ERR_INVALID_ARG
    cu = rb.cu_frontier.clone()
    cu[1], cu[2] = 4, 2                               # not monotone
    *_, ws = sv.spec_rheo_expand(rb.draft, cu, rb.frontier_score, rb.temperature, 1, 1,
                                 K=4, m=1, n_keep=4)
    assert sv.spec_get_status(ws) == sv.SPEC_ERR_INVALID_ARG
    n = sv.SPEC_RHEO_MAX_CANDIDATES // 4 + 1          # one tree over the limit
    big = S.make_rheo(device=DEV, input_seed=7206, B=1, W=n, V=128, K=4, m=1, n_keep=4,
                      dtype="bf16", T=1.0, level=1)
    *_, keep, ws = sv.spec_rheo_expand(big.draft, big.cu_frontier, big.frontier_score,
                                       big.temperature, 1, 1, K=4, m=1, n_keep=4)
    assert sv.spec_get_status(ws) == sv.SPEC_ERR_UNSUPPORTED
    # the workspace stays usable: a valid call afterwards is clean
    g = gpu_rheo(rb)
    assert g["status"] == sv.SPEC_OK


# ------------------------------ construction, then verification of the trees
def built_trees(tokens, K, m):
    """Depth-1 trees from one frontier row per tree: the probe (slot m)
    first, then the other slots in order, those flagged as point masses."""
    B = tokens.shape[0]
    order = [m] + [s for s in range(K) if s != m]
    node_token = np.full((B, K + 1), -1, dtype=np.int32)
    node_token[:, 1:] = tokens[:, order]
    parent = np.tile(np.array([-1] + [0] * K, dtype=np.int32), B)
    fixed = np.tile(np.array([0, 0] + [1] * (K - 1), dtype=np.int32), B)
    return node_token.reshape(-1), parent, fixed


def test_built_trees_verify_like_the_oracle():
    """Construction then verification, each side on its own outputs: the
    GPU verifies the trees the GPU built, the oracle the trees the oracle
    built; trees whose probe draw the oracle flags are skipped."""
    K, m, V, B = 5, 1, 3000, 12
    rb = S.make_rheo(device=DEV, input_seed=7301, B=B, W=1, V=V, K=K, m=m, n_keep=K,
                     dtype="bf16", T=0.9, level=0)
    g, r = gpu_rheo(rb), oracle_rheo(rb)
    gen = torch.Generator(device=DEV).manual_seed(7302)
    target = (2.0 * torch.randn(B * (K + 1), V, generator=gen, device=DEV)).to(torch.bfloat16)
    # each tree's root draft row is its frontier row; leaves' draft rows are unused
    draft = torch.zeros(B * (K + 1), V, dtype=torch.bfloat16, device=DEV)
    draft[0::K + 1] = rb.draft
    cu = np.arange(0, B * (K + 1) + 1, K + 1, dtype=np.int32)
    nt_g, par, fx = built_trees(g["child_token"], K, m)
    nt_o, _, _ = built_trees(r["child_token"].astype(np.int32), K, m)
    seed = 0x5EED
    tok, acc, path, ws = sv.spec_verify_tree(
        target, draft, torch.from_numpy(nt_g).to(DEV), torch.from_numpy(par).to(DEV),
        torch.from_numpy(cu).to(DEV), rb.temperature, seed, max_depth=1, max_branch=K,
        node_fixed=torch.from_numpy(fx).to(DEV))
    assert sv.spec_get_status(ws) == sv.SPEC_OK
    ro = O.verify_tree(target.cpu(), draft.cpu(), nt_o, par, cu, rb.temperature.cpu().numpy(),
                       seed, 1, node_fixed=fx)
    tok, acc = tok.cpu().numpy(), acc.cpu().numpy()
    compared = 0
    for b in range(B):
        if r["probe_flag"][b] or ro["flag_slot"][b] >= 0:
            continue
        assert np.array_equal(tok[b], ro["tokens"][b]) and acc[b] == ro["accepted"][b], b
        compared += 1
    assert compared >= B - 2


def test_built_and_verified_node_emits_the_target_law():
    """"RheoSampling 2026" §6 on the GPU: 8192 copies of one built node
    (probe drawn from q~, three point-mass leads, probe verified first);
    the first emitted token follows p = softmax(z_t / T) (chi-square)."""
    from scipy import special, stats
    B, V, K, m, T = 8192, 48, 4, 1, 0.9
    rng = np.random.default_rng(5)
    zd = rng.standard_normal(V) * 1.5
    zt = zd + rng.standard_normal(V)
    draft_rows = torch.tensor(np.tile(zd, (B, 1)), dtype=torch.float32, device=DEV)
    cu_f = torch.arange(0, B + 1, dtype=torch.int32, device=DEV)
    temp = torch.full((B,), T, dtype=torch.float32, device=DEV)
    tok, _, _, _, _, ws = sv.spec_rheo_expand(draft_rows, cu_f, torch.zeros(B, device=DEV), temp,
                                              11, 0, K=K, m=m, n_keep=0)
    assert sv.spec_get_status(ws) == sv.SPEC_OK
    nt, par, fx = built_trees(tok.cpu().numpy(), K, m)
    target = torch.tensor(np.tile(zt, (B * (K + 1), 1)), dtype=torch.float32, device=DEV)
    draft = torch.tensor(np.tile(zd, (B * (K + 1), 1)), dtype=torch.float32, device=DEV)
    cu = torch.arange(0, B * (K + 1) + 1, K + 1, dtype=torch.int32, device=DEV)
    out, acc, _, ws2 = sv.spec_verify_tree(
        target, draft, torch.from_numpy(nt).to(DEV), torch.from_numpy(par).to(DEV), cu, temp, 12,
        max_depth=1, max_branch=K, node_fixed=torch.from_numpy(fx).to(DEV))
    assert sv.spec_get_status(ws2) == sv.SPEC_OK
    first = out[:, 0].cpu().numpy()
    p = special.softmax(zt / T)
    obs = np.bincount(first, minlength=V).astype(np.float64)
    exp = p * B
    big = exp >= 5
    chi = np.sum((obs[big] - exp[big]) ** 2 / exp[big])
    rest_o, rest_e = obs[~big].sum(), exp[~big].sum()
    dof = int(big.sum()) - 1
    if rest_e > 0:
        chi += (rest_o - rest_e) ** 2 / rest_e
        dof += 1
    assert stats.chi2.sf(chi, dof) > 1e-4, (chi, dof)
    assert (acc.cpu().numpy() == 1).mean() > 0.3      # the built children are accepted often

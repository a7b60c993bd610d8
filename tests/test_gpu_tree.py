"""Parity of the CUDA tree verifier (RRSw, through the C ABI) with the oracle."""
import numpy as np
import pytest
import torch

import speculative_decoding_rejection_gb300 as sv
from oracle import spec_oracle as O
from speculative_decoding_rejection_gb300 import synthetic as S

from parity import probs_from_logits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def gpu_tree(tb, draft=None, draft_kind=sv.SPEC_DRAFT_LOGITS, node_fixed=None):
    draft = tb.draft if draft is None else draft
    tok, acc, path, ws = sv.spec_verify_tree(
        tb.target, draft, tb.node_token, tb.parent, tb.cu_nodes, tb.temperature, tb.seed,
        max_depth=tb.max_depth, max_branch=tb.max_branch, draft_kind=draft_kind,
        node_fixed=node_fixed)
    return dict(tokens=tok.cpu().numpy(), accepted=acc.cpu().numpy(), path=path.cpu().numpy(),
                status=sv.spec_get_status(ws))


def oracle_tree(tb, draft=None, draft_kind=sv.SPEC_DRAFT_LOGITS, requests=None,
                node_fixed=None):
    draft = tb.draft if draft is None else draft
    host = (lambda t: t.cpu()) if requests is None else (lambda t: t)
    return O.verify_tree(host(tb.target), host(draft), tb.node_token.cpu().numpy(),
                         tb.parent.cpu().numpy(), tb.cu_nodes.cpu().numpy(),
                         tb.temperature.cpu().numpy(), tb.seed, tb.max_depth,
                         requests=requests, draft_kind=draft_kind,
                         node_fixed=None if node_fixed is None else node_fixed.cpu().numpy())


def assert_tree_parity(g, r, min_compared):
    n_full = 0
    for j, b in enumerate(r["requests"]):
        fs = int(r["flag_slot"][j])
        if fs < 0:
            assert np.array_equal(g["tokens"][b], r["tokens"][j]), (b, g["tokens"][b], r["tokens"][j])
            assert g["accepted"][b] == r["accepted"][j]
            assert np.array_equal(g["path"][b], r["path"][j])
            n_full += 1
        else:
            assert np.array_equal(g["tokens"][b][:fs], r["tokens"][j][:fs])
    assert n_full >= min_compared
    return n_full


@pytest.mark.parametrize("T,V,dtype", [(0.8, 5003, "bf16"), (1.3, 4096, "f32"),
                                       (0.0, 3001, "bf16"), (0.3, 20000, "bf16")])
def test_random_trees_small_vocab(T, V, dtype):
    tb = S.make_tree(4, device=DEV, B=12, V=V, dtype=dtype, T=T, input_seed=V)
    g = gpu_tree(tb)
    assert g["status"] == sv.SPEC_OK
    r = oracle_tree(tb)
    assert_tree_parity(g, r, min_compared=10)
    assert g["accepted"].max() >= 1


def test_wide_shallow_trees_many_rejections():
    tb = S.make_tree(4, device=DEV, B=16, N=9, depth=1, branch=8, V=64, sigma=2.5, T=1.0,
                     input_seed=3)
    g = gpu_tree(tb)
    r = oracle_tree(tb)
    assert_tree_parity(g, r, min_compared=14)
    assert (g["accepted"] == 0).any()        # some nodes reject all 8 children


def test_tree_draft_given_as_probabilities():
    tb = S.make_tree(4, device=DEV, B=10, V=3000, input_seed=17)
    ones = torch.arange(0, tb.target.shape[0] + 1, dtype=torch.int32, device=DEV)
    T = tb.temperature.repeat_interleave(torch.diff(tb.cu_nodes.long()))
    probs = probs_from_logits(tb.draft, ones, T)
    g = gpu_tree(tb, draft=probs, draft_kind=sv.SPEC_DRAFT_PROBS)
    r = oracle_tree(tb, draft=probs, draft_kind=sv.SPEC_DRAFT_PROBS)
    assert_tree_parity(g, r, min_compared=8)


@pytest.mark.parametrize("T", [0.9, 0.0])
def test_chain_tree_equals_linear_verifier_on_the_gpu(T):
    lb = S.make_linear(1, device=DEV, B=24, K=5, V=4000, dtype="bf16", T=T, input_seed=41)
    B, K, V = lb.B, lb.max_k, lb.V
    tgt = lb.target.view(B, K + 1, V)
    drf = torch.cat([lb.draft.view(B, K, V), torch.zeros(B, 1, V, dtype=lb.draft.dtype,
                                                         device=DEV)], 1)
    node_tok = torch.cat([torch.full((B, 1), -1, dtype=torch.int32, device=DEV),
                          lb.draft_tokens.view(B, K)], 1).reshape(-1).contiguous()
    parent = torch.arange(-1, K, dtype=torch.int32, device=DEV).repeat(B).contiguous()
    cu = torch.arange(0, B * (K + 1) + 1, K + 1, dtype=torch.int32, device=DEV)
    tok_t, acc_t, _, ws = sv.spec_verify_tree(
        tgt.reshape(-1, V).contiguous(), drf.reshape(-1, V).contiguous(), node_tok, parent, cu,
        lb.temperature, lb.seed, max_depth=K, max_branch=1)
    assert sv.spec_get_status(ws) == sv.SPEC_OK
    tok_l, acc_l, _, _ = sv.spec_verify_linear(lb.target, lb.draft, lb.draft_tokens,
                                               lb.cu_draft, lb.temperature, lb.seed, max_k=K)
    assert torch.equal(acc_t, acc_l)
    assert torch.equal(tok_t, tok_l)


def test_full_size_tree_workload_whole_batch():
    """Every tree of the full-size workload against the oracle: tokens,
    accepted depth and path bit for bit up to the first flagged draw."""
    tb = S.make_tree(4, device=DEV)
    g = gpu_tree(tb)
    assert g["status"] == sv.SPEC_OK
    r = oracle_tree(tb)
    assert len(r["requests"]) == tb.B
    assert_tree_parity(g, r, min_compared=int((r["flag_slot"] < 0).sum()))
    assert np.all((g["accepted"] >= 0) & (g["accepted"] <= tb.max_depth))


def test_malformed_tree_sets_the_status_word():
    tb = S.make_tree(4, device=DEV, B=3, V=500, input_seed=5)
    bad = tb.parent.clone()
    bad[64 + 10] = 12                          # parent after its child
    tok, acc, _, ws = sv.spec_verify_tree(tb.target, tb.draft, tb.node_token, bad, tb.cu_nodes,
                                          tb.temperature, 1, max_depth=6, max_branch=4)
    assert sv.spec_get_status(ws) == sv.SPEC_ERR_INVALID_ARG
    assert torch.all(acc == -1)
    tok, acc, _, ws = sv.spec_verify_tree(tb.target, tb.draft, tb.node_token, tb.parent,
                                          tb.cu_nodes, tb.temperature, 1, max_depth=3,
                                          max_branch=4)
    assert sv.spec_get_status(ws) == sv.SPEC_ERR_INVALID_ARG    # deeper than max_depth


def test_repeated_drawn_sibling_sets_the_status_word():
    """Drawn siblings carry distinct tokens (they were drawn without
    replacement): a repeat is invalid input; a point-mass child may repeat a
    drawn sibling's token."""
    tb = S.make_tree(4, device=DEV, B=3, V=500, input_seed=5)
    par = tb.parent.cpu().numpy()[:64]
    kids = {}
    for c in range(1, 64):
        kids.setdefault(int(par[c]), []).append(c)
    first, second = next(v for v in kids.values() if len(v) >= 2)[:2]
    tok = tb.node_token.clone()
    tok[second] = tok[first]
    _, acc, _, ws = sv.spec_verify_tree(tb.target, tb.draft, tok, tb.parent, tb.cu_nodes,
                                        tb.temperature, 1, max_depth=6, max_branch=4)
    assert sv.spec_get_status(ws) == sv.SPEC_ERR_INVALID_ARG
    assert torch.all(acc == -1)
    nf = torch.zeros_like(tok)
    nf[second] = 1                             # the repeat is a point mass: allowed
    _, acc, _, ws = sv.spec_verify_tree(tb.target, tb.draft, tok, tb.parent, tb.cu_nodes,
                                        tb.temperature, 1, max_depth=6, max_branch=4,
                                        node_fixed=nf)
    assert sv.spec_get_status(ws) == sv.SPEC_OK
    assert torch.all(acc >= 0)


def test_walk_reads_only_the_rows_of_visited_nodes():
    """The rows of every node off the walked path are set to -inf (no mass):
    the outputs stay those of the clean call and no error is reported, since
    the walk reads only the root's and the accepted path's rows."""
    tb = S.make_tree(4, device=DEV, B=12, V=8192, input_seed=44)
    clean = gpu_tree(tb)
    assert clean["status"] == sv.SPEC_OK
    cu = tb.cu_nodes.cpu().numpy()
    keep = torch.zeros(tb.target.shape[0], dtype=torch.bool)
    for b in range(tb.B):
        nodes = [0] + [int(x) for x in clean["path"][b][:clean["accepted"][b]]]
        keep[[int(cu[b]) + v for v in nodes]] = True
    assert int((~keep).sum()) > tb.B * 30
    t2, d2 = tb.target.clone(), tb.draft.clone()
    gone = (~keep).nonzero().squeeze(1).to(DEV)
    t2[gone] = float("-inf")
    d2[gone] = float("-inf")
    tb2 = S.TreeBatch(**{**tb.__dict__, "target": t2, "draft": d2})
    g = gpu_tree(tb2)
    assert g["status"] == sv.SPEC_OK
    assert np.array_equal(g["tokens"], clean["tokens"])
    assert np.array_equal(g["accepted"], clean["accepted"])
    assert np.array_equal(g["path"], clean["path"])


# ------------------------------------------- point-mass children (ext entry)
def random_fixed(tb, frac, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.rand(tb.node_token.numel(), generator=g) < frac).to(torch.int32).to(DEV)


@pytest.mark.parametrize("T,V,frac", [(0.8, 5003, 0.3), (1.2, 4096, 0.6), (0.0, 3001, 0.5),
                                      (0.9, 64, 0.5), (0.7, 20000, 1.0)])
def test_point_mass_children_match_oracle(T, V, frac):
    tb = S.make_tree(4, device=DEV, B=12, V=V, dtype="bf16", T=T, input_seed=V + 1)
    nf = random_fixed(tb, frac, V)
    g = gpu_tree(tb, node_fixed=nf)
    assert g["status"] == sv.SPEC_OK
    assert_tree_parity(g, oracle_tree(tb, node_fixed=nf), min_compared=10)


def test_rheosampling_shaped_nodes_probe_first():
    """Depth-1 trees shaped like a built RheoSampling node: child 1 is drawn
    (the probe), children 2..K are the best draft tokens other than it,
    flagged as point masses; many rejections and final draws."""
    K = 6
    tb = S.make_tree(4, device=DEV, B=16, N=K + 1, depth=1, branch=K, V=2048, sigma=1.5,
                     T=1.0, input_seed=91)
    tok = tb.node_token.cpu().clone()
    drf = tb.draft.float().cpu()
    fixed = torch.zeros_like(tok)
    for b in range(tb.B):
        base = b * (K + 1)
        probe = int(tok[base + 1])
        order = torch.argsort(-drf[base], stable=True).tolist()   # ties to the lower id
        best = [x for x in order if x != probe][:K - 1]
        tok[base + 2:base + K + 1] = torch.tensor(best, dtype=tok.dtype)
        fixed[base + 2:base + K + 1] = 1
    tb2 = S.TreeBatch(**{**tb.__dict__, "node_token": tok.to(DEV).contiguous()})
    nf = fixed.to(torch.int32).to(DEV)
    g = gpu_tree(tb2, node_fixed=nf)
    assert g["status"] == sv.SPEC_OK
    assert_tree_parity(g, oracle_tree(tb2, node_fixed=nf), min_compared=14)


def test_full_size_tree_workload_with_point_mass_children():
    tb = S.make_tree(4, device=DEV)
    nf = random_fixed(tb, 0.5, 4)
    g = gpu_tree(tb, node_fixed=nf)
    assert g["status"] == sv.SPEC_OK
    r = oracle_tree(tb, node_fixed=nf)
    assert_tree_parity(g, r, min_compared=int((r["flag_slot"] < 0).sum()))

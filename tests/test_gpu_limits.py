"""The verifier at its documented limits, against the oracle: 256 drafts per
request (SPEC_MAX_K), a vocabulary of 2^24 (SPEC_MAX_V), a 4096-node tree
(SPEC_MAX_TREE_NODES), a chain of depth 64 (SPEC_MAX_TREE_DEPTH) and a node
with 64 children (SPEC_MAX_TREE_BRANCH)."""
import numpy as np
import pytest
import torch

import speculative_decoding_rejection_gb300 as sv
from oracle import spec_oracle as O
from speculative_decoding_rejection_gb300 import synthetic as S

from parity import assert_linear_parity, gpu_linear, oracle_linear

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
# the limits of include/specverify.h
MAX_K, MAX_DEPTH, MAX_BRANCH, MAX_NODES = 256, 64, 64, 4096


@pytest.mark.parametrize("V,limit", [(512, 32 << 20), (2048, 0)])
def test_linear_at_the_maximum_draft_count(V, limit):
    old = sv.spec_set_fused_limit(limit)
    try:
        lb = S.make_linear(1, device=DEV, B=3, K=MAX_K, V=V, dtype="bf16", sigma=0.05,
                           T=[1.0, 0.0, 0.7], input_seed=6000 + V)
        assert lb.max_k == MAX_K
        g = gpu_linear(lb)
        assert g["status"] == sv.SPEC_OK
        r = oracle_linear(lb)
        assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=2)
        assert g["accepted"].max() > 20          # long accepted prefixes
    finally:
        sv.spec_set_fused_limit(old)


def test_linear_at_the_maximum_vocabulary():
    """At V = 2^24 a token's probability (~6e-8) is far below the 1e-6
    margin of R8, so the final draw is nearly always flagged: the accepted
    drafts and counts are compared exactly, the final token checked to be a
    token of the vocabulary."""
    V = 1 << 24
    lb = S.make_linear(1, device=DEV, B=2, K=2, V=V, dtype="bf16", sigma=0.5, T=[1.0, 0.0],
                       input_seed=6100)
    g = gpu_linear(lb)
    assert g["status"] == sv.SPEC_OK
    r = oracle_linear(lb)
    assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=0)
    for j in range(lb.B):
        n = int(r["accepted"][j])
        if int(r["flag_slot"][j]) in (-1, n):     # only the final draw may be flagged
            assert g["accepted"][j] == n
            assert np.array_equal(g["tokens"][j][:n], r["tokens"][j][:n])
            assert 0 <= g["tokens"][j][n] < V
    assert g["tokens"][1][int(g["accepted"][1])] == r["tokens"][1][int(r["accepted"][1])]


def _tree_batch(target, draft, tokens, parent, T, max_depth, max_branch, seed):
    n = len(parent)
    return S.TreeBatch(target=target, draft=draft,
                       node_token=torch.tensor(tokens, dtype=torch.int32, device=DEV),
                       parent=torch.tensor(parent, dtype=torch.int32, device=DEV),
                       cu_nodes=torch.tensor([0, n], dtype=torch.int32, device=DEV),
                       temperature=torch.tensor([T], device=DEV), max_depth=max_depth,
                       max_branch=max_branch, seed=seed)


def _check_tree(tb):
    tok, acc, path, ws = sv.spec_verify_tree(
        tb.target, tb.draft, tb.node_token, tb.parent, tb.cu_nodes, tb.temperature, tb.seed,
        max_depth=tb.max_depth, max_branch=tb.max_branch)
    assert sv.spec_get_status(ws) == sv.SPEC_OK
    r = O.verify_tree(tb.target.cpu(), tb.draft.cpu(), tb.node_token.cpu().numpy(),
                      tb.parent.cpu().numpy(), tb.cu_nodes.cpu().numpy(),
                      tb.temperature.cpu().numpy(), tb.seed, tb.max_depth)
    fs = int(r["flag_slot"][0])
    tok, acc = tok.cpu().numpy(), acc.cpu().numpy()
    if fs < 0:
        assert np.array_equal(tok[0], r["tokens"][0]) and acc[0] == r["accepted"][0]
    else:
        assert np.array_equal(tok[0, :fs], r["tokens"][0, :fs])
    return acc[0]


def test_tree_chain_at_the_maximum_depth():
    """A chain of 64 drafts whose tokens are the target's argmax at a low
    temperature, so the walk reaches the deepest node."""
    D, V = MAX_DEPTH, 1024
    g = torch.Generator(device=DEV).manual_seed(5)
    zt = (2.0 * torch.randn(D + 1, V, generator=g, device=DEV))
    zt[:, 7] += 12.0                                  # a dominant token at every node
    zd = zt + 0.1 * torch.randn(D + 1, V, generator=g, device=DEV)
    tokens = [-1] + [7] * D
    parent = [-1] + list(range(D))
    tb = _tree_batch(zt.to(torch.bfloat16), zd.to(torch.bfloat16), tokens, parent, 0.8, D, 1,
                     77)
    assert _check_tree(tb) >= D - 2


def test_tree_node_with_the_maximum_branching():
    """The root has 64 children drawn without replacement from its draft law
    (Gumbel-top-64); the walk tests them in order."""
    Bn, V = MAX_BRANCH, 4096
    g = torch.Generator(device=DEV).manual_seed(6)
    zt = 2.0 * torch.randn(Bn + 1, V, generator=g, device=DEV)
    zd = zt + 2.5 * torch.randn(Bn + 1, V, generator=g, device=DEV)   # poor draft: many rejections
    gum = -torch.log(-torch.log(torch.rand(V, generator=g, device=DEV).clamp(1e-12, 1 - 1e-7)))
    order = torch.argsort(zd[0] / 1.0 + gum, descending=True)[:Bn].tolist()
    tokens = [-1] + order
    parent = [-1] + [0] * Bn
    tb = _tree_batch(zt.to(torch.bfloat16), zd.to(torch.bfloat16), tokens, parent, 1.0, 1, Bn,
                     78)
    _check_tree(tb)


def test_tree_with_the_maximum_node_count():
    tb = S.make_tree(4, device=DEV, B=1, N=MAX_NODES, depth=12, branch=8, V=512, dtype="bf16",
                     T=0.9, input_seed=79)
    _check_tree(tb)

"""The seeded workload generator produces what its recipe states."""
import numpy as np
import torch

from speculative_decoding_rejection_gb300 import synthetic as S


def test_linear_shapes_and_determinism():
    a = S.make_linear(2, B=10, V=500)
    b = S.make_linear(2, B=10, V=500)
    assert torch.equal(a.target, b.target) and torch.equal(a.draft_tokens, b.draft_tokens)
    K = torch.diff(a.cu_draft.long())
    assert int(K.min()) >= 1 and int(K.max()) <= 5
    assert a.target.shape == (int(a.cu_draft[-1]) + 10, 500)
    assert a.draft.shape == (int(a.cu_draft[-1]), 500)
    assert a.target.dtype == torch.bfloat16
    assert a.max_k == int(K.max())


def test_greedy_drafts_are_draft_argmax_and_top128_drafts_stay_in_top128():
    g = S.make_linear(2, B=8, V=300, T=[0.0] * 8)
    assert torch.equal(g.draft_tokens.long(), torch.argmax(g.draft.float(), 1))
    t = S.make_linear(3, B=6, K=3, V=2000)
    top = torch.topk(t.draft.float(), 128, dim=1).indices
    assert bool((top == t.draft_tokens.long()[:, None]).any(1).all())


def test_config5_temperatures_span_greedy_and_sampling():
    lb = S.make_linear(5, B=64, V=256)
    T = lb.temperature.numpy()
    assert T.min() >= 0.0 and T.max() <= 1.2
    assert (T < 0.05).any() or len(T) < 30


def test_tree_structure():
    tb = S.make_tree(4, B=5, V=400)
    par = tb.parent.numpy().reshape(5, 64)
    tok = tb.node_token.numpy().reshape(5, 64)
    for b in range(5):
        depth = np.zeros(64, int)
        for c in range(1, 64):
            assert 0 <= par[b, c] < c
            depth[c] = depth[par[b, c]] + 1
        assert depth.max() <= 6 and par[b, 0] == -1
        for v in range(64):
            kids = np.nonzero(par[b] == v)[0]
            assert len(kids) <= 4
            assert len(set(tok[b, kids])) == len(kids)   # without replacement

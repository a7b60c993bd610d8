"""The verifier's calls inside CUDA graphs: a captured call replays with the
same results as the eager call, on inputs refreshed in place between
replays (the way a decode loop reuses its buffers)."""
import time

import pytest
import torch

import speculative_decoding_rejection_gb300 as sv
from speculative_decoding_rejection_gb300 import synthetic as S

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _linear_graph_case(cfg, **over):
    lb = S.make_linear(cfg, device=DEV, **over)
    ws = torch.empty(sv.spec_verify_linear_workspace(lb.B, lb.max_k, lb.V), dtype=torch.uint8,
                     device=DEV)
    out = (torch.empty(lb.B, lb.max_k + 1, dtype=torch.int32, device=DEV),
           torch.empty(lb.B, dtype=torch.int32, device=DEV),
           torch.empty(lb.draft_tokens.numel(), 2, dtype=torch.float32, device=DEV))
    return lb, ws, out


def _call(lb, ws, out):
    sv.spec_verify_linear(lb.target, lb.draft, lb.draft_tokens, lb.cu_draft, lb.temperature,
                          lb.seed, max_k=lb.max_k, want_pq=True, workspace=ws, out=out)


@pytest.mark.parametrize("cfg,over", [(1, {}), (2, {}), (5, dict(B=64))])
def test_linear_call_replays_in_a_cuda_graph(cfg, over):
    lb, ws, out = _linear_graph_case(cfg, **over)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):          # warm-up outside the capture
        _call(lb, ws, out)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _call(lb, ws, out)
    # new inputs written into the captured buffers in place, then replay
    gen = torch.Generator(device=DEV).manual_seed(4242)
    lb.target.add_(torch.randn(lb.target.shape, generator=gen, device=DEV).to(lb.target.dtype))
    lb.draft.add_(torch.randn(lb.draft.shape, generator=gen, device=DEV).to(lb.draft.dtype))
    lb.temperature.copy_(torch.rand(lb.B, generator=gen, device=DEV) * 1.2)
    g.replay()
    torch.cuda.synchronize()
    assert sv.spec_get_status(ws) == sv.SPEC_OK
    got = [t.clone() for t in out]
    ref = sv.spec_verify_linear(lb.target, lb.draft, lb.draft_tokens, lb.cu_draft,
                                lb.temperature, lb.seed, max_k=lb.max_k, want_pq=True)
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
    assert torch.equal(got[2], ref[2])
    # launch cost: eager calls against replays of the same work
    n = 200
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n):
        _call(lb, ws, out)
    torch.cuda.synchronize()
    t_eager = (time.perf_counter() - t0) / n
    t0 = time.perf_counter()
    for _ in range(n):
        g.replay()
    torch.cuda.synchronize()
    t_graph = (time.perf_counter() - t0) / n
    print(f"cfg {cfg}: eager {t_eager * 1e6:.1f} us, graph replay {t_graph * 1e6:.1f} us per call")


def test_tree_and_construction_calls_replay_in_a_cuda_graph():
    tb = S.make_tree(4, device=DEV, B=6, V=4096, input_seed=5)
    rb = S.make_rheo(device=DEV, input_seed=6, B=6, W=3, V=4096, K=6, m=1, n_keep=6)
    n_nodes = tb.target.shape[0]
    wst = torch.empty(sv.spec_verify_tree_workspace(tb.B, n_nodes, tb.V, tb.max_depth,
                                                    tb.max_branch), dtype=torch.uint8,
                      device=DEV)
    tout = (torch.empty(tb.B, tb.max_depth + 1, dtype=torch.int32, device=DEV),
            torch.empty(tb.B, dtype=torch.int32, device=DEV),
            torch.empty(tb.B, tb.max_depth + 1, dtype=torch.int32, device=DEV))
    F = rb.draft.shape[0]
    wsr = torch.empty(sv.spec_rheo_expand_workspace(F, rb.V), dtype=torch.uint8, device=DEV)
    rout = (torch.empty(F, rb.K, dtype=torch.int32, device=DEV),
            torch.empty(F, rb.K, dtype=torch.float32, device=DEV),
            torch.empty(F, rb.K, dtype=torch.float32, device=DEV),
            torch.empty(F, rb.K, dtype=torch.float32, device=DEV),
            torch.empty(rb.B, rb.n_keep, dtype=torch.int32, device=DEV))

    def calls():
        sv.spec_verify_tree(tb.target, tb.draft, tb.node_token, tb.parent, tb.cu_nodes,
                            tb.temperature, tb.seed, max_depth=tb.max_depth,
                            max_branch=tb.max_branch, workspace=wst, out=tout)
        sv.spec_rheo_expand(rb.draft, rb.cu_frontier, rb.frontier_score, rb.temperature,
                            rb.seed, rb.level, K=rb.K, m=rb.m, n_keep=rb.n_keep,
                            workspace=wsr, out=rout)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        calls()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [t.clone() for t in tout + rout]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        calls()
    for t in tout + rout:
        t.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    assert sv.spec_get_status(wst) == sv.SPEC_OK and sv.spec_get_status(wsr) == sv.SPEC_OK
    for a, b in zip(eager, tout + rout):
        assert torch.equal(a, b)


@pytest.mark.parametrize("cfg,over", [(1, {}), (2, dict(B=16))])
def test_device_seed_gives_new_draws_on_each_replay(cfg, over):
    """With the seed in device memory, one captured call replays with the
    draws of whatever seed was last written there, equal to eager calls
    with that seed."""
    lb, ws, out = _linear_graph_case(cfg, **over)
    seed_dev = torch.zeros(1, dtype=torch.int64, device=DEV)

    def call():
        sv.spec_verify_linear_ext(lb.target, lb.draft, lb.draft_tokens, lb.cu_draft,
                                  lb.temperature, 0, max_k=lb.max_k, want_pq=True,
                                  seed_dev=seed_dev, workspace=ws, out=out + (None, None))

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    outs = []
    for seed in (11, 12345, 2 ** 40 + 7):
        seed_dev.fill_(seed)
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in out]
        ref = sv.spec_verify_linear(lb.target, lb.draft, lb.draft_tokens, lb.cu_draft,
                                    lb.temperature, seed, max_k=lb.max_k, want_pq=True)
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1]), seed
        outs.append(got[0])
    assert not (torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2]))


def test_tree_device_seed():
    tb = S.make_tree(4, device=DEV, B=8, V=3000, input_seed=31)
    seed_dev = torch.tensor([tb.seed + 5], dtype=torch.int64, device=DEV)
    a = sv.spec_verify_tree(tb.target, tb.draft, tb.node_token, tb.parent, tb.cu_nodes,
                            tb.temperature, 0, max_depth=tb.max_depth,
                            max_branch=tb.max_branch, seed_dev=seed_dev)
    b = sv.spec_verify_tree(tb.target, tb.draft, tb.node_token, tb.parent, tb.cu_nodes,
                            tb.temperature, tb.seed + 5, max_depth=tb.max_depth,
                            max_branch=tb.max_branch)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])

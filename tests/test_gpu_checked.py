"""The bounds-checked build (libspecverify_checked.so, built with
SPEC_CHECKED) on every entry point, against the oracle.

In that build every global access of the kernels is checked against the
byte ranges of the call's own buffers (inputs, outputs, workspace); an
access outside them is skipped and reported in the status word as
SPEC_ERR_BOUNDS. Each case below runs one schedule of one entry point on a
small input (V <= 16 where the schedule takes such rows, a few thousand
logits where it needs longer ones), checks the results against the oracle,
and requires the status word to stay SPEC_OK: no kernel index left its
buffers. The checker's self-test shows that an access outside the
registered ranges is reported."""
import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_rejection_gb300 as sv
from oracle import spec_oracle as O
from speculative_decoding_rejection_gb300 import synthetic as S

from parity import (assert_linear_parity, assert_probs_close, gpu_linear, oracle_linear,
                    probs_from_logits)
from test_gpu_rheo import assert_rheo_parity, gpu_rheo, oracle_rheo
from test_gpu_tree import assert_tree_parity, gpu_tree, oracle_tree

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(autouse=True)
def checked_library():
    sv.use_checked_library(True)
    old = sv.spec_set_fused_limit(32 << 20)
    yield
    sv.spec_set_fused_limit(old)
    sv.use_checked_library(False)


def test_checker_reports_an_access_outside_the_call():
    ws = sv.spec_check_selftest()
    assert sv.spec_get_status(ws) == sv.SPEC_ERR_BOUNDS
    assert int(ws[4:8].view(torch.int32).item()) > 0   # the detail word: a source line


def test_product_library_has_no_checker():
    sv.use_checked_library(False)
    with pytest.raises(sv.SpecError) as e:
        sv.spec_check_selftest()
    assert e.value.code == sv.SPEC_ERR_UNSUPPORTED


def _lazy_parity(g, ref, lb):
    lz = O.lazy_view(ref, lb.cu_draft.cpu().numpy())
    return assert_linear_parity(g, lz, lb.cu_draft.cpu(),
                                min_compared=int((ref["flag_slot"] < 0).sum()))


# (name, batch overrides, gpu_linear keywords, fused limit, lazy outputs)
LINEAR_CASES = [
    ("fused", dict(cfg=1, B=4, K=3, V=16, dtype="f32"), {}, 32 << 20, False),
    ("eager", dict(cfg=1, B=4, K=3, V=16, dtype="bf16"), {}, 0, False),
    ("eager-greedy-rule", dict(cfg=1, B=3, K=4, V=16, dtype="bf16"),
     dict(rule=sv.SPEC_RULE_GREEDY), 0, False),
    ("streaming", dict(cfg=1, B=4, K=3, V=16, dtype="bf16"), dict(plain=True), 0, True),
    ("lazy-rounds", dict(cfg=1, B=4, K=3, V=16, dtype="f32"), dict(lazy=True), 0, True),
    ("top-128", dict(cfg=3, B=3, K=2, V=16), dict(rule=sv.SPEC_RULE_STRICT_TOP128), 0, False),
    ("top-128-fast-select", dict(cfg=3, B=2, K=2, V=4096),
     dict(rule=sv.SPEC_RULE_STRICT_TOP128), 0, False),
    ("top-128-longer-rows", dict(cfg=3, B=2, K=3, V=16384),
     dict(rule=sv.SPEC_RULE_STRICT_TOP128), 0, False),
    ("cactus-rank", dict(cfg=1, B=4, K=3, V=16, dtype="bf16"),
     dict(rule=sv.SPEC_RULE_CACTUS, ext=dict(alpha=0.3, max_rank=3, min_prob=0.01)), 0, False),
    ("kl", dict(cfg=1, B=4, K=3, V=16, dtype="bf16"), dict(kl=True), 0, False),
    ("resident", dict(cfg=1, B=2, K=2, V=16384, dtype="bf16"), dict(resident=True, rank=False),
     0, True),
    ("cluster-small", dict(cfg=1, B=4, K=3, V=16384, dtype="bf16"), {}, 32 << 20, False),
]


@pytest.mark.parametrize("name,over,kw,limit,lazy", LINEAR_CASES, ids=[c[0] for c in LINEAR_CASES])
def test_linear_schedules_checked(name, over, kw, limit, lazy):
    over = dict(over)
    cfg = over.pop("cfg")
    lb = S.make_linear(cfg, device=DEV, input_seed=8800 + len(name), sigma=0.8,
                       T=[1.0, 0.0, 0.7, 1.3][:over["B"]], **over)
    sv.spec_set_fused_limit(limit)
    g = gpu_linear(lb, **kw)
    assert g["status"] == sv.SPEC_OK, sv.spec_status_string(g["status"])
    ref = oracle_linear(lb, rule=kw.get("rule", sv.SPEC_RULE_STRICT), ext=kw.get("ext"))
    if lazy:
        _lazy_parity(g, ref, lb)
    else:
        assert_linear_parity(g, ref, lb.cu_draft.cpu(),
                             min_compared=int((ref["flag_slot"] < 0).sum()))


def test_linear_draft_probabilities_and_sparse_laws_checked():
    lb = S.make_linear(1, device=DEV, B=4, K=3, V=16, dtype="f32", T=[1.0, 0.0, 0.7, 1.3],
                       input_seed=8901)
    sv.spec_set_fused_limit(0)
    probs = probs_from_logits(lb.draft, lb.cu_draft, lb.temperature)
    g = gpu_linear(lb, draft_kind=sv.SPEC_DRAFT_PROBS, draft=probs)
    assert g["status"] == sv.SPEC_OK
    ref = oracle_linear(lb, draft_kind=sv.SPEC_DRAFT_PROBS, draft=probs)
    assert_linear_parity(g, ref, lb.cu_draft.cpu(), min_compared=int((ref["flag_slot"] < 0).sum()))
    idx, prob, ws = sv.draft_topk_softmax(lb.draft, lb.cu_draft, lb.temperature)
    assert sv.spec_get_status(ws) == sv.SPEC_OK
    g = gpu_linear(lb, draft_kind=sv.SPEC_DRAFT_SPARSE128, draft=prob, draft_idx=idx)
    assert g["status"] == sv.SPEC_OK
    ref = oracle_linear(lb, draft_kind=sv.SPEC_DRAFT_SPARSE128, draft=prob, draft_idx=idx)
    assert_linear_parity(g, ref, lb.cu_draft.cpu(), min_compared=int((ref["flag_slot"] < 0).sum()))


@pytest.mark.parametrize("V,dtype", [(16, "f32"), (4096, "bf16"), (16384, "bf16")])
def test_draft_topk_softmax_checked(V, dtype):
    lb = S.make_linear(3, device=DEV, B=3, K=2, V=V, dtype=dtype, T=[1.0, 0.0, 0.6],
                       input_seed=9000 + V)
    idx, prob, ws = sv.draft_topk_softmax(lb.draft, lb.cu_draft, lb.temperature)
    assert sv.spec_get_status(ws) == sv.SPEC_OK
    ri, rp = O.draft_topk_softmax(lb.draft.cpu(), lb.cu_draft.cpu().numpy(),
                                  lb.temperature.cpu().numpy())
    assert np.array_equal(idx.cpu().numpy(), ri)
    assert_probs_close(prob.cpu().numpy(), rp, "top-128 probabilities")


@pytest.mark.parametrize("fixed", [False, True])
def test_tree_checked(fixed):
    tb = S.make_tree(4, device=DEV, B=3, N=9, depth=3, branch=3, V=16, T=[0.8, 0.0, 1.2],
                     input_seed=9100)
    nf = None
    if fixed:
        g_ = torch.Generator().manual_seed(3)
        nf = (torch.rand(tb.node_token.numel(), generator=g_) < 0.4).to(torch.int32).to(DEV)
    g = gpu_tree(tb, node_fixed=nf)
    assert g["status"] == sv.SPEC_OK, sv.spec_status_string(g["status"])
    r = oracle_tree(tb, node_fixed=nf)
    assert_tree_parity(g, r, min_compared=int((r["flag_slot"] < 0).sum()))


def test_rheo_expand_checked():
    rb = S.make_rheo(device=DEV, input_seed=9200, B=3, W=(1, 3), V=256, K=4, m=1, n_keep=5,
                     dtype="bf16", T=0.9, level=1)
    assert_rheo_parity(rb, gpu_rheo(rb), oracle_rheo(rb), 1)


def test_uniforms_checked():
    rng = np.random.default_rng(5)
    b, pos, st = rng.integers(0, 1 << 20, 64), rng.integers(0, 1 << 10, 64), rng.integers(0, 3, 64)
    seed = 0x243F6A8885A308D3
    got = sv.spec_uniforms(seed, *(torch.tensor(x, dtype=torch.int32, device=DEV)
                                   for x in (b, pos, st))).cpu().numpy()
    want = np.array([O.uniform(seed, int(x), int(y), int(z)) for x, y, z in zip(b, pos, st)])
    assert np.array_equal(got.astype(np.float64), want)


def test_noalloc_checked():
    lb = S.make_linear(1, device=DEV, B=4, K=3, V=16, dtype="bf16", T=[1.0, 0.0, 0.7, 1.3],
                       input_seed=9300)
    tokens = torch.empty(lb.B, lb.max_k + 1, dtype=torch.int32, device=DEV)
    acc = torch.empty(lb.B, dtype=torch.int32, device=DEV)
    status = torch.full((1,), 99, dtype=torch.int32, device=DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    code = sv.lib().spec_verify_linear_noalloc(
        p(lb.target), sv.SPEC_BF16, p(lb.draft), sv.SPEC_BF16, sv.SPEC_DRAFT_LOGITS, None,
        p(lb.draft_tokens), p(lb.cu_draft), p(lb.temperature), lb.B, lb.V, lb.max_k,
        ctypes.c_uint64(lb.seed), sv.SPEC_RULE_STRICT, p(tokens), p(acc), None, p(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == sv.SPEC_OK
    torch.cuda.synchronize()
    assert int(status.item()) == sv.SPEC_OK
    g = dict(tokens=tokens.cpu().numpy(), accepted=acc.cpu().numpy(), pq=None)
    ref = oracle_linear(lb)
    _lazy_parity(g, ref, lb)


def test_wait_selftest_checked():
    ws = sv.spec_wait_selftest(1, 20_000_000)
    assert sv.spec_get_status(ws) == sv.SPEC_ERR_TIMEOUT

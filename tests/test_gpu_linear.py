"""Parity of the CUDA linear verifier (through the C ABI) with the CPU oracle."""
import numpy as np
import pytest
import torch

import speculative_decoding_rejection_gb300 as sv
from oracle import spec_oracle as O
from speculative_decoding_rejection_gb300 import synthetic as S

from parity import (assert_linear_parity, assert_probs_close, gpu_linear, oracle_linear,
                    probs_from_logits, sample_requests)

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["fused", "multi"])
def schedule(request):
    """Runs a test under both schedules of the linear verifier: the fused
    small-batch kernel (taken by calls under its size limit) and the
    multi-kernel path (limit 0)."""
    old = sv.spec_set_fused_limit((32 << 20) if request.param == "fused" else 0)
    yield request.param
    sv.spec_set_fused_limit(old)
DEV = "cuda:0"


@pytest.fixture(autouse=True, scope="module")
def _lib():
    sv.lib()


def test_device_uniforms_equal_the_oracle_hash():
    rng = np.random.default_rng(0)
    n = 4096
    b = rng.integers(0, 1 << 31, n)
    pos = rng.integers(0, 1 << 24, n)
    st = rng.integers(0, 3, n)
    seed = 0x243F6A8885A308D3
    got = sv.spec_uniforms(seed, *(torch.tensor(x, dtype=torch.int32, device=DEV)
                                   for x in (b, pos, st))).cpu().numpy()
    want = np.array([O.uniform(seed, int(x), int(y), int(z)) for x, y, z in zip(b, pos, st)])
    assert np.array_equal(got.astype(np.float64), want)


@pytest.mark.usefixtures("schedule")
def test_workload1_full():
    lb = S.make_linear(1, device=DEV)
    g = gpu_linear(lb)
    assert g["status"] == sv.SPEC_OK
    r = oracle_linear(lb)
    assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=3)


@pytest.mark.usefixtures("schedule")
def test_workload2_full_mixed_greedy_and_sampling():
    lb = S.make_linear(2, device=DEV)
    g = gpu_linear(lb)
    assert g["status"] == sv.SPEC_OK
    r = oracle_linear(lb)
    n_full, n_flag = assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=60)
    # greedy half: argmax prefix, cross-checked against a direct argmax
    tgt = lb.target.float()
    cu = lb.cu_draft.cpu().numpy()
    for b in range(32):
        t0, K = cu[b] + b, cu[b + 1] - cu[b]
        am = torch.argmax(tgt[t0:t0 + K + 1], 1).cpu().numpy()
        d = lb.draft_tokens[cu[b]:cu[b + 1]].cpu().numpy()
        n = 0
        while n < K and d[n] == am[n]:
            n += 1
        assert g["accepted"][b] == n and g["tokens"][b][n] == am[n]


@pytest.mark.parametrize("dtype,V", [("bf16", 5003), ("f32", 4099), ("bf16", 100003),
                                     ("f32", 50001), ("bf16", 7)])
@pytest.mark.usefixtures("schedule")
def test_ragged_batches_unaligned_rows_and_multiple_chunks(dtype, V):
    T = [0.0, 0.04, 0.05, 0.3, 0.7, 1.0, 1.6, 2.5] * 5
    lb = S.make_linear(2, device=DEV, B=40, K=(0, 7), V=V, dtype=dtype, sigma=0.8, T=T,
                       input_seed=1234 + V)
    assert int(torch.diff(lb.cu_draft).min()) == 0      # includes K = 0
    g = gpu_linear(lb)
    assert g["status"] == sv.SPEC_OK
    r = oracle_linear(lb)
    assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=30)


@pytest.mark.usefixtures("schedule")
def test_mixed_target_and_draft_dtypes():
    lb = S.make_linear(1, device=DEV, B=12, K=5, V=3001, dtype="bf16", input_seed=77)
    draft32 = lb.draft.float().contiguous()
    g = gpu_linear(lb, draft=draft32)
    r = oracle_linear(lb, draft=draft32)
    assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=10)


@pytest.mark.parametrize("V", [20000, 6000])
@pytest.mark.usefixtures("schedule")
def test_draft_given_as_probabilities(V):
    lb = S.make_linear(2, device=DEV, B=24, K=(1, 6), V=V, input_seed=5,
                       T=[0.0, 0.8, 1.2] * 8)
    probs = probs_from_logits(lb.draft, lb.cu_draft, lb.temperature)
    g = gpu_linear(lb, draft_kind=sv.SPEC_DRAFT_PROBS, draft=probs)
    r = oracle_linear(lb, draft_kind=sv.SPEC_DRAFT_PROBS, draft=probs)
    assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=20)


def test_sparse_draft_in_any_order_with_empty_slots():
    lb = S.make_linear(3, device=DEV, B=20, K=4, V=9000, input_seed=9)
    R_d = lb.draft.shape[0]
    gen = torch.Generator(device=DEV).manual_seed(3)
    top = torch.topk(lb.draft.float(), 128, dim=1).indices
    perm = torch.argsort(torch.rand(R_d, 128, generator=gen, device=DEV), dim=1)
    idx = torch.gather(top, 1, perm).to(torch.int32)
    idx[:, 120:] = -1                                     # some empty slots
    w = torch.rand(R_d, 128, generator=gen, device=DEV) * (idx >= 0)
    prob = (w / w.sum(1, keepdim=True)).contiguous()
    # drafts drawn from the sparse law
    pick = torch.multinomial(prob, 1, generator=gen).squeeze(1)
    lb.draft_tokens = torch.gather(idx, 1, pick[:, None]).squeeze(1).contiguous()
    g = gpu_linear(lb, draft_kind=sv.SPEC_DRAFT_SPARSE128, draft=prob, draft_idx=idx.contiguous())
    r = oracle_linear(lb, draft_kind=sv.SPEC_DRAFT_SPARSE128, draft=prob, draft_idx=idx)
    assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=15)


@pytest.mark.parametrize("V", [12288, 10001])
def test_top128_rule_with_f32_logits(V):
    """The top-128 rule on f32 logits: the final draws sweep a chunk of the
    target row four tiles of loads at a time, as 16-byte vectors (V = 12288:
    aligned rows, whole tiles) or element by element (V = 10001: rows off
    16-byte alignment, a ragged last tile)."""
    lb = S.make_linear(3, device=DEV, B=16, K=5, V=V, dtype="f32", input_seed=V)
    g = gpu_linear(lb, rule=sv.SPEC_RULE_STRICT_TOP128)
    assert g["status"] == sv.SPEC_OK
    r = oracle_linear(lb, rule=sv.SPEC_RULE_STRICT_TOP128)
    assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=12)
    assert (g["accepted"] == 5).any() and (g["accepted"] < 5).any()   # bonus and residual draws


def test_top128_rule_reduced_workload3():
    lb = S.make_linear(3, device=DEV, B=24, K=7, V=20011, input_seed=31)
    g = gpu_linear(lb, rule=sv.SPEC_RULE_STRICT_TOP128)
    assert g["status"] == sv.SPEC_OK
    r = oracle_linear(lb, rule=sv.SPEC_RULE_STRICT_TOP128)
    assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=20)


def test_top128_rule_ragged_drafts_after_a_full_call_on_one_workspace():
    """Under the top-128 rule the select's scratch holds B * max_k rows. A
    call with every request at max_k fills them all; a ragged call on the
    same workspace has fewer rows, and the scan marks the rest empty, so the
    finishing launch never reads the lists the first call left there. Both
    calls against the oracle (bf16, V % 8 == 0: the two-launch select)."""
    full = S.make_linear(3, device=DEV, B=24, K=7, V=20480, input_seed=40)
    rag = S.make_linear(3, device=DEV, B=24, K=(1, 7), V=20480, input_seed=41)
    assert rag.max_k == full.max_k == 7
    assert int(rag.cu_draft[-1]) < 24 * 7
    rule = sv.SPEC_RULE_STRICT_TOP128
    ws = torch.empty(sv.spec_verify_linear_workspace(24, 7, 20480, rule), dtype=torch.uint8,
                     device=DEV)
    for lb in (full, rag):
        tokens, acc, pq, _ = sv.spec_verify_linear(
            lb.target, lb.draft, lb.draft_tokens, lb.cu_draft, lb.temperature, lb.seed,
            max_k=7, rule=rule, want_pq=True, workspace=ws)
        g = dict(tokens=tokens.cpu().numpy(), accepted=acc.cpu().numpy(),
                 pq=pq.cpu().numpy().astype(np.float64), status=sv.spec_get_status(ws))
        assert g["status"] == sv.SPEC_OK
        r = oracle_linear(lb, rule=rule)
        assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=18)


@pytest.mark.usefixtures("schedule")
def test_greedy_rule_forces_prefix_matching():
    lb = S.make_linear(1, device=DEV, B=16, K=6, V=2048, input_seed=4)
    g = gpu_linear(lb, rule=sv.SPEC_RULE_GREEDY)
    r = oracle_linear(lb, rule=sv.SPEC_RULE_GREEDY)
    assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=16)
    assert np.all(g["pq"][:, 1] == -1.0)


@pytest.mark.usefixtures("schedule")
def test_vocabulary_of_one_token():
    lb = S.make_linear(1, device=DEV, B=3, K=2, V=1, input_seed=2)
    lb.draft_tokens.zero_()
    g = gpu_linear(lb)
    assert np.all(g["accepted"] == 2) and np.all(g["tokens"][:, :3] == 0)


@pytest.mark.usefixtures("schedule")
def test_repeat_calls_are_bitwise_deterministic():
    lb = S.make_linear(2, device=DEV, B=32, V=12000, input_seed=8)
    a, b = gpu_linear(lb), gpu_linear(lb)
    assert np.array_equal(a["tokens"], b["tokens"]) and np.array_equal(a["pq"], b["pq"])


@pytest.mark.usefixtures("schedule")
def test_invalid_device_inputs_set_the_status_word():
    lb = S.make_linear(1, device=DEV, B=4, K=3, V=512, input_seed=3)
    bad_cu = lb.cu_draft.clone()
    bad_cu[2] = bad_cu[1] - 1                             # negative draft count
    _, acc, _, ws = sv.spec_verify_linear(lb.target, lb.draft, lb.draft_tokens, bad_cu,
                                          lb.temperature, 1, max_k=lb.max_k)
    assert sv.spec_get_status(ws) == sv.SPEC_ERR_INVALID_ARG
    assert torch.all(acc == -1)
    bad_tok = lb.draft_tokens.clone()
    bad_tok[1] = 10 ** 6
    _, _, _, ws = sv.spec_verify_linear(lb.target, lb.draft, bad_tok, lb.cu_draft,
                                        lb.temperature, 1, max_k=lb.max_k)
    assert sv.spec_get_status(ws) == sv.SPEC_ERR_INVALID_ARG
    bad_T = lb.temperature.clone()
    bad_T[0] = float("nan")
    _, _, _, ws = sv.spec_verify_linear(lb.target, lb.draft, lb.draft_tokens, lb.cu_draft,
                                        bad_T, 1, max_k=lb.max_k)
    assert sv.spec_get_status(ws) == sv.SPEC_ERR_INVALID_ARG
    # a good call on the same workspace clears the word
    _, _, _, ws = sv.spec_verify_linear(lb.target, lb.draft, lb.draft_tokens, lb.cu_draft,
                                        lb.temperature, 1, max_k=lb.max_k, workspace=ws)
    assert sv.spec_get_status(ws) == sv.SPEC_OK


@pytest.mark.parametrize("cfg", [3, 5])
def test_full_size_workloads_whole_batch(cfg):
    """Every request of the full-size batch against the oracle: tokens and
    counts bit for bit up to the first draw the oracle flags."""
    lb = S.make_linear(cfg, device=DEV)
    rule = sv.SPEC_RULE_STRICT_TOP128 if lb.top128 else sv.SPEC_RULE_STRICT
    g = gpu_linear(lb, rule=rule)
    assert g["status"] == sv.SPEC_OK
    r = oracle_linear(lb, rule=rule)
    assert len(r["requests"]) == lb.B
    unflagged = int((r["flag_slot"] < 0).sum())
    n_full, n_flag = assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=unflagged)
    print(f"workload {cfg}: {n_full} requests compared in full, {n_flag} flagged")
    assert n_full == unflagged and n_full + n_flag == lb.B
    if cfg == 5:   # greedy requests are never flagged
        greedy = lb.temperature.cpu().numpy() < 0.05
        assert greedy.any() and np.all(r["flag_slot"][greedy] < 0)
        # the plain call (no p(d), q(d)) takes the position-lazy streaming
        # schedule: the same parity on the whole batch
        p = gpu_linear(lb, rule=rule, plain=True)
        assert p["status"] == sv.SPEC_OK and p["pq"] is None
        assert np.array_equal(p["accepted"], g["accepted"])
        assert_linear_parity(p, r, lb.cu_draft.cpu(), min_compared=unflagged)
    # whole-batch invariants
    acc = g["accepted"]
    K = np.diff(lb.cu_draft.cpu().numpy())
    assert np.all((acc >= 0) & (acc <= K))
    tok = g["tokens"]
    for b in range(lb.B):
        assert np.all(tok[b, :acc[b] + 1] >= 0) and np.all(tok[b, :acc[b] + 1] < lb.V)
        assert np.all(tok[b, acc[b] + 1:] == -1)


def test_draft_topk_softmax_matches_oracle():
    lb = S.make_linear(3, device=DEV, B=10, K=7, V=151936, input_seed=12)
    idx, prob, ws = sv.draft_topk_softmax(lb.draft, lb.cu_draft, lb.temperature)
    assert sv.spec_get_status(ws) == sv.SPEC_OK
    ri, rp = O.draft_topk_softmax(lb.draft.cpu(), lb.cu_draft.cpu().numpy(),
                                  lb.temperature.cpu().numpy())
    assert np.array_equal(idx.cpu().numpy(), ri)
    assert_probs_close(prob.cpu().numpy(), rp, "top-128 probabilities")


@pytest.mark.parametrize("dtype,V,T", [("bf16", 100, 1.0), ("f32", 3000, 0.7),
                                       ("bf16", 777, 0.0), ("f32", 129, 2.0),
                                       ("bf16", 4096, 1.0), ("bf16", 65536, 0.5)])
def test_draft_topk_softmax_edge_cases(dtype, V, T):
    g = torch.Generator(device=DEV).manual_seed(V)
    z = torch.randn(9, V, generator=g, device=DEV)
    z = (torch.round(z * 3) / 3).to(S._DTYPES[dtype])    # many exact ties
    if V == 65536:   # one row of a logit shape (few ties), one constant row
        z[0] = (2.0 * torch.randn(V, generator=g, device=DEV)
                - 1.1 * torch.log(torch.randperm(V, generator=g, device=DEV).float() + 1)).to(z.dtype)
        z[1] = 0.25
    cu = torch.tensor([0, 4, 9], dtype=torch.int32, device=DEV)
    temp = torch.tensor([T, T], device=DEV)
    idx, prob, ws = sv.draft_topk_softmax(z.contiguous(), cu, temp)
    assert sv.spec_get_status(ws) == sv.SPEC_OK
    ri, rp = O.draft_topk_softmax(z.cpu(), cu.cpu().numpy(), temp.cpu().numpy())
    assert np.array_equal(idx.cpu().numpy(), ri)
    assert_probs_close(prob.cpu().numpy(), rp, "top-128 probabilities")


def test_draft_topk_softmax_row_orders():
    """Rows that defeat a bound taken from the leading logits (ascending
    ramps, whose leading block holds the smallest logits), rows whose top 128
    sit inside it (descending ramps), a block of ties straddling the 128th
    logit, and logit-shaped rows: the one-pass selection, its overflow
    fallback and the tie rule against the oracle."""
    g = torch.Generator(device=DEV).manual_seed(17)
    V = 20480
    ramp = torch.arange(V, device=DEV, dtype=torch.float32) / 64
    rows = [ramp, ramp.flip(0), torch.zeros(V, device=DEV), ramp.clone(), ramp.clone()]
    rows[2][5000:5300] = 3.0                       # 300 ties: 128 lowest ids win
    rows[3][100:400] = 1000.0                      # ties inside the leading block
    rows[4] = (2.0 * torch.randn(V, generator=g, device=DEV)
               - 1.1 * torch.log(torch.randperm(V, generator=g, device=DEV).float() + 1))
    z = torch.stack(rows).to(torch.bfloat16).contiguous()
    cu = torch.tensor([0, 5], dtype=torch.int32, device=DEV)
    temp = torch.tensor([1.0], device=DEV)
    idx, prob, ws = sv.draft_topk_softmax(z, cu, temp)
    assert sv.spec_get_status(ws) == sv.SPEC_OK
    ri, rp = O.draft_topk_softmax(z.cpu(), cu.cpu().numpy(), temp.cpu().numpy())
    assert np.array_equal(idx.cpu().numpy(), ri)
    assert_probs_close(prob.cpu().numpy(), rp, "top-128 probabilities")


def test_draft_topk_softmax_predicted_bound_misses():
    """Each block predicts a row's bound from its previous row. Rows whose
    scale and offset change from row to row make that prediction too high
    (too few candidates), too low (an overflow) or right, so all three
    outcomes and the second pass they fall back to are compared with the
    oracle. 1400 rows put several rows on every block."""
    g = torch.Generator(device=DEV).manual_seed(23)
    R, V = 1400, 4096
    base = (2.0 * torch.randn(R, V, generator=g, device=DEV)
            - 1.1 * torch.log(torch.rand(R, V, generator=g, device=DEV) * V + 1))
    scale = torch.tensor([1.0, 8.0, 0.05, 1.0, 3.0, 0.5, 20.0], device=DEV)
    shift = torch.tensor([0.0, -30.0, 20.0, 5.0, -2.0, 60.0, 0.0], device=DEV)
    k = torch.arange(R, device=DEV) % 7
    z = base * scale[k, None] + shift[k, None]
    z[5::11] = torch.round(z[5::11])                  # ties at the 128th logit
    z = z.to(torch.bfloat16).contiguous()
    cu = torch.tensor([0, R], dtype=torch.int32, device=DEV)
    temp = torch.tensor([0.8], device=DEV)
    idx, prob, ws = sv.draft_topk_softmax(z, cu, temp)
    assert sv.spec_get_status(ws) == sv.SPEC_OK
    rows = np.r_[0:40, 300:340, 600:640, 1300:1400]
    cu_s = np.array([0, rows.size], dtype=np.int32)
    ri, rp = O.draft_topk_softmax(z[rows].cpu(), cu_s, temp.cpu().numpy())
    assert np.array_equal(idx[rows].cpu().numpy(), ri)
    assert_probs_close(prob[rows].cpu().numpy(), rp, "top-128 probabilities")


@pytest.mark.parametrize("B", [20, 700])
def test_draft_topk_softmax_request_lookup(B):
    """Each row's temperature is its request's: rows map to requests through
    cu (the largest b with cu[b] <= r), with empty requests among them, and
    the search narrows in one (20) or two (700) 32-way steps. Every
    request has its own temperature, greedy ones among them, so a row given
    a neighbour's temperature fails the comparison."""
    g = torch.Generator(device="cpu").manual_seed(B)
    V = 4096
    K = torch.randint(0, 4, (B,), generator=g)
    K[0], K[-1] = 0, 2                                  # an empty first request
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(K, 0)
    R = int(cu[-1])
    temp = 0.3 + 0.004 * torch.arange(B, dtype=torch.float32)
    temp[::9] = 0.0                                      # greedy requests
    z = (2.0 * torch.randn(R, V, generator=g)
         - 1.1 * torch.log(torch.rand(R, V, generator=g) * V + 1)).to(torch.bfloat16)
    idx, prob, ws = sv.draft_topk_softmax(z.to(DEV), cu.to(DEV), temp.to(DEV))
    assert sv.spec_get_status(ws) == sv.SPEC_OK
    ri, rp = O.draft_topk_softmax(z, cu.numpy(), temp.numpy())
    assert np.array_equal(idx.cpu().numpy(), ri)
    assert_probs_close(prob.cpu().numpy(), rp, "top-128 probabilities")


# ------------------------------------------- relaxed CACTUS rule and ranks
CACTUS_CASES = [
    dict(alpha=0.0, max_rank=0, min_prob=0.0),     # the lossless test
    dict(alpha=0.05, max_rank=0, min_prob=0.0),
    dict(alpha=0.5, max_rank=10, min_prob=0.10),   # the recommended guard
    dict(alpha=2.0, max_rank=3, min_prob=0.0),
    dict(alpha=0.2, max_rank=0, min_prob=0.02),
]


@pytest.mark.parametrize("ext", CACTUS_CASES)
@pytest.mark.parametrize("dtype,V", [("bf16", 50021), ("f32", 3001), ("bf16", 262144)])
def test_cactus_rule_and_target_ranks(ext, dtype, V):
    T = [0.0, 0.3, 0.7, 1.0, 1.4] * 6
    lb = S.make_linear(2, device=DEV, B=30, K=(0, 6), V=V, dtype=dtype, sigma=0.6, T=T,
                       input_seed=900 + V)
    g = gpu_linear(lb, rule=sv.SPEC_RULE_CACTUS, ext=ext)
    assert g["status"] == sv.SPEC_OK
    r = oracle_linear(lb, rule=sv.SPEC_RULE_CACTUS, ext=ext)
    assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=20)
    if ext["alpha"] == 0.0:   # alpha 0, guard off: the strict rule bit for bit
        s = gpu_linear(lb)
        assert np.array_equal(s["tokens"], g["tokens"])


def test_target_ranks_under_the_strict_rule_with_ties():
    """Ranks through the extended entry point with the lossless rule; logits
    rounded to a coarse grid so many tokens tie with the draft token."""
    lb = S.make_linear(1, device=DEV, B=16, K=5, V=70001, input_seed=21)
    lb.target = (torch.round(lb.target.float() * 4) / 4).to(lb.target.dtype).contiguous()
    g = gpu_linear(lb, ext=dict(alpha=0.0, max_rank=0, min_prob=0.0))
    r = oracle_linear(lb)
    assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=12)
    s = gpu_linear(lb)
    assert np.array_equal(s["tokens"], g["tokens"])


def test_cactus_full_size_workload5_sampled():
    lb = S.make_linear(5, device=DEV)
    ext = dict(alpha=0.5, max_rank=10, min_prob=0.10)
    g = gpu_linear(lb, rule=sv.SPEC_RULE_CACTUS, ext=ext)
    assert g["status"] == sv.SPEC_OK
    req = sample_requests(lb.B, 16, seed=55)
    r = oracle_linear(lb, rule=sv.SPEC_RULE_CACTUS, requests=req, ext=ext)
    assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=13)


def test_cactus_argument_errors():
    lb = S.make_linear(1, device=DEV, B=2, K=2, V=64, input_seed=3)
    with pytest.raises(sv.SpecError):   # the relaxed rule needs its options
        sv.spec_verify_linear(lb.target, lb.draft, lb.draft_tokens, lb.cu_draft,
                              lb.temperature, 1, max_k=lb.max_k, rule=sv.SPEC_RULE_CACTUS)
    for bad in (dict(alpha=-1.0), dict(alpha=float("nan")), dict(max_rank=-2),
                dict(min_prob=float("inf"))):
        with pytest.raises(sv.SpecError):
            sv.spec_verify_linear_ext(lb.target, lb.draft, lb.draft_tokens, lb.cu_draft,
                                      lb.temperature, 1, max_k=lb.max_k,
                                      rule=sv.SPEC_RULE_CACTUS, **bad)


# ---------------------------------------------- position-lazy verification
def assert_lazy_matches(g, ref, lb, min_compared=10):
    """Tokens and counts as the oracle; p(d), q(d) and ranks on the read
    positions, NaN / -1 exactly on the unread ones."""
    lz = O.lazy_view(ref, lb.cu_draft.cpu().numpy())
    assert np.array_equal(np.isnan(g["pq"][:, 0]), np.isnan(lz["pq"][:, 0]))
    if "rank" in g:
        assert np.array_equal(g["rank"] == -1, lz["rank"] == -1)
    assert_linear_parity(g, lz, lb.cu_draft.cpu(), min_compared=min_compared)


LAZY_CASES = [
    dict(cfg=2, over=dict(B=40, K=(0, 7), V=30011, dtype="bf16", sigma=0.9,
                          T=[0.0, 0.6, 1.0, 1.3] * 10), kw={}),
    dict(cfg=2, over=dict(B=24, K=(1, 6), V=4099, dtype="f32", sigma=1.2,
                          T=[0.7, 1.0] * 12), kw={}),
    dict(cfg=1, over=dict(B=16, K=8, V=100003, dtype="bf16", sigma=1.0, T=1.0),
         kw=dict(rule=sv.SPEC_RULE_CACTUS, ext=dict(alpha=0.2, max_rank=10, min_prob=0.05))),
]


@pytest.mark.parametrize("case", LAZY_CASES)
def test_lazy_equals_eager_and_the_oracle(case):
    lb = S.make_linear(case["cfg"], device=DEV, input_seed=4242, **case["over"])
    kw = dict(case["kw"])
    g = gpu_linear(lb, lazy=True, **kw)
    assert g["status"] == sv.SPEC_OK
    e = gpu_linear(lb, **kw)
    assert np.array_equal(g["tokens"], e["tokens"]) and np.array_equal(g["accepted"], e["accepted"])
    ref = oracle_linear(lb, rule=kw.get("rule", sv.SPEC_RULE_STRICT), ext=kw.get("ext"))
    assert_lazy_matches(g, ref, lb)
    assert 0 < g["accepted"].mean() < lb.max_k


# The position-lazy schedule of dense bf16 logits with V % 8 == 0 runs as one
# persistent kernel (decisions, residual tile sums and final draws inside
# it); these cases reach it, with and without the rank count.
STREAM_CASES = [
    dict(cfg=2, over=dict(B=48, K=(0, 7), V=32000, dtype="bf16", sigma=0.9,
                          T=[0.0, 0.6, 1.0, 1.3] * 12), kw={}),
    dict(cfg=2, over=dict(B=24, K=(1, 6), V=201088, dtype="bf16", sigma=1.2,
                          T=[0.7, 1.0, 0.03] * 8), kw={}),
    dict(cfg=1, over=dict(B=20, K=8, V=100000, dtype="bf16", sigma=1.0, T=1.0),
         kw=dict(rule=sv.SPEC_RULE_CACTUS, ext=dict(alpha=0.2, max_rank=10, min_prob=0.05))),
    # a ragged last residual tile (4104 = 4096 + 8) and mostly accepted drafts
    dict(cfg=1, over=dict(B=12, K=5, V=4104, dtype="bf16", sigma=0.3, T=0.9), kw={}),
]


@pytest.mark.parametrize("rank", [True, False])
@pytest.mark.parametrize("case", STREAM_CASES)
def test_stream_schedule_equals_eager_and_the_oracle(case, rank):
    lb = S.make_linear(case["cfg"], device=DEV, input_seed=5151, **case["over"])
    kw = dict(case["kw"])
    if not rank and kw.get("ext", {}).get("max_rank", 0) > 0:
        pytest.skip("the guard on target rank needs the rank count")
    g = gpu_linear(lb, lazy=True, rank=rank, **kw)
    assert g["status"] == sv.SPEC_OK
    e = gpu_linear(lb, **kw)
    assert np.array_equal(g["tokens"], e["tokens"]) and np.array_equal(g["accepted"], e["accepted"])
    ref = oracle_linear(lb, rule=kw.get("rule", sv.SPEC_RULE_STRICT), ext=kw.get("ext"))
    assert_lazy_matches(g, ref, lb)
    assert 0 < g["accepted"].mean() < lb.max_k
    again = gpu_linear(lb, lazy=True, rank=rank, **kw)   # bitwise deterministic
    assert np.array_equal(again["tokens"], g["tokens"])
    assert np.array_equal(again["pq"], g["pq"], equal_nan=True)


def test_stream_schedule_full_size_workload5_whole_batch():
    """Full size, every request: counts equal to the eager schedule; tokens
    equal except where the oracle flags a draw within 1e-6 of a boundary
    (the schedules sum the chunk statistics in different orders); parity
    with the oracle on the whole batch."""
    lb = S.make_linear(5, device=DEV)
    g = gpu_linear(lb, lazy=True, rank=False)
    assert g["status"] == sv.SPEC_OK
    e = gpu_linear(lb)
    assert np.array_equal(g["accepted"], e["accepted"])
    diff = np.nonzero((g["tokens"] != e["tokens"]).any(1))[0]
    print("requests where the schedules differ:", diff.tolist())
    ref = oracle_linear(lb)
    lz = O.lazy_view(ref, lb.cu_draft.cpu().numpy())
    for b in diff:
        print(b, "lazy", g["tokens"][b], "eager", e["tokens"][b], "oracle",
              ref["tokens"][b], "flag slot", ref["flag_slot"][b])
        assert ref["flag_slot"][b] >= 0, "the schedules differ on an unflagged draw"
    unflagged = int((ref["flag_slot"] < 0).sum())
    n_full, n_flag = assert_linear_parity(g, lz, lb.cu_draft.cpu(), min_compared=unflagged)
    print(f"{n_full} requests compared in full, {n_flag} flagged")


# The cluster-resident schedule (SPEC_EXT_RESIDENT): strict rule, dense bf16
# logits, 16384 <= V <= 204800. Fewer requests than clusters, ragged and
# empty drafts, greedy and sampling requests, the smallest and largest V,
# slices of unequal length (V / 8 not a multiple of 8).
RESIDENT_CASES = [
    dict(B=1, K=4, V=16384, sigma=0.8, T=1.0),
    dict(B=40, K=(0, 6), V=65536, sigma=0.9, T=[0.0, 0.5, 1.0, 1.5] * 10),
    dict(B=16, K=3, V=204800, sigma=1.0, T=0.9),
    dict(B=24, K=(1, 5), V=30008, sigma=0.4, T=[0.7, 0.02, 1.2] * 8),
    dict(B=70, K=4, V=201088, sigma=1.3, T=0.8),
]


@pytest.mark.parametrize("over", RESIDENT_CASES)
def test_resident_schedule_equals_eager_and_the_oracle(over):
    lb = S.make_linear(2, device=DEV, input_seed=6161, dtype="bf16", **over)
    g = gpu_linear(lb, resident=True, rank=False)
    assert g["status"] == sv.SPEC_OK
    e = gpu_linear(lb, eager=True, rank=False)
    same = (g["tokens"] == e["tokens"]).all(1)
    assert np.array_equal(g["accepted"], e["accepted"])
    ref = oracle_linear(lb)
    for b in np.nonzero(~same)[0]:   # the schedules sum rows in different orders
        assert ref["flag_slot"][b] >= 0, ("differs from eager on an unflagged draw", b)
    assert_lazy_matches(g, ref, lb, min_compared=int((ref["flag_slot"] < 0).sum()))
    again = gpu_linear(lb, resident=True, rank=False)   # bitwise deterministic
    assert np.array_equal(again["tokens"], g["tokens"])
    assert np.array_equal(again["pq"], g["pq"], equal_nan=True)


def test_resident_schedule_full_size_workload5_whole_batch():
    """B = 1024, K = 4, V = 201088: every request against the oracle."""
    lb = S.make_linear(5, device=DEV)
    g = gpu_linear(lb, resident=True, rank=False)
    assert g["status"] == sv.SPEC_OK
    ref = oracle_linear(lb)
    lz = O.lazy_view(ref, lb.cu_draft.cpu().numpy())
    unflagged = int((ref["flag_slot"] < 0).sum())
    n_full, n_flag = assert_linear_parity(g, lz, lb.cu_draft.cpu(), min_compared=unflagged)
    print(f"resident: {n_full} requests compared in full, {n_flag} flagged")


def test_resident_schedule_reports_invalid_inputs():
    lb = S.make_linear(2, device=DEV, B=6, K=3, V=16384, dtype="bf16", T=1.0, input_seed=3)
    assert gpu_linear(lb, resident=True, rank=False)["status"] == sv.SPEC_OK
    bad = lb.draft_tokens.clone()
    bad[4] = lb.V                               # a draft token outside the vocabulary
    b2 = S.LinearBatch(**{**lb.__dict__, "draft_tokens": bad})
    g = gpu_linear(b2, resident=True, rank=False)
    assert g["status"] == sv.SPEC_ERR_INVALID_ARG
    assert np.all(g["accepted"] == -1)
    assert gpu_linear(lb, resident=True, rank=False)["status"] == sv.SPEC_OK


# Small calls of longer bf16 rows (at most 128 requests and 8 drafts, row
# slices of V/8 fitting a cluster's shared memory) run as one cluster per
# request with every row resident: the same results as the multi-kernel path
# and the oracle, p(d) and q(d) for every position (every row is read).
CLUSTER_SMALL_CASES = [
    dict(B=64, K=(1, 5), V=32000, sigma=0.7, T=[0.0, 0.7] * 32),
    dict(B=1, K=8, V=16384, sigma=0.2, T=1.0),
    dict(B=128, K=(0, 4), V=20000, sigma=1.2, T=("uniform", 0.0, 1.4)),
    dict(B=37, K=3, V=36864, sigma=0.9, T=[1.3, 0.5, 0.01] * 12 + [0.9]),
    dict(B=9, K=(2, 8), V=9000, sigma=0.5, T=0.8),
]


@pytest.mark.parametrize("over", CLUSTER_SMALL_CASES)
def test_cluster_small_calls_equal_the_multi_kernel_path_and_the_oracle(over):
    lb = S.make_linear(2, device=DEV, input_seed=7272, dtype="bf16", **over)
    old = sv.spec_set_fused_limit(32 << 20)
    try:
        g = gpu_linear(lb)
        assert g["status"] == sv.SPEC_OK
        again = gpu_linear(lb)                      # bitwise deterministic
        assert np.array_equal(again["tokens"], g["tokens"])
        assert np.array_equal(again["pq"], g["pq"])
        sv.spec_set_fused_limit(0)
        e = gpu_linear(lb)                          # the multi-kernel path
    finally:
        sv.spec_set_fused_limit(old)
    assert np.array_equal(g["accepted"], e["accepted"])
    ref = oracle_linear(lb)
    for b in np.nonzero((g["tokens"] != e["tokens"]).any(1))[0]:
        assert ref["flag_slot"][b] >= 0, ("differs from the multi-kernel path unflagged", b)
    assert_linear_parity(g, ref, lb.cu_draft.cpu(), min_compared=int((ref["flag_slot"] < 0).sum()))


def test_cluster_small_reports_invalid_inputs():
    lb = S.make_linear(2, device=DEV, B=6, K=3, V=16384, dtype="bf16", T=1.0, input_seed=3)
    assert gpu_linear(lb)["status"] == sv.SPEC_OK
    bad = lb.draft_tokens.clone()
    bad[2] = -5
    b2 = S.LinearBatch(**{**lb.__dict__, "draft_tokens": bad})
    g = gpu_linear(b2)
    assert g["status"] == sv.SPEC_ERR_INVALID_ARG and np.all(g["accepted"] == -1)


def test_stream_schedule_invalid_inputs_and_empty_rows():
    lb = S.make_linear(1, device=DEV, B=6, K=3, V=4096, dtype="bf16", T=1.0, input_seed=3)
    clean = gpu_linear(lb, lazy=True)
    assert clean["status"] == sv.SPEC_OK

    def run(**over):
        b2 = S.LinearBatch(**{**lb.__dict__, **over})
        return gpu_linear(b2, lazy=True)

    bad_cu = lb.cu_draft.clone()
    bad_cu[2] = bad_cu[1] - 1                             # negative draft count
    r = run(cu_draft=bad_cu)
    assert r["status"] == sv.SPEC_ERR_INVALID_ARG and np.all(r["accepted"] == -1)
    bad_tok = lb.draft_tokens.clone()
    bad_tok[4] = 10 ** 6
    r = run(draft_tokens=bad_tok)
    assert r["status"] == sv.SPEC_ERR_INVALID_ARG and np.all(r["accepted"] == -1)
    bad_T = lb.temperature.clone()
    bad_T[1] = float("nan")
    assert run(temperature=bad_T)["status"] == sv.SPEC_ERR_INVALID_ARG
    # a row without mass found while the kernel runs: the other requests are
    # still verified, and the status word reports it at the end
    t2 = lb.target.clone()
    t2[int(lb.cu_draft[2]) + 2] = float("-inf")           # request 2, position 1
    r = run(target=t2)
    assert r["status"] == sv.SPEC_ERR_INVALID_ARG
    keep = [b for b in range(lb.B) if b != 2]
    assert np.array_equal(r["tokens"][keep], clean["tokens"][keep])
    assert gpu_linear(lb, lazy=True)["status"] == sv.SPEC_OK


def test_lazy_with_probability_and_sparse_drafts():
    lb = S.make_linear(2, device=DEV, B=20, K=(1, 6), V=20000, input_seed=515,
                       T=[0.0, 0.8, 1.2, 1.0] * 5)
    probs = probs_from_logits(lb.draft, lb.cu_draft, lb.temperature)
    g = gpu_linear(lb, draft_kind=sv.SPEC_DRAFT_PROBS, draft=probs, lazy=True)
    ref = oracle_linear(lb, draft_kind=sv.SPEC_DRAFT_PROBS, draft=probs)
    assert_lazy_matches(g, ref, lb)
    idx, prob, _ = sv.draft_topk_softmax(lb.draft, lb.cu_draft, lb.temperature)
    g = gpu_linear(lb, draft_kind=sv.SPEC_DRAFT_SPARSE128, draft=prob, draft_idx=idx, lazy=True)
    ref = oracle_linear(lb, draft_kind=sv.SPEC_DRAFT_SPARSE128, draft=prob, draft_idx=idx)
    assert_lazy_matches(g, ref, lb)


def test_lazy_never_uses_rows_after_the_first_rejection():
    """Rows after position n+1 are set to -inf everywhere (no mass): the
    eager call reports them, the lazy call never uses them (the streaming
    kernel may read some of them before the rejection is known)."""
    lb = S.make_linear(2, device=DEV, B=32, K=(2, 6), V=8192, input_seed=99, sigma=1.5,
                       T=[0.0, 1.0] * 16)
    ref = oracle_linear(lb)
    cu = lb.cu_draft.cpu().numpy()
    t2, d2 = lb.target.clone(), lb.draft.clone()
    for j, b in enumerate(ref["requests"]):
        n, K = int(ref["accepted"][j]), int(cu[b + 1] - cu[b])
        t0, d0 = int(cu[b]) + int(b), int(cu[b])
        t2[t0 + n + 1:t0 + K + 1] = float("-inf")
        d2[d0 + min(n + 1, K):d0 + K] = float("-inf")
    assert (t2 == float("-inf")).all(1).sum() > 10
    lb2 = S.LinearBatch(**{**lb.__dict__, "target": t2, "draft": d2})
    g = gpu_linear(lb2, lazy=True)
    assert g["status"] == sv.SPEC_OK
    assert_lazy_matches(g, ref, lb)
    e = gpu_linear(lb2)
    assert e["status"] == sv.SPEC_ERR_INVALID_ARG


# ------------------------------------------------- per-position KL(p || q)
from parity import assert_kl_close  # noqa: E402


@pytest.mark.parametrize("dtype,V,over", [
    ("bf16", 32000, dict(cfg=2, B=40, K=(0, 6), T=[0.0, 0.4, 0.8, 1.0, 1.7] * 8)),
    ("f32", 1024, dict(cfg=1, B=12, K=5, T=1.0)),
    ("bf16", 200000, dict(cfg=2, B=10, K=(1, 4), T=[0.6, 1.2] * 5)),
])
def test_kl_per_position_eager(dtype, V, over):
    cfg = over.pop("cfg")
    lb = S.make_linear(cfg, device=DEV, V=V, dtype=dtype, sigma=0.8, input_seed=77 + V, **over)
    g = gpu_linear(lb, kl=True)
    assert g["status"] == sv.SPEC_OK
    r = oracle_linear(lb)
    assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=8)
    rows = np.arange(int(lb.cu_draft[-1]))
    print("kl err / scale", assert_kl_close(g["kl"], r, lb, rows))


def test_kl_with_cactus_rank_and_lazy_rounds():
    lb = S.make_linear(2, device=DEV, B=24, K=(1, 6), V=65536, sigma=1.0,
                       T=[0.0, 0.7, 1.0, 1.3] * 6, input_seed=321)
    ext = dict(alpha=0.3, max_rank=5, min_prob=0.01)
    g = gpu_linear(lb, rule=sv.SPEC_RULE_CACTUS, ext=ext, kl=True)
    r = oracle_linear(lb, rule=sv.SPEC_RULE_CACTUS, ext=ext)
    assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=18)
    assert_kl_close(g["kl"], r, lb, np.arange(int(lb.cu_draft[-1])))
    gl = gpu_linear(lb, rule=sv.SPEC_RULE_CACTUS, ext=ext, kl=True, lazy=True)
    lz = O.lazy_view(r, lb.cu_draft.cpu().numpy())
    assert_linear_parity(gl, lz, lb.cu_draft.cpu(), min_compared=18)
    assert_kl_close(gl["kl"], lz, lb, np.arange(int(lb.cu_draft[-1])))


def test_kl_full_size_workload5_sampled():
    lb = S.make_linear(5, device=DEV)
    g = gpu_linear(lb, kl=True)
    assert g["status"] == sv.SPEC_OK
    req = sample_requests(lb.B, 12, seed=8)
    r = oracle_linear(lb, requests=req)
    assert_linear_parity(g, r, lb.cu_draft.cpu(), min_compared=9)
    cu = lb.cu_draft.cpu().numpy()
    rows = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in req])
    assert_kl_close(g["kl"], r, lb, rows)


def test_kl_argument_errors():
    lb = S.make_linear(1, device=DEV, B=2, K=2, V=64, input_seed=3)
    probs = probs_from_logits(lb.draft, lb.cu_draft, lb.temperature)
    with pytest.raises(sv.SpecError):   # q given as probabilities
        sv.spec_verify_linear_ext(lb.target, probs, lb.draft_tokens, lb.cu_draft,
                                  lb.temperature, 1, max_k=lb.max_k,
                                  draft_kind=sv.SPEC_DRAFT_PROBS, want_kl=True)
    with pytest.raises(sv.SpecError):   # truncated draft law
        sv.spec_verify_linear_ext(lb.target, lb.draft, lb.draft_tokens, lb.cu_draft,
                                  lb.temperature, 1, max_k=lb.max_k,
                                  rule=sv.SPEC_RULE_STRICT_TOP128, want_kl=True)
    odd = S.make_linear(1, device=DEV, B=2, K=2, V=5003, dtype="bf16", input_seed=3)
    with pytest.raises(sv.SpecError):   # rows not 16-byte multiples
        sv.spec_verify_linear_ext(odd.target, odd.draft, odd.draft_tokens, odd.cu_draft,
                                  odd.temperature, 1, max_k=odd.max_k, want_kl=True)

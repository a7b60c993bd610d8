"""Helpers comparing the CUDA verifier with the CPU oracle on the same inputs.

Tolerances: committed tokens and accepted counts bit-exact, except from the
first output slot whose draw the oracle flags as within 1e-6 of a decision
boundary; probabilities within 1e-5 relative (fp32 GPU vs fp64 oracle).
"""
import math

import numpy as np
import torch

import speculative_decoding_rejection_gb300 as sv
from oracle import spec_oracle as O

PROB_RTOL = 1e-5
PROB_ATOL = 1e-30


def gpu_linear(lb, rule=sv.SPEC_RULE_STRICT, draft_kind=sv.SPEC_DRAFT_LOGITS, draft=None,
               draft_idx=None, ext=None, lazy=False, kl=False, rank=True, resident=False,
               eager=False, plain=False):
    """Runs the CUDA verifier; `ext` (a dict of alpha / max_rank / min_prob),
    `lazy`, `resident` or `eager` go through spec_verify_linear_ext, which
    also returns target ranks unless `rank` is False. `plain` calls
    spec_verify_linear without p(d), q(d) (the library picks the schedule);
    the other plain calls ask for them."""
    draft = lb.draft if draft is None else draft
    if ext is None and not (lazy or kl or resident or eager):
        tokens, acc, pq, ws = sv.spec_verify_linear(
            lb.target, draft, lb.draft_tokens, lb.cu_draft, lb.temperature, lb.seed,
            max_k=lb.max_k, rule=rule, draft_kind=draft_kind, draft_idx=draft_idx,
            want_pq=not plain)
        rank = None
    else:
        tokens, acc, pq, rank, klv, ws = sv.spec_verify_linear_ext(
            lb.target, draft, lb.draft_tokens, lb.cu_draft, lb.temperature, lb.seed,
            max_k=lb.max_k, rule=rule, draft_kind=draft_kind, draft_idx=draft_idx,
            want_pq=True, want_rank=rank, want_kl=kl, lazy=lazy, resident=resident,
            eager=eager, **(ext or {}))
    status = sv.spec_get_status(ws)
    out = dict(tokens=tokens.cpu().numpy(), accepted=acc.cpu().numpy(),
               pq=None if pq is None else pq.cpu().numpy().astype(np.float64), status=status)
    if rank is not None:
        out["rank"] = rank.cpu().numpy().astype(np.int64)
    if kl:
        out["kl"] = klv.cpu().numpy().astype(np.float64)
    return out


def oracle_linear(lb, rule=sv.SPEC_RULE_STRICT, draft_kind=sv.SPEC_DRAFT_LOGITS, draft=None,
                  draft_idx=None, requests=None, ext=None):
    draft = lb.draft if draft is None else draft
    host = (lambda t: t.cpu()) if requests is None else (lambda t: t)
    return O.verify_linear(host(lb.target), host(draft), lb.draft_tokens.cpu().numpy(),
                           lb.cu_draft.cpu().numpy(), lb.temperature.cpu().numpy(), lb.seed,
                           rule=rule, draft_kind=draft_kind,
                           draft_idx=None if draft_idx is None else draft_idx.cpu().numpy(),
                           max_k=lb.max_k, requests=requests, **(ext or {}))


def assert_probs_close(g, o, what="probabilities"):
    g = np.asarray(g, np.float64)
    o = np.asarray(o, np.float64)
    bad = np.abs(g - o) > PROB_RTOL * np.abs(o) + PROB_ATOL
    assert not bad.any(), (what, np.argwhere(bad)[:5], g[bad][:5], o[bad][:5])


def assert_linear_parity(gpu, ref, cu_draft, min_compared=1):
    """Token/accepted parity per request, skipping from the first flagged slot;
    p(d), q(d) parity for every draft position of the compared requests.
    Returns (n_requests_fully_compared, n_flagged)."""
    cu = np.asarray(cu_draft)
    n_full = n_flag = 0
    rows = []
    for j, b in enumerate(ref["requests"]):
        fs = int(ref["flag_slot"][j])
        gt, rt = gpu["tokens"][b], ref["tokens"][j]
        if fs < 0:
            assert np.array_equal(gt, rt), (b, gt, rt)
            assert gpu["accepted"][b] == ref["accepted"][j], (b, gpu["accepted"][b], ref["accepted"][j])
            n_full += 1
        else:
            assert np.array_equal(gt[:fs], rt[:fs]), (b, fs, gt, rt)
            n_flag += 1
        rows.extend(range(int(cu[b]), int(cu[b + 1])))
    rows = np.asarray(rows, dtype=np.int64)
    if rows.size and gpu["pq"] is not None:
        assert_probs_close(gpu["pq"][rows], ref["pq"][rows], "p(d), q(d)")
        if "rank" in gpu:   # integer counts: bit-exact
            bad = gpu["rank"][rows] != ref["rank"][rows]
            assert not bad.any(), ("rank", rows[bad][:5], gpu["rank"][rows][bad][:5],
                                   ref["rank"][rows][bad][:5])
    assert n_full >= min_compared
    return n_full, n_flag


# KL(p || q) = (A/S - (m_t - m_d))/T - ln S_t + ln S_d from fp32 sums: each
# term is bounded by (max|z_t| + max|z_d|)/T or by ln V, and fp32 sums over a
# row carry ~1e-7 relative error (measured: at most 4e-8 of the scale), so
# the bound is KL_RTOL of that scale.
KL_RTOL = 1e-6


def assert_kl_close(g_kl, ref, lb, rows):
    """KL per draft row `rows`: NaN exactly where the oracle has NaN, +inf
    where it has +inf, else within KL_RTOL * (1 + R/T + ln V)."""
    o = ref["kl"][rows]
    g = g_kl[rows]
    assert np.array_equal(np.isnan(g), np.isnan(o)), ("kl NaN pattern", rows[np.isnan(g) != np.isnan(o)][:5])
    assert np.array_equal(np.isinf(g), np.isinf(o))
    ok = np.isfinite(o)
    if not ok.any():
        return 0.0
    cu = lb.cu_draft.cpu().numpy()
    req = np.searchsorted(cu, rows, side="right") - 1
    t_rows = rows + req
    T = lb.temperature.cpu().numpy()[req]
    zt = lb.target.float()[torch.as_tensor(t_rows, device=lb.target.device)]
    zd = lb.draft.float()[torch.as_tensor(rows, device=lb.draft.device)]
    R = (zt.abs().amax(1) + zd.abs().amax(1)).cpu().numpy().astype(np.float64)
    scale = 1.0 + R / np.maximum(T, 1e-30) + math.log(lb.V)
    err = np.abs(g[ok] - o[ok]) / scale[ok]
    assert err.max() <= KL_RTOL, ("kl", float(err.max()), rows[ok][np.argmax(err)])
    return float(err.max())


def sample_requests(B, n, seed=0):
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(B, size=min(n, B), replace=False))


def probs_from_logits(draft, cu, temperature):
    """Draft probabilities softmax(z/T) for the PROBS draft kind (input
    preparation with torch; T < 0.05 rows get a one-hot on the argmax)."""
    cu = cu.long().cpu()
    T = temperature.cpu()
    req = torch.repeat_interleave(torch.arange(T.numel()), torch.diff(cu)).to(draft.device)
    Tr = T.to(draft.device)[req]
    z = draft.float()
    soft = torch.softmax(z / torch.clamp(Tr, min=0.05)[:, None], dim=1)
    hard = torch.nn.functional.one_hot(torch.argmax(z, 1), z.shape[1]).float()
    return torch.where((Tr < 0.05)[:, None], hard, soft).contiguous()

"""Plain fp64 CPU oracle for the batched speculative-decoding verifier.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module. The product path (the CUDA library and its Python binding) never does,
and shares no code with it: its own hash, its own softmax, its own search.

Everything is computed in float64 with numpy, one request at a time, in the
order the sources state the steps. Logits arrive as bf16 or fp32 and are
upcast exactly to float64 before any arithmetic.

Sources (web pages; cited by title and section):

* "Acceptance Is Not Speed (arXiv:2610.23818)" (newsaint.id), §1 "Ilusi Metrik
  Spekulatif" (lossless verification keeps the output distribution equal to
  the target's p) and §6 "Implementasi Referensi" (a draft token is accepted
  outright when q(x) <= p(x); otherwise a coin decides).
* "RheoSampling 2026" (newsaint.id), §1 (temperature acts on sampling and the
  verification gate), §3 "Optimasi Sparse Top-128" (draft logits cut to their
  128 largest before the softmax, the rest at -inf), §4 "RheoVerification"
  (accept with min(1, p/q~); on rejection use the normalised residual
  norm(max(0, p - q~)) and test the remaining drafts against it; descend into
  the subtree on acceptance), §6 "Teorema 1" (the output law equals p).
* "Acceptance Is Not Speed (arXiv:2610.23818)", §2 "Taksonomi 5 Aturan Lossy
  Speculative Decoding" (relaxed rules replace the target law in the
  acceptance test), §6 RULE 1-3 of the reference harness (the low-support
  guard on target rank and p(x), then the strict test, then the CACTUS test
  gamma(x) = min(p(x) + sqrt(2 alpha p(x) (1 - p(x))), 1) against q(x)) and §7
  item 3 (the guard with p(x) < 0.10 or outside the top k = 10).
* "Test-Time Speculation" (gist.science summary of arXiv 2605.09329), §2
  "Methodik" step 3: the verification step's target law p and draft law q
  over the drafted canvas give the distillation signal KL(p || q).
* "Speculative decoding: memverifikasi token draft sebelum diterima"
  (nalar.dev), sections "Draft mengubah tebakan serial menjadi batch
  verifikasi" (one target pass scores positions 1..K+1, each conditioned on
  the drafts before it), "Semantik penerimaan" (greedy: accept while the draft
  equals the target's greedy choice, the target's choice replaces the first
  mismatch; sampling: acceptance from p and q, correction draw on rejection)
  and "Penolakan memendekkan pekerjaan speculative" (drafts after the first
  rejection are discarded).

Readings where the pages are silent (each also listed in the design notes):

R1  Uniforms come from a counter hash: u = (splitmix64(seed ^ splitmix64(key))
    >> 40) * 2^-24 with key = (b << 32) | (pos << 8) | stream; splitmix64 is
    the public SplitMix64 output function (Steele, Lea & Flood 2014) applied to
    x + 0x9E3779B97F4A7C15. Streams: 0 acceptance coin, 1 residual draw,
    2 bonus draw.
R2  Greedy when T < 0.05; argmax ties go to the lowest token id.
R3  Accept iff u < a with a = 1 when q(d) <= p(d), else p(d)/q(d).
R4  Inverse CDF in ascending token id with inclusive prefix sums: the token is
    the smallest x with u*Z < C_x. If rounding leaves no such x, the largest x
    of positive weight. If the residual has Z == 0, p is sampled instead.
R5  Bonus token when all K drafts are accepted: a draw from p_{K+1}.
R6  Top-128: the 128 largest logits with ties to the lower id; the softmax at
    temperature T runs over the survivors only.
R7  Tree: children of a node are tested in node-index order (the order they
    were drawn without replacement). After rejecting x, the draft law drops x
    and is renormalised by 1 - q(E). Coins are keyed by the child's node
    index; the final draw at node v by v + 1, so a chain tree reproduces the
    linear verifier bit for bit. Greedy trees accept the first child equal to
    argmax p_v.
R8  A draw is *flagged* when the exact value sits within 1e-6 of a decision
    boundary (|u - a| <= 1e-6 for a coin, |u*Z - C| <= 1e-6*Z for either
    cumulative bracketing the chosen token, |p(d) - min_prob| <= 1e-6 for the
    low-support guard). Tokens from that output slot on are not compared bit
    for bit against a fp32 implementation.
R9  Target rank of d: 1 + the number of tokens whose target logit is strictly
    larger than d's (tied tokens share the better rank; temperature does not
    change it).
R10 CACTUS rule: accept d iff u < min(1, gamma(d) / q(d)) (accepted outright
    when q(d) <= gamma(d), which covers q <= p); the guard, when on, rejects
    first, without a coin, when rank(d) > max_rank (max_rank > 0) or
    p(d) < min_prob. Greedy requests (R2) keep the greedy rule.
R11 The CACTUS residual is not given (its table is lost): after a rejection
    the final token is drawn from norm(max(0, p - q)) as in the lossless rule
    (p itself when that has no mass), the bonus from p_{K+1}.
R12 Position-lazy verification reads, per request, target rows 1..n+1 and
    the draft rows 1..min(n+1, K) a sampling request with dense draft rows
    needs; it returns the same tokens and counts, and p(d), q(d) and the rank
    only for the positions it read (NaN and -1 after them).
R13 Per-position KL(p_i || q_i) = sum_y p(y) ln(p(y) / q(y)), natural log,
    for every draft position of a sampling request, with p and q the laws the
    verifier uses (softmax at the request's temperature; the given or sparse
    draft law): +inf where q has no mass under p's, NaN for greedy requests.
    The second TTS term, KL(q_t || q), compares the drafter before and after
    an update; a verifier sees one draft law, so it is 0 here and not
    reported.

RheoSampling tree construction ("RheoSampling 2026", §2 "Dual-Identity
Decoupling", §3 "Parameter Kendali Rheostat", §7 "Rekomendasi"), one
expansion level of a batch of dynamic trees:

R14 Every frontier row keeps its top-128 logits (R6). Ranking, expansion and
    pruning use q = softmax(z) over them with no temperature (§7, first
    item); the probe is drawn from q~ = softmax(z / T) over the same 128
    (greedy T: one-hot on the argmax), its true sampling law (§2).
R15 Rheostat m: the children of a frontier node, in slot order, are the m
    best tokens by q (the deterministic lead), the probe, then the next best
    tokens up to K children. The deterministic children skip the probe's
    token, so siblings are distinct. The probe's proxy probability is
    q(x_{m+1}) + eps, x_j the j-th best token of the row (ties to the lower
    id): for m = 0 this is the page's q(x_1) + eps, and for every m it ranks
    the probe in slot m+1. eps is the caller's (the page names no value).
    Deterministic children rank by their own q.
R16 A child's path score is ln of the product of proxy probabilities along
    its path: the frontier node's score + ln q_proxy(child). Pruning keeps,
    per tree, the n_keep candidates with the largest scores (ties to the
    lower candidate index f * K + slot), in descending score order.
R17 The probe's uniform is u(seed, f, level, 3): key b = the global frontier
    row f, pos = the expansion level, stream 3; the draw is the inverse CDF
    over q~ in ascending token id (R4).
R18 The deterministic children depend on the probe's token (R15), so a
    verifier of these trees tests the probe first, as "RheoSampling 2026" §4
    step 1 does, and the deterministic children after it as point masses.
R19 Point-mass children ("RheoSampling 2026" §4 steps 1-3 with deterministic
    candidates): a child flagged fixed was not drawn from its parent's draft
    law, so its draft law is the point mass on its token. It is accepted with
    probability min(1, p_j(x) / 1) = p_j(x). On rejection the target law
    becomes norm(max(0, p_j - delta_x)), i.e. p_j without x, renormalised,
    and the draft law of the drawn children is unchanged (without replacement
    runs over drawn children only). Children are still tested in node-index
    order; a tree whose fixed children depend on a drawn sibling's token must
    list that sibling first.
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN_GAMMA = 0x9E3779B97F4A7C15
GREEDY_T = 0.05          # R2
FLAG_EPS = 1e-6          # R8
TOPK = 128               # R6

STREAM_COIN = 0
STREAM_RESIDUAL = 1
STREAM_BONUS = 2
STREAM_PROBE = 3         # R17

RULE_STRICT = 0
RULE_GREEDY = 1
RULE_STRICT_TOP128 = 2
RULE_CACTUS = 3

DRAFT_LOGITS = 0
DRAFT_PROBS = 1
DRAFT_SPARSE128 = 2


# --------------------------------------------------------------------------
# R1: the counter hash
# --------------------------------------------------------------------------
def splitmix64(x: int) -> int:
    """SplitMix64 output function applied to x + gamma (Steele, Lea & Flood,
    "Fast splittable pseudorandom number generators", OOPSLA 2014)."""
    z = (x + GOLDEN_GAMMA) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def hash_key(b: int, pos: int, stream: int) -> int:
    """Pack (request, position, stream) into one 64-bit counter (R1)."""
    assert 0 <= b < (1 << 32) and 0 <= pos < (1 << 24) and 0 <= stream < 256
    return (b << 32) | (pos << 8) | stream


def uniform(seed: int, b: int, pos: int, stream: int) -> float:
    """u in {0, 2^-24, ..., 1 - 2^-24} (R1)."""
    h = splitmix64((seed & MASK64) ^ splitmix64(hash_key(b, pos, stream)))
    return float(h >> 40) * 2.0 ** -24


# --------------------------------------------------------------------------
# Distributions
# --------------------------------------------------------------------------
def as_f64(row) -> np.ndarray:
    """Exact upcast of a bf16/fp32 row (torch tensor or numpy) to float64."""
    if hasattr(row, "detach"):           # a torch tensor
        return row.detach().cpu().double().numpy()
    return np.asarray(row, dtype=np.float64)


def is_greedy(T: float, rule: int) -> bool:
    """R2: greedy when the rule forces it or T < 0.05."""
    return rule == RULE_GREEDY or T < GREEDY_T


def softmax_T(z: np.ndarray, T: float) -> np.ndarray:
    """p = softmax(z / T) over the whole row (RheoSampling 2026, §1 and §7:
    temperature scales the sampling and verification distributions)."""
    z = np.asarray(z, dtype=np.float64)
    m = np.max(z)
    e = np.exp((z - m) / T)
    return e / np.sum(e)


def argmax_lowest(z: np.ndarray) -> int:
    """Greedy choice: the largest logit, lowest id on ties (R2)."""
    return int(np.argmax(z))  # numpy returns the first maximal index


def top128_select(z: np.ndarray, k: int = TOPK) -> np.ndarray:
    """Ids of the k largest logits, ties to the lower id, in ascending id
    order (RheoSampling 2026, §3; R6)."""
    z = np.asarray(z, dtype=np.float64)
    order = np.lexsort((np.arange(z.size), -z))   # by -z, then by id
    return np.sort(order[: min(k, z.size)])


def top128_softmax(z: np.ndarray, T: float, k: int = TOPK):
    """Sparse draft law: softmax(z/T) over the top-k logits, 0 elsewhere.
    Returns (ids ascending, probs). Greedy T gives a one-hot on the argmax
    (R2)."""
    z = np.asarray(z, dtype=np.float64)
    ids = top128_select(z, k)
    if T < GREEDY_T:
        probs = np.zeros(ids.size)
        probs[np.searchsorted(ids, argmax_lowest(z))] = 1.0
        return ids, probs
    return ids, softmax_T(z[ids], T)


def sparse_to_dense(ids: np.ndarray, probs: np.ndarray, V: int) -> np.ndarray:
    q = np.zeros(V, dtype=np.float64)
    keep = ids >= 0
    q[ids[keep]] = probs[keep]
    return q


# --------------------------------------------------------------------------
# Decisions
# --------------------------------------------------------------------------
def acceptance_prob(p_d: float, q_d: float) -> float:
    """a = min(1, p/q) with the outright accept when q <= p ("Acceptance Is
    Not Speed", §6; RheoSampling 2026, §4 step 1; R3)."""
    if q_d <= p_d:
        return 1.0
    return p_d / q_d


def coin_accepts(u: float, a: float) -> bool:
    """R3: strict comparison, so a == 1 always accepts."""
    return u < a


def coin_flagged(u: float, a: float) -> bool:
    return abs(u - a) <= FLAG_EPS


def target_rank(zt: np.ndarray, d: int) -> int:
    """R9: 1 + #{y : z_y > z_d} over the target logits of the position."""
    zt = np.asarray(zt, dtype=np.float64)
    return 1 + int(np.count_nonzero(zt > zt[d]))


def cactus_gamma(p_d: float, alpha: float) -> float:
    """Relaxed target mass of the CACTUS rule ("Acceptance Is Not Speed", §6
    RULE 3): min(p + sqrt(2 alpha p (1 - p)), 1)."""
    return min(p_d + float(np.sqrt(2.0 * alpha * p_d * (1.0 - p_d))), 1.0)


def low_support(p_d: float, rank: int, max_rank: int, min_prob: float) -> bool:
    """Low-support guard ("Acceptance Is Not Speed", §6 RULE 1 and §7 item
    3): reject outright a draft whose target rank exceeds max_rank (when
    max_rank > 0) or whose target probability is below min_prob."""
    return (max_rank > 0 and rank > max_rank) or p_d < min_prob


def kl_divergence(p: np.ndarray, q: np.ndarray) -> float:
    """KL(p || q) in nats over the support of p (R13): terms with p = 0 are
    0; a token with p > 0 and q = 0 makes it +inf."""
    p = np.asarray(p, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    on = p > 0.0
    if np.any(q[on] <= 0.0):
        return float("inf")
    return float(np.sum(p[on] * (np.log(p[on]) - np.log(q[on]))))


def residual(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """Unnormalised residual max(0, p - q) (RheoSampling 2026, §4 step 3)."""
    return np.maximum(0.0, p - q)


def inverse_cdf(w: np.ndarray, u: float):
    """Draw from w / sum(w) at u (R4). Returns (token, flagged)."""
    C = np.cumsum(w)                      # inclusive prefix, ascending id
    Z = C[-1]
    t = u * Z
    x = int(np.searchsorted(C, t, side="right"))   # first x with t < C_x
    if x >= w.size:                       # rounding guard
        x = int(np.nonzero(w > 0)[0][-1])
    flagged = abs(t - C[x]) <= FLAG_EPS * Z
    if x > 0:
        flagged = flagged or abs(t - C[x - 1]) <= FLAG_EPS * Z
    return x, bool(flagged)


def sample_residual_or_p(p: np.ndarray, q: np.ndarray, u: float):
    """Correction draw after a rejection: norm(max(0, p - q)); p itself if
    the residual carries no mass (R4)."""
    r = residual(p, q)
    if not np.sum(r) > 0.0:
        return inverse_cdf(p, u)
    return inverse_cdf(r, u)


# --------------------------------------------------------------------------
# Linear verifier
# --------------------------------------------------------------------------
def _draft_law(draft, draft_kind, draft_idx, row, T, V, rule):
    """q for one draft row: softmax(z/T), given probabilities, or the sparse
    top-128 law (given, or cut here from dense logits under the top-128
    rule)."""
    if draft_kind == DRAFT_PROBS:
        return as_f64(draft[row])
    if draft_kind == DRAFT_SPARSE128:
        ids = np.asarray(draft_idx[row]).astype(np.int64)
        return sparse_to_dense(ids, as_f64(draft[row]), V)
    z = as_f64(draft[row])
    if rule == RULE_STRICT_TOP128:
        ids, probs = top128_softmax(z, T)
        return sparse_to_dense(ids, probs, V)
    return softmax_T(z, T)


def verify_linear(target, draft, draft_tokens, cu_draft, temperature, seed,
                  rule=RULE_STRICT, draft_kind=DRAFT_LOGITS, draft_idx=None,
                  max_k=None, requests=None, alpha=0.0, max_rank=0,
                  min_prob=0.0):
    """One verification round for a batch of requests.

    Request b owns drafts d_1..d_K (K = cu_draft[b+1] - cu_draft[b]), target
    rows p_1..p_{K+1} at rows cu_draft[b] + b + i and draft rows q_1..q_K at
    rows cu_draft[b] + i ("Draft mengubah tebakan serial menjadi batch
    verifikasi": one pass scores K+1 positions, each conditioned on the
    drafts before it).

    Returns a dict with, per processed request: ``tokens`` [n, max_k+1]
    (accepted drafts, then the final token, -1 padded), ``accepted`` [n],
    ``pq`` [R_d, 2] (p(d), q(d) for each draft row; greedy rows give
    (1 or 0, -1)), ``flag_slot`` [n] (first output slot decided by a flagged
    draw, -1 if none) and ``requests`` (the request ids processed).
    ``requests`` restricts the work to a subset (the hash still uses the
    global request id). ``rank`` [R_d] is the target rank of every draft
    token (R9), ``kl`` [R_d] the per-position KL(p || q) (R13). Under ``RULE_CACTUS`` the acceptance test is R10 with
    ``alpha``, ``max_rank`` and ``min_prob``; the final token follows R11.
    """
    cu = np.asarray(cu_draft, dtype=np.int64)
    B = cu.size - 1
    if max_k is None:
        max_k = int(np.max(np.diff(cu))) if B > 0 else 0
    V = target.shape[1]
    req = list(range(B)) if requests is None else [int(b) for b in requests]
    tokens = np.full((len(req), max_k + 1), -1, dtype=np.int64)
    accepted = np.zeros(len(req), dtype=np.int64)
    flag_slot = np.full(len(req), -1, dtype=np.int64)
    R_d = int(cu[-1])
    pq = np.full((R_d, 2), np.nan)
    rank = np.full(R_d, -1, dtype=np.int64)
    kl = np.full(R_d, np.nan)
    toks = np.asarray(draft_tokens, dtype=np.int64)
    temps = np.asarray(temperature, dtype=np.float64)

    for j, b in enumerate(req):
        K = int(cu[b + 1] - cu[b])
        t0, d0 = int(cu[b]) + b, int(cu[b])
        T = float(temps[b])
        greedy = is_greedy(T, rule)
        # per-position p(d), q(d) and the acceptance decisions
        n = K
        flagged_at = -1
        for i in range(K):
            d = int(toks[d0 + i])
            zt = as_f64(target[t0 + i])
            rank[d0 + i] = target_rank(zt, d)
            if greedy:
                ok = d == argmax_lowest(zt)          # "Semantik penerimaan"
                pq[d0 + i] = (1.0 if ok else 0.0, -1.0)
            else:
                p = softmax_T(zt, T)
                q = _draft_law(draft, draft_kind, draft_idx, d0 + i, T, V, rule)
                pq[d0 + i] = (p[d], q[d])
                kl[d0 + i] = kl_divergence(p, q)
                if rule == RULE_CACTUS:
                    a = acceptance_prob(cactus_gamma(p[d], alpha), q[d])
                    guard = low_support(p[d], rank[d0 + i], max_rank, min_prob)
                else:
                    a = acceptance_prob(p[d], q[d])
                    guard = False
                if n == K:   # still scanning: draw this position's coin
                    u = uniform(seed, b, i + 1, STREAM_COIN)
                    if rule == RULE_CACTUS and min_prob > 0.0 \
                            and abs(p[d] - min_prob) <= FLAG_EPS and flagged_at < 0:
                        flagged_at = i
                    if not guard and coin_flagged(u, a) and flagged_at < 0:
                        flagged_at = i
                    ok = not guard and coin_accepts(u, a)
            if n == K and not ok:
                n = i      # first rejection stops the scan ("Penolakan")
        # the final token, from target row n+1
        zt = as_f64(target[t0 + n])
        if greedy:
            final = argmax_lowest(zt)   # the target's choice replaces d_{n+1}
        else:
            p = softmax_T(zt, T)
            if n < K:
                q = _draft_law(draft, draft_kind, draft_idx, d0 + n, T, V, rule)
                u = uniform(seed, b, n + 1, STREAM_RESIDUAL)
                final, fl = sample_residual_or_p(p, q, u)
            else:
                u = uniform(seed, b, K + 1, STREAM_BONUS)
                final, fl = inverse_cdf(p, u)
            if fl and flagged_at < 0:
                flagged_at = n
        tokens[j, :n] = toks[d0:d0 + n]
        tokens[j, n] = final
        accepted[j] = n
        flag_slot[j] = flagged_at
    return dict(tokens=tokens, accepted=accepted, pq=pq, rank=rank, kl=kl,
                flag_slot=flag_slot, requests=np.asarray(req))


def lazy_positions(cu_draft, accepted, requests=None):
    """R12: for each request, the number of draft positions whose target and
    draft rows a position-lazy verifier reads: min(n + 1, K). Rows after the
    first rejection are never used ("Penolakan memendekkan pekerjaan
    speculative": the proposals after a rejected one are not continuations
    of the committed prefix)."""
    cu = np.asarray(cu_draft, dtype=np.int64)
    req = range(cu.size - 1) if requests is None else requests
    return np.array([min(int(n) + 1, int(cu[b + 1] - cu[b]))
                     for b, n in zip(req, accepted)], dtype=np.int64)


def lazy_view(result, cu_draft):
    """The eager result as a position-lazy verifier reports it (R12): p(d),
    q(d) become NaN and the rank -1 on the draft positions it never read."""
    cu = np.asarray(cu_draft, dtype=np.int64)
    out = dict(result)
    pq = np.array(result["pq"], dtype=np.float64, copy=True)
    rank = np.array(result["rank"], copy=True)
    kl = np.array(result["kl"], dtype=np.float64, copy=True)
    req = result["requests"]
    for b, m in zip(req, lazy_positions(cu, result["accepted"], req)):
        d0, d1 = int(cu[b]), int(cu[b + 1])
        pq[d0 + m:d1] = np.nan
        rank[d0 + m:d1] = -1
        kl[d0 + m:d1] = np.nan
    out["pq"], out["rank"], out["kl"] = pq, rank, kl
    return out


# --------------------------------------------------------------------------
# Tree verifier (RRSw)
# --------------------------------------------------------------------------
def children_of(parent: np.ndarray, v: int):
    """Children of v in node-index order (= the order they were drawn)."""
    return [int(c) for c in np.nonzero(np.asarray(parent) == v)[0]]


def rrsw_node(p, q, child_tokens, coins, fixed=None):
    """Recursive rejection sampling without replacement at one node
    (RheoSampling 2026, §4; R7, R19).

    p, q: the node's target and draft laws. child_tokens: the children's
    tokens in the order they were drawn. coins: one uniform per child.
    fixed: optional flags, one per child; a fixed child is a point mass on
    its token (R19). Returns (index of the accepted child or -1, the law to
    sample when all are rejected (unnormalised), list of (u, a) pairs that
    were tested).
    """
    p_j = np.asarray(p, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    excluded = np.zeros(q.size, dtype=bool)
    q_j = q.copy()
    tested = []
    for j, x in enumerate(child_tokens):
        if fixed is not None and fixed[j]:
            # point mass: accept with min(1, p_j(x) / 1); on rejection the
            # residual max(0, p_j - delta_x) is p_j without x
            a = acceptance_prob(p_j[x], 1.0)
            tested.append((coins[j], a))
            if coin_accepts(coins[j], a):
                return j, None, tested
            r = np.maximum(0.0, p_j - (np.arange(p_j.size) == x))
            Z = np.sum(r)
            if Z > 0.0:
                p_j = r / Z
            continue
        a = acceptance_prob(p_j[x], q_j[x])
        tested.append((coins[j], a))
        if coin_accepts(coins[j], a):
            return j, None, tested
        # rejection: p <- norm(max(0, p - q)); q <- q without the drawn
        # tokens, renormalised by 1 - q(E)
        r = residual(p_j, q_j)
        Z = np.sum(r)
        if Z > 0.0:
            p_j = r / Z
        excluded[x] = True
        mass_left = 1.0 - np.sum(q[excluded])
        if not mass_left > 0.0:
            return -1, p_j, tested      # every draft token used up
        q_j = np.where(excluded, 0.0, q) / mass_left
    return -1, p_j, tested


def verify_tree(target, draft, node_token, parent, cu_nodes, temperature,
                seed, max_depth, rule=RULE_STRICT, requests=None,
                draft_kind=DRAFT_LOGITS, node_fixed=None):
    """Multi-draft tree verification by RRSw.

    Request b owns nodes cu_nodes[b] .. cu_nodes[b+1]-1; local node 0 is the
    root. parent[] holds local parent ids (-1 for the root), topologically
    ordered. Target row n is the target law after the path to node n; draft
    row n is the law node n's children were drawn from: logits (q =
    softmax(z/T)) or, with draft_kind == DRAFT_PROBS, the probabilities
    themselves. node_fixed[n] != 0 marks node n as a point-mass child (R19).

    Returns tokens [n, max_depth+1], accepted [n], path [n, max_depth+1]
    (local node ids of accepted nodes), flag_slot [n], requests.
    """
    cu = np.asarray(cu_nodes, dtype=np.int64)
    B = cu.size - 1
    req = list(range(B)) if requests is None else [int(b) for b in requests]
    W = max_depth + 1
    tokens = np.full((len(req), W), -1, dtype=np.int64)
    path = np.full((len(req), W), -1, dtype=np.int64)
    accepted = np.zeros(len(req), dtype=np.int64)
    flag_slot = np.full(len(req), -1, dtype=np.int64)
    ntok = np.asarray(node_token, dtype=np.int64)
    par = np.asarray(parent, dtype=np.int64)
    temps = np.asarray(temperature, dtype=np.float64)

    for j, b in enumerate(req):
        base, N = int(cu[b]), int(cu[b + 1] - cu[b])
        lpar = par[base:base + N]
        T = float(temps[b])
        greedy = is_greedy(T, rule)
        v, depth, flagged_at = 0, 0, -1
        while True:
            kids = children_of(lpar, v)
            zt = as_f64(target[base + v])
            if greedy:
                g = argmax_lowest(zt)
                hit = [c for c in kids if ntok[base + c] == g]
                if hit:
                    v = hit[0]
                    path[j, depth] = v
                    tokens[j, depth] = ntok[base + v]
                    depth += 1
                    continue
                tokens[j, depth] = g
                break
            p = softmax_T(zt, T)
            if not kids:                       # accepted leaf: bonus draw
                u = uniform(seed, b, v + 1, STREAM_BONUS)
                x, fl = inverse_cdf(p, u)
                if fl and flagged_at < 0:
                    flagged_at = depth
                tokens[j, depth] = x
                break
            if draft_kind == DRAFT_PROBS:
                q = as_f64(draft[base + v])
            else:
                q = softmax_T(as_f64(draft[base + v]), T)
            coins = [uniform(seed, b, c, STREAM_COIN) for c in kids]
            fx = None if node_fixed is None else [bool(node_fixed[base + c]) for c in kids]
            acc, law, tested = rrsw_node(p, q, [ntok[base + c] for c in kids],
                                         coins, fx)
            if flagged_at < 0 and any(coin_flagged(u, a) for u, a in tested):
                flagged_at = depth
            if acc >= 0:
                v = kids[acc]
                path[j, depth] = v
                tokens[j, depth] = ntok[base + v]
                depth += 1
                continue
            u = uniform(seed, b, v + 1, STREAM_RESIDUAL)
            x, fl = inverse_cdf(law, u)
            if fl and flagged_at < 0:
                flagged_at = depth
            tokens[j, depth] = x
            break
        accepted[j] = depth
        flag_slot[j] = flagged_at
        if depth > max_depth:
            raise ValueError("tree deeper than max_depth")
    return dict(tokens=tokens, accepted=accepted, path=path,
                flag_slot=flag_slot, requests=np.asarray(req))


# --------------------------------------------------------------------------
# Top-128 over a batch of rows
# --------------------------------------------------------------------------
def draft_topk_softmax(draft_logits, cu_rows, temperature, k=TOPK):
    """Per draft row: ids of the top-k logits (ascending id, -1 padded when
    V < k) and softmax(z/T) over them (RheoSampling 2026, §3; R6)."""
    cu = np.asarray(cu_rows, dtype=np.int64)
    R = int(cu[-1])
    idx = np.full((R, k), -1, dtype=np.int64)
    prob = np.zeros((R, k), dtype=np.float64)
    temps = np.asarray(temperature, dtype=np.float64)
    for b in range(cu.size - 1):
        for r in range(int(cu[b]), int(cu[b + 1])):
            ids, probs = top128_softmax(as_f64(draft_logits[r]),
                                        float(temps[b]), k)
            idx[r, :ids.size] = ids
            prob[r, :ids.size] = probs
    return idx, prob


# --------------------------------------------------------------------------
# RheoSampling tree construction, one expansion level (R14-R18)
# --------------------------------------------------------------------------
def rheo_ranking_order(z: np.ndarray, k: int = TOPK) -> np.ndarray:
    """The row's top-k token ids from best to worst: logit descending, ties
    to the lower id ("RheoSampling 2026", §3; R6, R15)."""
    z = np.asarray(z, dtype=np.float64)
    order = np.lexsort((np.arange(z.size), -z))
    return order[: min(k, z.size)]


def rheo_ranking_law(z: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """q over the surviving ids with no temperature ("RheoSampling 2026", §7:
    tree expansion and ranking run on the unscaled draft law; R14)."""
    zs = np.asarray(z, dtype=np.float64)[ids]
    e = np.exp(zs - np.max(zs))
    return e / np.sum(e)


def rheo_slots(order: np.ndarray, probe: int, K: int, m: int) -> list:
    """Children in slot order: the m best tokens other than the probe, the
    probe, then the next best up to K children (§3 rheostat; R15)."""
    det = [int(x) for x in order if int(x) != probe][: K - 1]
    return det[:m] + [probe] + det[m:]


def rheo_probe_proxy(q_by_rank: np.ndarray, m: int, eps: float) -> float:
    """q_proxy of the probe: q(x_{m+1}) + eps, x ranked best first (§3: m = 0
    gives q(x_1) + eps; R15). Beyond the last survivor it is eps."""
    return (float(q_by_rank[m]) if m < q_by_rank.size else 0.0) + eps


def rheo_select(scores: np.ndarray, n_keep: int) -> np.ndarray:
    """Pruning: indices of the n_keep largest scores, descending, ties to the
    lower index, -1 padded (§2 global pruning; R16)."""
    scores = np.asarray(scores, dtype=np.float64)
    order = np.lexsort((np.arange(scores.size), -scores))
    out = np.full(n_keep, -1, dtype=np.int64)
    take = order[:n_keep]
    out[: take.size] = take
    return out


def rheo_expand(draft, cu_frontier, frontier_score, temperature, seed, level,
                K, m, eps, n_keep):
    """One level of RheoSampling dynamic-tree expansion for a batch of trees.

    draft [F, V] logits: row f is the draft model's output at frontier node
    f; tree b owns rows cu_frontier[b] .. cu_frontier[b+1]-1.
    frontier_score [F]: ln of each frontier node's path score (0 at a root).
    Returns child_token, child_qproxy, child_qtrue, child_score (each
    [F, K], slot order of R15), keep [B, n_keep] (candidate ids f * K +
    slot, R16) and probe_flag [F] (the probe draw sat within R8's margin of
    a CDF boundary).
    """
    cu = np.asarray(cu_frontier, dtype=np.int64)
    B, F = cu.size - 1, int(cu[-1])
    temps = np.asarray(temperature, dtype=np.float64)
    fscore = np.asarray(frontier_score, dtype=np.float64)
    token = np.full((F, K), -1, dtype=np.int64)
    qproxy = np.zeros((F, K))
    qtrue = np.zeros((F, K))
    score = np.full((F, K), -np.inf)
    flag = np.zeros(F, dtype=bool)
    for b in range(B):
        T = float(temps[b])
        for f in range(int(cu[b]), int(cu[b + 1])):
            z = as_f64(draft[f])
            order = rheo_ranking_order(z)                # R14: top-128, best first
            ids = np.sort(order)                         # ascending id
            q = rheo_ranking_law(z, ids)                 # unscaled, by ascending id
            q_of = dict(zip(ids.tolist(), q.tolist()))
            _, qt = top128_softmax(z, T)                 # q~, by ascending id
            qt_of = dict(zip(ids.tolist(), qt.tolist()))
            u = uniform(seed, f, level, STREAM_PROBE)    # R17
            j, fl = inverse_cdf(qt, u)
            probe = int(ids[j])
            flag[f] = fl
            slots = rheo_slots(order, probe, K, m)       # R15
            q_rank = np.array([q_of[int(x)] for x in order])
            for s, x in enumerate(slots):
                pr = rheo_probe_proxy(q_rank, m, eps) if x == probe else q_of[x]
                token[f, s] = x
                qproxy[f, s] = pr
                qtrue[f, s] = qt_of[x]
                score[f, s] = fscore[f] + np.log(pr)     # R16
    keep = np.full((B, n_keep), -1, dtype=np.int64)
    for b in range(B):
        lo, hi = int(cu[b]) * K, int(cu[b + 1]) * K
        sel = rheo_select(score.reshape(-1)[lo:hi], n_keep)
        keep[b] = np.where(sel >= 0, sel + lo, -1)
    return dict(child_token=token, child_qproxy=qproxy, child_qtrue=qtrue,
                child_score=score, keep=keep, probe_flag=flag)

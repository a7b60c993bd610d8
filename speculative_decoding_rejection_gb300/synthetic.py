"""Seeded synthetic verifier workloads.

This module only builds inputs: logits, draft tokens, ragged offsets, trees
and temperatures. It holds none of the verifier's arithmetic (no acceptance
rule, no residual, no inverse CDF), so both the CUDA path and the CPU oracle
can take their inputs from it.

Recipe (the pages run on real models and public datasets; these synthetic
rows stand in for them):

* target logits  z_t = 2.0 * N(0, 1) - 1.1 * ln(rank), where rank is a
  uniform random permutation of 1..V drawn once per request and shared by that
  request's rows (a Zipf-like long tail);
* draft logits   z_d = z_t + sigma * N(0, 1), row i of the draft matching
  target row i (the draft's guess for the same position);
* both rounded to the storage dtype (bf16 round-to-nearest-even, or fp32);
* stochastic drafts d_i are drawn from softmax(z_d / T) (Gumbel-max), from
  the top-128 of z_d when the workload truncates the draft; greedy drafts are
  argmax z_d;
* trees: node 0 is the root; each new node picks its parent uniformly among
  nodes of depth < max_depth with fewer than max_branch children; the
  children of a node carry tokens drawn without replacement from that node's
  draft law, in node-index order (Gumbel-top-k);
* tree-expansion frontiers: W draft rows per tree with the draft logit
  recipe above (one Zipf permutation per tree), and ln path scores uniform
  in [-3 * level, 0] (0 at level 0, where each tree's frontier is its root).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

INPUT_SEED_BASE = 0x5EED0000
VERIFY_SEED_BASE = 0x243F6A8885A308D3

GREEDY_T = 0.05
TOPK = 128

# Named workloads. "sigma" / "T" may be a float, a list (per request), a
# ("uniform", lo, hi) tuple drawn per request, or ("halves", a, b): the first
# half of the requests get a, the rest b.
WORKLOADS = {
    1: dict(name="linear-strict-B4-K4-V1024-f32", kind="linear", B=4, K=4,
            V=1024, dtype="f32", sigma=0.5, T=1.0, top128=False),
    2: dict(name="linear-mixed-B64-K1..5-V32000-bf16", kind="linear", B=64,
            K=(1, 5), V=32000, dtype="bf16", sigma=0.7,
            T=("halves", 0.0, 0.7), top128=False),
    3: dict(name="linear-top128-B256-K7-V151936-bf16", kind="linear", B=256,
            K=7, V=151936, dtype="bf16", sigma=0.5, T=1.0, top128=True),
    4: dict(name="tree-rrsw-B32-N64-D6-W4-V128256-bf16", kind="tree", B=32,
            N=64, depth=6, branch=4, V=128256, dtype="bf16", sigma=0.6,
            T=0.8),
    5: dict(name="linear-large-B1024-K4-V201088-bf16", kind="linear", B=1024,
            K=4, V=201088, dtype="bf16", sigma=("uniform", 0.3, 1.5),
            T=("uniform", 0.0, 1.2), top128=False),
}

_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def _per_request(spec, B, g, device):
    if isinstance(spec, (int, float)):
        return torch.full((B,), float(spec), dtype=torch.float32)
    if isinstance(spec, tuple) and spec[0] == "halves":
        return torch.tensor([spec[1]] * (B // 2) + [spec[2]] * (B - B // 2),
                            dtype=torch.float32)
    if isinstance(spec, tuple) and spec[0] == "uniform":
        lo, hi = spec[1], spec[2]
        return lo + (hi - lo) * torch.rand(B, generator=g, device=device).cpu()
    vals = torch.tensor([float(x) for x in spec], dtype=torch.float32)
    assert vals.numel() == B, "per-request list must have B entries"
    return vals


def _zipf_bias(B, V, g, device):
    """-1.1 * ln(rank) with rank a random permutation of 1..V per request."""
    bias = torch.empty(B, V, dtype=torch.float32, device=device)
    for b in range(B):
        rank = torch.randperm(V, generator=g, device=device).to(torch.float32) + 1.0
        bias[b] = -1.1 * torch.log(rank)
    return bias


def _gumbel(shape, g, device):
    u = torch.rand(shape, generator=g, device=device).clamp_(1e-12, 1.0 - 1e-7)
    return -torch.log(-torch.log(u))


@dataclass
class LinearBatch:
    target: torch.Tensor          # [R_t, V]
    draft: torch.Tensor           # [R_d, V]
    draft_tokens: torch.Tensor    # [R_d] int32
    cu_draft: torch.Tensor        # [B+1] int32
    temperature: torch.Tensor     # [B] float32
    max_k: int
    seed: int
    top128: bool
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.cu_draft.numel() - 1

    @property
    def V(self):
        return self.target.shape[1]


@dataclass
class TreeBatch:
    target: torch.Tensor          # [N_tot, V]
    draft: torch.Tensor           # [N_tot, V]
    node_token: torch.Tensor      # [N_tot] int32, -1 at roots
    parent: torch.Tensor          # [N_tot] int32, local ids, -1 at roots
    cu_nodes: torch.Tensor        # [B+1] int32
    temperature: torch.Tensor     # [B] float32
    max_depth: int
    max_branch: int
    seed: int
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.cu_nodes.numel() - 1

    @property
    def V(self):
        return self.target.shape[1]


def workload(cfg: int, **overrides) -> dict:
    w = dict(WORKLOADS[cfg])
    w.update(overrides)
    return w


def make_linear(cfg: int = 1, device="cpu", input_seed=None, **overrides) -> LinearBatch:
    """Build a linear-verify batch for workload ``cfg`` (fields overridable:
    B, K, V, dtype, sigma, T, top128)."""
    w = workload(cfg, **overrides)
    assert w["kind"] == "linear"
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(INPUT_SEED_BASE + cfg if input_seed is None else input_seed)
    B, V = w["B"], w["V"]
    if isinstance(w["K"], tuple):
        lo, hi = w["K"]
        K = torch.randint(lo, hi + 1, (B,), generator=g, device=device).cpu()
    else:
        K = torch.full((B,), int(w["K"]), dtype=torch.int64)
    cu = torch.zeros(B + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(K, 0)
    R_d = int(cu[-1])
    R_t = R_d + B
    T = _per_request(w["T"], B, g, device)
    sigma = _per_request(w["sigma"], B, g, device)
    bias = _zipf_bias(B, V, g, device)
    dt = _DTYPES[w["dtype"]]

    t_req = torch.repeat_interleave(torch.arange(B), K + 1).to(device)
    d_req = torch.repeat_interleave(torch.arange(B), K).to(device)
    zt32 = 2.0 * torch.randn(R_t, V, generator=g, device=device) + bias[t_req]
    # draft row r of request b pairs with target row r + b
    t_of_d = torch.arange(R_d, device=device) + d_req
    zd32 = zt32[t_of_d] + sigma.to(device)[d_req, None] * torch.randn(
        R_d, V, generator=g, device=device)
    del bias
    target = zt32.to(dt)
    del zt32
    draft = zd32.to(dt)
    del zd32

    # draft tokens: greedy -> argmax; otherwise Gumbel-max at temperature T
    tokens = torch.empty(R_d, dtype=torch.int64, device=device)
    Td = T.to(device)[d_req]
    chunk = max(1, (1 << 28) // max(V, 1))
    for s in range(0, R_d, chunk):
        e = min(R_d, s + chunk)
        z = draft[s:e].to(torch.float32)
        Tc = Td[s:e]
        greedy = Tc < GREEDY_T
        if w.get("top128"):
            k = min(TOPK, V)
            keep = torch.zeros_like(z, dtype=torch.bool)
            keep.scatter_(1, torch.topk(z, k, dim=1).indices, True)
            z = torch.where(keep, z, torch.full_like(z, -math.inf))
        scores = z / torch.where(greedy, torch.ones_like(Tc), Tc)[:, None]
        scores = scores + _gumbel(z.shape, g, device)
        samp = torch.argmax(scores, dim=1)
        tokens[s:e] = torch.where(greedy, torch.argmax(z, dim=1), samp)
    return LinearBatch(target=target, draft=draft,
                       draft_tokens=tokens.to(torch.int32),
                       cu_draft=cu.to(torch.int32).to(device),
                       temperature=T.to(device), max_k=int(K.max()) if B else 0,
                       seed=VERIFY_SEED_BASE + cfg, top128=bool(w.get("top128")),
                       meta=dict(workload=w["name"] if not overrides else
                                 f"{w['name']}+{sorted(overrides.items())}",
                                 cfg=cfg, **{k: v for k, v in w.items()
                                             if k in ("B", "V", "dtype")}))


def _random_tree(N, max_depth, max_branch, g):
    parent = [-1]
    depth = [0]
    nkids = [0]
    for _ in range(1, N):
        cand = [v for v in range(len(parent))
                if depth[v] < max_depth and nkids[v] < max_branch]
        v = cand[int(torch.randint(len(cand), (1,), generator=g))]
        parent.append(v)
        depth.append(depth[v] + 1)
        nkids.append(0)
        nkids[v] += 1
    return parent


def make_tree(cfg: int = 4, device="cpu", input_seed=None, **overrides) -> TreeBatch:
    """Build a tree-verify batch (fields overridable: B, N, depth, branch, V,
    dtype, sigma, T)."""
    w = workload(cfg, **overrides)
    assert w["kind"] == "tree"
    device = torch.device(device)
    seed = INPUT_SEED_BASE + cfg if input_seed is None else input_seed
    gcpu = torch.Generator().manual_seed(seed)
    g = torch.Generator(device=device)
    g.manual_seed(seed + 1)
    B, N, V = w["B"], w["N"], w["V"]
    parents = [_random_tree(N, w["depth"], w["branch"], gcpu) for _ in range(B)]
    T = _per_request(w["T"], B, gcpu, "cpu")
    sigma = _per_request(w["sigma"], B, gcpu, "cpu")
    bias = _zipf_bias(B, V, g, device)
    dt = _DTYPES[w["dtype"]]
    req = torch.repeat_interleave(torch.arange(B), N).to(device)
    zt32 = 2.0 * torch.randn(B * N, V, generator=g, device=device) + bias[req]
    zd32 = zt32 + sigma.to(device)[req, None] * torch.randn(
        B * N, V, generator=g, device=device)
    target, draft = zt32.to(dt), zd32.to(dt)
    del zt32, zd32, bias

    tokens = torch.full((B * N,), -1, dtype=torch.int64)
    for b in range(B):
        par = parents[b]
        greedy = float(T[b]) < GREEDY_T
        for v in range(N):
            kids = [c for c in range(N) if par[c] == v]
            if not kids:
                continue
            z = draft[b * N + v].to(torch.float32)
            if greedy:
                order = torch.argsort(z, descending=True, stable=True)
            else:
                order = torch.argsort(z / float(T[b]) + _gumbel(z.shape, g, device),
                                      descending=True)
            for j, c in enumerate(kids):
                tokens[b * N + c] = int(order[j])
    cu = torch.arange(0, B * N + 1, N, dtype=torch.int32)
    parent = torch.tensor([p for par in parents for p in par], dtype=torch.int32)
    return TreeBatch(target=target, draft=draft,
                     node_token=tokens.to(torch.int32).to(device),
                     parent=parent.to(device), cu_nodes=cu.to(device),
                     temperature=T.to(device), max_depth=w["depth"],
                     max_branch=w["branch"], seed=VERIFY_SEED_BASE + cfg,
                     meta=dict(workload=w["name"], cfg=cfg, B=B, V=V,
                               dtype=w["dtype"]))


# One level of dynamic-tree expansion on the setting "RheoSampling 2026" §5
# measures on (EAGLE-3 trees, temperature 1.0, Llama-3.1's 128256-token
# vocabulary): 64 trees, 10 frontier nodes each, 10 children per node,
# rheostat m = 1 (the page's recommended value), 10 nodes kept per tree.
RHEO_WORKLOAD = dict(name="rheo-expand-B64-W10-K10-m1-V128256-bf16", B=64, W=10, K=10, m=1,
                     n_keep=10, V=128256, dtype="bf16", T=1.0, level=3, eps=1e-6)


@dataclass
class RheoBatch:
    draft: torch.Tensor           # [F, V] draft logits of the frontier nodes
    cu_frontier: torch.Tensor     # [B+1] int32
    frontier_score: torch.Tensor  # [F] float32, ln path score
    temperature: torch.Tensor     # [B] float32
    K: int
    m: int
    n_keep: int
    eps: float
    level: int
    seed: int
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.cu_frontier.numel() - 1

    @property
    def V(self):
        return self.draft.shape[1]


def make_rheo(device="cpu", input_seed=None, **overrides) -> RheoBatch:
    """Frontier rows for one expansion level (fields overridable: B, W (an
    int or a (lo, hi) range per tree), K, m, n_keep, V, dtype, T, level,
    eps)."""
    w = dict(RHEO_WORKLOAD)
    w.update(overrides)
    device = torch.device(device)
    seed = INPUT_SEED_BASE + 0x100 if input_seed is None else input_seed
    gcpu = torch.Generator().manual_seed(seed)
    g = torch.Generator(device=device)
    g.manual_seed(seed + 1)
    B, V = w["B"], w["V"]
    if isinstance(w["W"], tuple):
        lo, hi = w["W"]
        W = torch.randint(lo, hi + 1, (B,), generator=gcpu)
    else:
        W = torch.full((B,), int(w["W"]), dtype=torch.int64)
    cu = torch.zeros(B + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(W, 0)
    F = int(cu[-1])
    T = _per_request(w["T"], B, gcpu, "cpu")
    bias = _zipf_bias(B, V, g, device)
    req = torch.repeat_interleave(torch.arange(B), W).to(device)
    z = 2.0 * torch.randn(F, V, generator=g, device=device) + bias[req]
    draft = z.to(_DTYPES[w["dtype"]])
    del z, bias
    level = int(w["level"])
    score = -3.0 * level * torch.rand(F, generator=gcpu)
    return RheoBatch(draft=draft, cu_frontier=cu.to(torch.int32).to(device),
                     frontier_score=score.to(torch.float32).to(device),
                     temperature=T.to(device), K=int(w["K"]), m=int(w["m"]),
                     n_keep=int(w["n_keep"]), eps=float(w["eps"]), level=level,
                     seed=VERIFY_SEED_BASE + 0x100,
                     meta=dict(workload=w["name"] if not overrides else
                               f"{w['name']}+{sorted(overrides.items())}",
                               B=B, V=V, dtype=w["dtype"]))

#!/usr/bin/env python
"""Throughput of the batched speculative-decoding verifier on GB300.

A step is one verification call over one batch of synthetic requests. The
default workload is B=1024 requests x K=4 drafts, V=201088, bf16 target and
draft logits, per-request T ~ U[0, 1.2] (greedy below 0.05): one
spec_verify_linear call per step. The headline value is verified draft
positions per second (draft positions in the batch / step time); the JSON
line also carries the achieved HBM bandwidth of the dominant kernel (the
row-statistics pass) against the measured copy peak, an end-to-end number
through the same C ABI with host buffers, and the CPU oracle timed on a
bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--config 1|2|3|4|5]

--config 3 is the top-128 truncation workload, --config 4 the tree (RRSw)
workload (spec_verify_tree; positions = draft nodes). Workloads whose call
reads less than twice the L2 (configs 1, 2 and 4) write twice the L2 before
every call, outside the call's timing. Under torchrun each rank
verifies its own batch (weak scaling, no data-path collective); rank 0 prints
the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("verified draft positions/sec and achieved HBM GB/s (% of GB300 peak), 1 GPU")
UNIT = "positions/s"
FALLBACK_HBM_GBS = 6800.0

# DRAM traffic of the row pass per algorithmic byte, from an ncu capture of
# a smaller case of the same kernel (dram__bytes_read.sum +
# dram__bytes_write.sum over the algorithmic bytes it streams). Each figure
# below is valid only for the sources it was taken on (KERNEL_SOURCES).
# Captured on B=128, K=4, V=201088 bf16 (460.09 MB streamed by the launch):
# 460.19 MB read + 3.43 MB written (the per-chunk partial statistics).
ROWPASS_TRAFFIC = {"source_sha1": "6f64b6019569898dcbfb786b84f81e6a98e4f7e3",
                   "dram_per_algorithmic_byte": (460192768 + 3425280) / 460089344}
# The same for the streaming verifier (position-lazy schedule), per byte of
# the rows the schedule must read (target rows 1..n+1, dense draft rows
# 1..min(n+1, K) of sampling requests). Captured on the full B=1024, K=4,
# V=201088 workload (one pass): 2708.1 MB read + 23.3 MB written for
# 1975.1 MB; the excess is the residual rows read a second time and rows
# read before a rejection made them unneeded, so the ratio holds for this
# workload and source only.
STREAM_TRAFFIC = {"source_sha1": "5017700c1d26c56531cf5112684a963d1e4d8325",
                  "dram_per_algorithmic_byte": (2708053248 + 23286528) / 1975086336}
# The top-128 select (two passes, the second mostly from L2), per byte of
# the draft rows; captured on the full B=256, K=7, V=151936 workload (one
# pass): 556.56 MB read + 4.54 MB written for 544.54 MB. Valid for these
# sources and this workload.
TOPK_TRAFFIC = {"source_sha1": "e8249b1d1907a23dfa3f849dc81e33617e583623",
                "dram_per_algorithmic_byte": (556563456 + 4540928) / 544538624}
# The top-128 select with its construction epilogue on the construction
# workload (640 frontier rows, V = 128256 bf16; L2 flushed before the call):
# 164.55 MB read + 3.21 MB written for 164.17 MB (most of the write is
# dirty lines of the L2 flush buffer, written back as the rows evict them).
# Valid for these sources and workload.
RHEO_TRAFFIC = {"source_sha1": "e8249b1d1907a23dfa3f849dc81e33617e583623",
                "dram_per_algorithmic_byte": (164545024 + 3206912) / 164167680}
# The tree walk (no row pass: only visited nodes' rows), per byte of those
# rows' first read; captured on the full 32-tree workload (one pass): 63.30 MB
# read + 0.49 MB written for 59.25 MB. Valid for these sources and workload.
TREE_TRAFFIC = {"source_sha1": "0a249bdc0ac97606bbfcbb25420fbb6d07129a26",
                "dram_per_algorithmic_byte": (63298560 + 493056) / 59254272}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", type=int, default=5, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--V", type=int, default=None,
                    help="linear workloads: override the vocabulary size (size sweeps)")
    ap.add_argument("--B", type=int, default=None,
                    help="override the number of requests (small profiling cases)")
    ap.add_argument("--e2e-steps", type=int, default=6)
    ap.add_argument("--cpu-requests", type=int, default=1024,
                    help="requests (or trees) in the oracle's timed sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kl", action="store_true",
                    help="linear workloads: also emit the per-position KL(p || q)")
    ap.add_argument("--lazy", action="store_true",
                    help="linear workloads: position-lazy verification (rows 1..n+1 only)")
    ap.add_argument("--rule", default="default", choices=["default", "cactus"],
                    help="linear workloads: the workload's lossless rule, or the relaxed "
                         "CACTUS rule with the recommended low-support guard")
    ap.add_argument("--rheo", action="store_true",
                    help="time one level of RheoSampling tree construction (spec_rheo_expand) "
                         "on its own workload instead of a verify workload")
    ap.add_argument("--fused-limit", type=int, default=None,
                    help="linear workloads: largest call (bytes of rows) the fused small-batch "
                         "kernel takes; 0 forces the multi-kernel schedule")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


# Every source a kernel is compiled from: a traffic figure holds only while
# all of them are unchanged.
KERNEL_SOURCES = {
    "rowpass": ("rowpass.cu", "rowpass.cuh", "common.cuh", "internal.h"),
    "stream": ("stream.cu", "linear.cuh", "rowpass.cuh", "common.cuh", "internal.h"),
    "topk": ("topk.cu", "common.cuh", "internal.h"),
    "tree": ("tree.cu", "common.cuh", "internal.h"),
}


def source_sha1(kernel):
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "speculative_decoding_rejection_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    with open(os.path.join(ROOT, "include", "specverify.h"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (read only)."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for name, v in zip(self.NAMES, f[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- workloads
class LinearWork:
    """spec_verify_linear on a linear workload (configs 1, 2, 3, 5)."""
    unit_name = "requests"

    # relaxed rule options: the guard the page recommends (p >= 0.10, top 10)
    CACTUS = {"alpha": 0.5, "max_rank": 10, "min_prob": 0.10}

    def __init__(self, cfg, dev, input_seed=None, B=None, rule=None, lazy=False, kl=False,
                 V=None):
        import torch
        import speculative_decoding_rejection_gb300 as sv
        from speculative_decoding_rejection_gb300 import synthetic as S
        self.sv = sv
        over = {} if B is None else {"B": B}
        if V is not None:
            over["V"] = V
        self.lb = lb = S.make_linear(cfg, device=dev, input_seed=input_seed, **over)
        self.rule = sv.SPEC_RULE_STRICT_TOP128 if lb.top128 else sv.SPEC_RULE_STRICT
        self.ext = None
        if rule == "cactus":
            self.rule, self.ext = sv.SPEC_RULE_CACTUS, dict(self.CACTUS)
        self.lazy = lazy
        self.kl = (torch.empty(lb.draft_tokens.numel(), dtype=torch.float32, device=dev)
                   if kl else None)
        K = torch.diff(lb.cu_draft.cpu().long())
        samp = lb.temperature.cpu() >= 0.05
        self.positions = int(K.sum())
        self.tgt_bytes = int((K + 1).sum()) * lb.V * lb.target.element_size()
        self.drf_bytes = int(K[samp].sum()) * lb.V * lb.draft.element_size()
        # the dominant kernel's bytes: the row pass reads the target rows and
        # the dense draft rows of sampling requests; under truncation the
        # top-128 select, which then dominates, reads every draft row
        self.rowpass_bytes = (lb.draft.numel() * lb.draft.element_size() if lb.top128
                              else self.tgt_bytes + self.drf_bytes)
        if lb.top128:
            self.kernel = "k_topk128"
        # setup, row pass, accept, final draws, + the residual sums (dense
        # drafts) or the top-128 select (truncation); the header memset is
        # not ours
        self.launches = 5
        self.outs = (torch.empty(lb.B, lb.max_k + 1, dtype=torch.int32, device=dev),
                     torch.empty(lb.B, dtype=torch.int32, device=dev), None)
        self.ws = torch.empty(sv.spec_verify_linear_workspace(lb.B, lb.max_k, lb.V, self.rule),
                              dtype=torch.uint8, device=dev)
        self.config = {"workload": lb.meta["workload"], "B": lb.B, "K": lb.max_k, "V": lb.V,
                       "logits": "bf16" if lb.target.element_size() == 2 else "f32",
                       "rule": "strict_top128" if lb.top128 else "strict"}
        if self.ext is not None:
            self.config["rule"] = ("cactus(alpha={alpha},max_rank={max_rank},"
                                   "min_prob={min_prob})".format(**self.ext))
        if kl:
            self.config["outputs"] = "tokens, counts and per-position KL(p || q)"
        # the position-lazy schedule of dense bf16 logits (V % 8 == 0, no KL)
        # runs as one persistent kernel: setup, streaming verifier, final draws
        self.stream = (lazy and not lb.top128 and not kl and lb.V % 8 == 0
                       and lb.target.dtype == torch.bfloat16)
        if lazy:
            self.config["schedule"] = "position-lazy (rows 1..n+1 per request)"
            # rounds: a row pass and a decision launch per position; around
            # them the setup, the top-128 select or the residual sums, and
            # the final draws
            self.launches = 3 if self.stream else 3 + 2 * (lb.max_k + 1)
        # small calls of the strict or greedy rule on dense logits or
        # probabilities run as one fused kernel (the library's own test:
        # rows of at most 8192 logits, at most 1 MiB of rows per request and
        # the fused limit in all)
        limit = sv.spec_set_fused_limit(0)
        sv.spec_set_fused_limit(limit)
        esz = lb.target.element_size()
        per_req = (lb.max_k + 1) * lb.V * esz + lb.max_k * lb.V * lb.draft.element_size()
        self.fused = (not lazy and not kl and self.ext is None and not lb.top128
                      and lb.V <= 8192 and per_req <= 1 << 20 and lb.B * per_req <= limit)
        if self.fused:
            self.launches = 1
            self.kernel = "k_verify_small"
            self.config["schedule"] = "fused (one block per request)"

    def input_tensors(self):
        lb = self.lb
        return {"target": lb.target, "draft": lb.draft, "draft_tokens": lb.draft_tokens,
                "cu_draft": lb.cu_draft, "temperature": lb.temperature}

    def call(self, inputs=None):
        lb = self.lb
        t = inputs or self.input_tensors()
        if self.ext is not None or self.lazy or self.kl is not None:
            self.sv.spec_verify_linear_ext(t["target"], t["draft"], t["draft_tokens"],
                                           t["cu_draft"], t["temperature"], lb.seed,
                                           max_k=lb.max_k, rule=self.rule, workspace=self.ws,
                                           out=self.outs + (None, self.kl), lazy=self.lazy,
                                           **(self.ext or {}))
            return
        self.sv.spec_verify_linear(t["target"], t["draft"], t["draft_tokens"], t["cu_draft"],
                                   t["temperature"], lb.seed, max_k=lb.max_k, rule=self.rule,
                                   workspace=self.ws, out=self.outs)

    def result_tensors(self):
        return [self.outs[0], self.outs[1]] + ([self.kl] if self.kl is not None else [])

    def settle(self):
        """Position-lazy: the bytes a call reads follow from its outcome
        (target rows 1..n+1, dense draft rows 1..min(n+1, K) of sampling
        requests), fixed for fixed inputs and seed."""
        if not self.lazy:
            return
        import torch
        lb = self.lb
        n = self.outs[1].cpu().long()
        K = torch.diff(lb.cu_draft.cpu().long())
        samp = lb.temperature.cpu() >= 0.05
        self.tgt_bytes = int((n + 1).sum()) * lb.V * lb.target.element_size()
        self.drf_bytes = int(torch.minimum(n + 1, K)[samp].sum()) * lb.V * lb.draft.element_size()
        if not lb.top128:
            self.rowpass_bytes = self.tgt_bytes + self.drf_bytes

    def mean_accepted(self):
        return float(self.outs[1].float().mean())

    def oracle_sample(self, units, offset=0):
        """Runs the oracle on `units` requests; returns the draft positions done."""
        import numpy as np
        from oracle import spec_oracle as O
        lb = self.lb
        if not hasattr(self, "_host"):
            self._host = (lb.target.cpu(), lb.draft.cpu(), lb.draft_tokens.cpu().numpy(),
                          lb.cu_draft.cpu().numpy(), lb.temperature.cpu().numpy())
            self._order = np.random.default_rng(1).permutation(lb.B)
        tgt, drf, toks, cu, T = self._host
        req = np.sort(np.roll(self._order, -offset)[:min(units, lb.B)])
        O.verify_linear(tgt, drf, toks, cu, T, lb.seed, rule=self.rule, max_k=lb.max_k,
                        requests=req, **(self.ext or {}))
        return int(sum(cu[b + 1] - cu[b] for b in req))


class TreeWork:
    """spec_verify_tree on the tree workload (config 4)."""
    unit_name = "trees"

    def __init__(self, cfg, dev, input_seed=None, B=None):
        import torch
        import speculative_decoding_rejection_gb300 as sv
        from speculative_decoding_rejection_gb300 import synthetic as S
        self.sv = sv
        over = {} if B is None else {"B": B}
        self.tb = tb = S.make_tree(cfg, device=dev, input_seed=input_seed, **over)
        cu = tb.cu_nodes.cpu().long()
        par = tb.parent.cpu().long()
        base = torch.repeat_interleave(cu[:-1], torch.diff(cu))
        n = tb.target.shape[0]
        internal = torch.zeros(n, dtype=torch.bool)
        has_parent = par >= 0
        internal[(par + base)[has_parent]] = True
        samp = (tb.temperature.cpu() >= 0.05).repeat_interleave(torch.diff(cu))
        self.positions = n - tb.B
        self._internal, self._samp, self._base = internal, samp, cu[:-1]
        # until a call's paths are known: every node's rows (settle() narrows
        # this to the nodes the walks visit)
        self.tgt_bytes = n * tb.V * tb.target.element_size()
        self.drf_bytes = int((internal & samp).sum()) * tb.V * tb.draft.element_size()
        self.rowpass_bytes = self.tgt_bytes + self.drf_bytes
        self.launches = 2   # setup, walk
        self.kernel = "k_tree_walk"
        W = tb.max_depth + 1
        self.outs = (torch.empty(tb.B, W, dtype=torch.int32, device=dev),
                     torch.empty(tb.B, dtype=torch.int32, device=dev),
                     torch.empty(tb.B, W, dtype=torch.int32, device=dev))
        self.ws = torch.empty(sv.spec_verify_tree_workspace(tb.B, n, tb.V, tb.max_depth,
                                                            tb.max_branch),
                              dtype=torch.uint8, device=dev)
        self.config = {"workload": tb.meta["workload"], "B": tb.B, "nodes": n, "V": tb.V,
                       "logits": "bf16" if tb.target.element_size() == 2 else "f32",
                       "rule": "rrsw_tree"}

    def input_tensors(self):
        tb = self.tb
        return {"target": tb.target, "draft": tb.draft, "node_token": tb.node_token,
                "parent": tb.parent, "cu_nodes": tb.cu_nodes, "temperature": tb.temperature}

    def call(self, inputs=None):
        tb = self.tb
        t = inputs or self.input_tensors()
        self.sv.spec_verify_tree(t["target"], t["draft"], t["node_token"], t["parent"],
                                 t["cu_nodes"], t["temperature"], tb.seed,
                                 max_depth=tb.max_depth, max_branch=tb.max_branch,
                                 workspace=self.ws, out=self.outs)

    def result_tensors(self):
        return list(self.outs)

    def settle(self):
        """The rows a call reads: the walk of each tree visits the root and
        the nodes of its accepted path (out_path), and reads their target
        rows and, for a sampling node with children, its draft row; fixed for
        fixed inputs and seed."""
        import torch
        tb = self.tb
        acc = self.outs[1].cpu().long()
        path = self.outs[2].cpu().long()
        visited = []
        for b in range(tb.B):
            nodes = [0] + [int(path[b, k]) for k in range(int(acc[b])) if path[b, k] >= 0]
            visited += [int(self._base[b]) + v for v in nodes]
        vis = torch.tensor(visited, dtype=torch.long)
        self.tgt_bytes = len(visited) * tb.V * tb.target.element_size()
        self.drf_bytes = (int((self._internal[vis] & self._samp[vis]).sum())
                          * tb.V * tb.draft.element_size())
        self.rowpass_bytes = self.tgt_bytes + self.drf_bytes

    def mean_accepted(self):
        return float(self.outs[1].float().mean())

    def oracle_sample(self, units, offset=0):
        import numpy as np
        from oracle import spec_oracle as O
        tb = self.tb
        if not hasattr(self, "_host"):
            self._host = (tb.target.cpu(), tb.draft.cpu(), tb.node_token.cpu().numpy(),
                          tb.parent.cpu().numpy(), tb.cu_nodes.cpu().numpy(),
                          tb.temperature.cpu().numpy())
        tgt, drf, tok, par, cu, T = self._host
        req = np.sort((np.arange(min(units, tb.B)) + offset) % tb.B)
        O.verify_tree(tgt, drf, tok, par, cu, T, tb.seed, tb.max_depth, requests=req)
        return int(sum(cu[b + 1] - cu[b] - 1 for b in req))


class RheoWork:
    """spec_rheo_expand: one expansion level of RheoSampling dynamic trees
    (64 trees x 10 frontier nodes, V = 128256 bf16, K = 10, m = 1)."""
    unit_name = "trees"
    metric = ("expanded frontier nodes/sec (RheoSampling tree construction, one level) and "
              "achieved HBM GB/s (% of GB300 peak), 1 GPU")
    unit = "frontier nodes/s"

    def __init__(self, dev, input_seed=None, B=None):
        import torch
        import speculative_decoding_rejection_gb300 as sv
        from speculative_decoding_rejection_gb300 import synthetic as S
        self.sv = sv
        rb = S.make_rheo(device=dev, input_seed=input_seed, **({"B": B} if B else {}))
        self.rb = rb
        F, V = rb.draft.shape
        self.positions = F
        self.tgt_bytes = 0
        self.drf_bytes = F * V * rb.draft.element_size()
        self.rowpass_bytes = self.drf_bytes       # the top-128 select reads every row once
        self.launches = 3   # validate, top-128 select with the expansion epilogue, selection
        self.kernel = "k_topk128"
        self.outs = (torch.empty(F, rb.K, dtype=torch.int32, device=dev),
                     torch.empty(F, rb.K, dtype=torch.float32, device=dev),
                     torch.empty(F, rb.K, dtype=torch.float32, device=dev),
                     torch.empty(F, rb.K, dtype=torch.float32, device=dev),
                     torch.empty(rb.B, rb.n_keep, dtype=torch.int32, device=dev))
        self.ws = torch.empty(sv.spec_rheo_expand_workspace(F, V), dtype=torch.uint8,
                              device=dev)
        self.config = {"workload": rb.meta["workload"], "B": rb.B, "frontier": F, "K": rb.K,
                       "m": rb.m, "n_keep": rb.n_keep, "V": V,
                       "logits": "bf16" if rb.draft.element_size() == 2 else "f32",
                       "rule": "rheo_expand"}

    def input_tensors(self):
        rb = self.rb
        return {"draft": rb.draft, "cu_frontier": rb.cu_frontier,
                "frontier_score": rb.frontier_score, "temperature": rb.temperature}

    def call(self, inputs=None):
        rb = self.rb
        t = inputs or self.input_tensors()
        self.sv.spec_rheo_expand(t["draft"], t["cu_frontier"], t["frontier_score"],
                                 t["temperature"], rb.seed, rb.level, K=rb.K, m=rb.m, eps=rb.eps,
                                 n_keep=rb.n_keep, workspace=self.ws, out=self.outs)

    def result_tensors(self):
        return [self.outs[0], self.outs[3], self.outs[4]]   # tokens, scores, kept ids

    def mean_accepted(self):
        return None

    def oracle_sample(self, units, offset=0):
        import numpy as np
        from oracle import spec_oracle as O
        rb = self.rb
        if not hasattr(self, "_host"):
            self._host = (rb.draft.cpu(), rb.cu_frontier.cpu().numpy(),
                          rb.frontier_score.cpu().numpy(), rb.temperature.cpu().numpy())
        drf, cu, fs, T = self._host
        b0 = offset % rb.B
        b1 = min(rb.B, b0 + units)
        lo, hi = int(cu[b0]), int(cu[b1])
        O.rheo_expand(drf[lo:hi], cu[b0:b1 + 1] - lo, fs[lo:hi], T[b0:b1], rb.seed, rb.level,
                      rb.K, rb.m, rb.eps, rb.n_keep)
        return hi - lo


def make_work(cfg, dev, input_seed=None, B=None, rule=None, lazy=False, kl=False, rheo=False,
              V=None):
    if rheo:
        return RheoWork(dev, input_seed, B)
    if cfg == 4:
        return TreeWork(cfg, dev, input_seed, B)
    return LinearWork(cfg, dev, input_seed, B, rule, lazy, kl, V)


def cpu_baseline(work, n_units):
    """The oracle, as it stands, on a bounded sample of the same workload."""
    t0 = time.perf_counter()
    pos = work.oracle_sample(n_units)
    dt = time.perf_counter() - t0
    n = min(n_units, work.config["B"])
    unit = getattr(work, "unit", UNIT)
    return {"value": pos / dt, "unit": unit, "cores": 1, "kind": "oracle",
            "sample": f"{n} of {work.config['B']} {work.unit_name} ({pos} "
                      f"{unit.split('/')[0]}) of the same workload, fp64 numpy, one thread, "
                      f"{dt:.1f} s"}


def run_reference(args):
    """Reference arm: the CPU oracle timed as it stands (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    import torch
    dev = "cuda:0" if torch.cuda.is_available() else "cpu"
    work = make_work(args.config, dev, B=args.B, rule=args.rule, rheo=args.rheo)
    per_step = 1 if args.config == 4 and not args.rheo else 2
    metric, unit = getattr(work, "metric", METRIC), getattr(work, "unit", UNIT)
    for k in range(args.warmup):
        work.oracle_sample(per_step, offset=k * per_step)
    pos = 0
    t0 = time.perf_counter()
    for k in range(args.steps):
        pos += work.oracle_sample(per_step, offset=(args.warmup + k) * per_step)
    dt = time.perf_counter() - t0
    value = pos / dt
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(work.config, step=f"{per_step} {work.unit_name} of the batch per step"),
        "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle",
                         "sample": f"{per_step} {work.unit_name} per step, {args.steps} steps, "
                                   "fp64 numpy, one thread"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    import speculative_decoding_rejection_gb300 as sv
    from speculative_decoding_rejection_gb300 import synthetic as S

    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    sv.lib()
    if args.fused_limit is not None:
        sv.spec_set_fused_limit(args.fused_limit)
    seed_base = S.INPUT_SEED_BASE + (0x100 if args.rheo else args.config)
    work = make_work(args.config, dev, input_seed=seed_base + 7919 * rank, B=args.B, V=args.V,
                     rule=args.rule, lazy=args.lazy, kl=args.kl, rheo=args.rheo)
    unit = getattr(work, "unit", UNIT)

    for _ in range(max(3, args.warmup)):
        work.call()
    torch.cuda.synchronize()
    if hasattr(work, "settle"):
        work.settle()
    assert sv.spec_get_status(work.ws) == sv.SPEC_OK
    K = args.steps
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # a call that touches less than twice the L2 would find its rows there
    # on the next call: such workloads write a buffer of twice the L2 before
    # every call, outside the call's own timing
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or 128 << 20
    touched = work.tgt_bytes + work.drf_bytes
    flush = touched < 2 * l2_bytes
    if flush:
        scratch = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
        ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else torch.cuda.current_device())
    clocks.start()
    time.sleep(0.25)
    barrier(world)
    torch.cuda.synchronize()
    e0.record()
    for k in range(K):
        if flush:
            scratch.fill_(k & 255)
            ev_s[k].record()
        sv.spec_profile_row_pass(ev_b[k], ev_a[k])
        work.call()
        if flush:
            ev_e[k].record()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    clocks.stop()
    if flush:
        ms_step = max_over_ranks(statistics.mean(s_.elapsed_time(e_) for s_, e_ in
                                                 zip(ev_s, ev_e)), world)
    else:
        ms_step = max_over_ranks(e0.elapsed_time(e1) / K, world)
    rp_ms = statistics.mean(b.elapsed_time(a) for b, a in zip(ev_b, ev_a))

    peaks, peak_src = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    achieved = work.rowpass_bytes / (rp_ms * 1e-3) / 1e9
    traffic = None
    lazy = getattr(work, "lazy", False)
    stream = getattr(work, "stream", False)
    plain = (not lazy and getattr(work, "kl", None) is None and getattr(work, "ext", None) is None
             and getattr(work, "kernel", None) is None)
    if ROWPASS_TRAFFIC["source_sha1"] == source_sha1("rowpass") and plain:
        traffic = ROWPASS_TRAFFIC["dram_per_algorithmic_byte"] * work.rowpass_bytes
    if (getattr(work, "kernel", None) == "k_topk128" and args.B is None and args.V is None and args.rheo
            and RHEO_TRAFFIC["source_sha1"] == source_sha1("topk")):
        traffic = RHEO_TRAFFIC["dram_per_algorithmic_byte"] * work.rowpass_bytes
    if (getattr(work, "kernel", None) == "k_topk128" and args.B is None and args.V is None and args.config == 3
            and not args.rheo
            and TOPK_TRAFFIC["source_sha1"] == source_sha1("topk")):
        traffic = TOPK_TRAFFIC["dram_per_algorithmic_byte"] * work.rowpass_bytes
    if (getattr(work, "kernel", None) == "k_tree_walk" and args.B is None and args.V is None and args.config == 4
            and TREE_TRAFFIC["source_sha1"] == source_sha1("tree")):
        traffic = TREE_TRAFFIC["dram_per_algorithmic_byte"] * work.rowpass_bytes
    if (stream and getattr(work, "ext", None) is None and args.B is None and args.V is None and args.config == 5
            and STREAM_TRAFFIC["source_sha1"] == source_sha1("stream")):
        traffic = STREAM_TRAFFIC["dram_per_algorithmic_byte"] * work.rowpass_bytes

    # end to end through the same API: pinned host inputs copied in, the
    # results read back, every step
    e2e = None
    if not args.no_e2e:
        host = {n: t.cpu().pin_memory() for n, t in work.input_tensors().items()}
        dev_in = {n: torch.empty_like(t) for n, t in work.input_tensors().items()}
        res = work.result_tensors()
        host_out = [torch.empty(r.shape, dtype=r.dtype).pin_memory() for r in res]
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out)

        def e2e_step():
            for n, t in host.items():
                dev_in[n].copy_(t, non_blocking=True)
            work.call(dev_in)
            for h, r in zip(host_out, res):
                h.copy_(r, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record()
        for _ in range(args.e2e_steps):
            e2e_step()
        f1.record()
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(f0.elapsed_time(f1) / args.e2e_steps, world)
        e2e = {"value": world * work.positions / (e2e_ms * 1e-3), "unit": unit,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}
        del host, dev_in

    algo = work.tgt_bytes + work.drf_bytes
    line = {
        "metric": getattr(work, "metric", METRIC),
        "value": world * work.positions / (ms_step * 1e-3),
        "unit": unit,
        "n_gpus": world,
        "steps": K,
        "warmup": max(3, args.warmup),
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "impl": "gb300",
        "config": dict(work.config,
                       l2=(f"{algo / 1e9:.3f} GB read per step; L2 ({l2_bytes >> 20} MiB) "
                           "flushed before every call by writing twice its size, untimed"
                           if flush else
                           f"inputs {algo / 1e9:.2f} GB per step, larger than L2"),
                       parallelism=f"replicas x{world} (independent request batches)"),
        "hbm_gbs_whole_call": algo / (ms_step * 1e-3) / 1e9,
        "algorithmic_bytes_per_step": algo,
        "mean_accepted": work.mean_accepted(),
        "roofline": {
            "kernel": (getattr(work, "kernel", None) or
                       ("k_verify_stream" if stream
                        else "k_row_pass rounds with k_lazy_decide (one span)" if lazy
                        else "k_row_pass")),
            "bound": "hbm", "achieved": achieved, "peak": peak,
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
            else "fallback", "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
            "algorithmic_bytes_per_launch": work.rowpass_bytes, "ms_per_launch": rp_ms,
        },
        "gpu_launches": K * work.launches,
        "clocks": clocks.summary(),
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(
            work, 8 if args.config == 4 and not args.rheo else 16 if args.rheo
            else args.cpu_requests)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Throughput of the batched speculative-decoding verifier on GB300.

A step is one verification call over one batch of synthetic requests. The
default workload is B=1024 requests x K=4 drafts, V=201088, bf16 target and
draft logits, per-request T ~ U[0, 1.2] (greedy below 0.05): one
spec_verify_linear call per step. The headline value is verified draft
positions per second (draft positions in the batch / step time); the JSON
line also carries the achieved HBM bandwidth of the dominant kernel against
the measured copy peak, an end-to-end number through the same C ABI with
host buffers, the CPU oracle timed on the whole batch, and the parity of the
timed call's outputs with the oracle's (requests compared, mismatched, and
flagged: draws the oracle finds within 1e-6 of a decision boundary).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--config 1|2|3|4|5]

Without --config, the line also carries `per_config`: workloads 1-4 timed
the same way in the same run, each with its dominant kernel's roofline, its
clocks and its whole-batch parity. --config 3 is the top-128 truncation
workload, --config 4 the tree (RRSw) workload (spec_verify_tree; positions =
draft nodes). Workloads whose call reads less than twice the L2 (configs 1,
2 and 4) write twice the L2 before every call, outside the call's timing.
Under torchrun each rank verifies its own batch (weak scaling, no data-path
collective); rank 0 prints the line.
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

# DRAM traffic of the dominant kernels per algorithmic byte, each from a
# one-pass ncu capture (dram__bytes_read.sum + dram__bytes_write.sum over the
# algorithmic bytes the launch must read). Each figure holds only for the
# sources it was taken on (KERNEL_SOURCES, by SHA-1) and the workload named.
# The eager row pass, captured on B=128, K=4, V=201088 bf16 (460.09 MB
# streamed by the statistics launch): 460.19 MB read + 3.17 MB written (the
# per-chunk partial statistics); traffic grows with the rows streamed.
ROWPASS_TRAFFIC = {"source_sha1": "9878f7b237af20ab178ca224a5091735221d7f8b",
                   "dram_per_algorithmic_byte": (460191232 + 3168000) / 460089344}
# The streaming verifier (the plain call's schedule on dense bf16 logits),
# per byte of the rows the schedule must read (target rows 1..n+1, dense
# draft rows 1..min(n+1, K) of sampling requests), on the full B=1024, K=4,
# V=201088 workload: 2641.1 MB read + 30.0 MB written for 1975.1 MB. The
# excess is the residual row pairs read a second time (they miss L2).
STREAM_TRAFFIC = {"source_sha1": "d08b101f3f959ee87d8d759e447d40cde7e2009f",
                  "dram_per_algorithmic_byte": (2641137920 + 29974016) / 1975086336}
# The scan launch of the top-128 select (every draft row streamed once through
# a TMA ring; the candidate lists written), per byte of the draft rows, on the
# full B=256, K=7, V=151936 workload: 544.65 MB read + 5.63 MB written for
# 544.54 MB.
TOPK_TRAFFIC = {"source_sha1": "ed7ecf1a0747b8da35cd79b1383b1b98545c0ea0",
                "dram_per_algorithmic_byte": (544654080 + 5634560) / 544538624}
# The scan launch of the top-128 select on the construction workload (640
# frontier rows, V = 128256 bf16; L2 flushed before the call): 164.25 MB read
# + 3.03 MB written for 164.17 MB (most of the write is dirty lines of the L2
# flush buffer, written back as the rows evict them).
RHEO_TRAFFIC = {"source_sha1": "ed7ecf1a0747b8da35cd79b1383b1b98545c0ea0",
                "dram_per_algorithmic_byte": (164250624 + 3033856) / 164167680}
# The tree walk (only visited nodes' rows), per byte of those rows, on the
# full 32-tree workload: 59.44 MB read + 0.34 MB written for 59.25 MB.
TREE_TRAFFIC = {"source_sha1": "eb4d59e452da4f1cc7d8c74d221cdbde618aaa9b",
                "dram_per_algorithmic_byte": (59441408 + 336640) / 59254272}
# One cluster per request, on the 64-request, V = 32000 workload (L2 flushed):
# 20.87 MB read, nothing written back, for 20.80 MB of rows.
CLUSTER_TRAFFIC = {"source_sha1": "717c67a9cac4e35bdb735988e27010492532521e",
                   "dram_per_algorithmic_byte": (20869632 + 0) / 20800000}
# The cluster-resident schedule on the full B=1024 workload: 1975.56 MB read
# + 3.77 MB written for 1975.09 MB of first reads (each row read once).
RESIDENT_TRAFFIC = {"source_sha1": "717c67a9cac4e35bdb735988e27010492532521e",
                    "dram_per_algorithmic_byte": (1975558656 + 3765248) / 1975086336}


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", type=int, default=None, choices=[1, 2, 3, 4, 5],
                    help="time this workload alone (default: workload 5, with workloads 1-4 "
                         "in per_config)")
    ap.add_argument("--V", type=int, default=None,
                    help="linear workloads: override the vocabulary size (size sweeps)")
    ap.add_argument("--B", type=int, default=None,
                    help="override the number of requests (small profiling cases)")
    ap.add_argument("--e2e-steps", type=int, default=6)
    ap.add_argument("--cpu-requests", type=int, default=None,
                    help="requests (or trees) in the oracle's timed sample (default: the "
                         "whole batch, 16 trees for the construction workload)")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle (and so the parity check)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time workload 5 alone")
    ap.add_argument("--kl", action="store_true",
                    help="linear workloads: also emit the per-position KL(p || q)")
    ap.add_argument("--lazy", action="store_true",
                    help="linear workloads: position-lazy verification (rows 1..n+1 only)")
    ap.add_argument("--eager", action="store_true",
                    help="linear workloads: force the eager schedule (every row read)")
    ap.add_argument("--resident", action="store_true",
                    help="linear workloads: the cluster-resident position-lazy schedule "
                         "(every needed row read once)")
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
    args = ap.parse_args(argv)
    args.headline_only = args.config is not None or args.no_per_config
    if args.config is None:
        args.config = 5
    return args


# Every source a kernel is compiled from: a traffic figure holds only while
# all of them are unchanged.
KERNEL_SOURCES = {
    "rowpass": ("rowpass.cu", "rowpass.cuh", "common.cuh", "internal.h"),
    "stream": ("stream.cu", "linear.cuh", "rowpass.cuh", "common.cuh", "internal.h"),
    "topk": ("topk.cu", "common.cuh", "internal.h"),
    "tree": ("tree.cu", "common.cuh", "internal.h"),
    "resident": ("resident.cu", "linear.cuh", "rowpass.cuh", "common.cuh", "internal.h"),
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
def _overrides(B=None, V=None):
    over = {}
    if B is not None:
        over["B"] = B
    if V is not None:
        over["V"] = V
    return over


def shape_config(cfg, rheo=False, B=None, V=None):
    """The workload's name and sizes, from its definition alone (no inputs
    are built and the library is not loaded)."""
    from speculative_decoding_rejection_gb300 import synthetic as S
    over = _overrides(B, V)
    if rheo:
        w = dict(S.RHEO_WORKLOAD)
        w.update(over)
        name = w["name"] if not over else f"{w['name']}+{sorted(over.items())}"
        return {"workload": name, "B": w["B"], "frontier": w["B"] * w["W"], "K": w["K"],
                "m": w["m"], "n_keep": w["n_keep"], "V": w["V"], "logits": w["dtype"],
                "rule": "rheo_expand"}
    w = S.workload(cfg, **over)
    if w["kind"] == "tree":
        return {"workload": w["name"], "B": w["B"], "nodes": w["B"] * w["N"], "V": w["V"],
                "logits": w["dtype"], "rule": "rrsw_tree"}
    name = w["name"] if not over else f"{w['name']}+{sorted(over.items())}"
    K = w["K"][1] if isinstance(w["K"], tuple) else int(w["K"])
    return {"workload": name, "B": w["B"], "K": K, "V": w["V"], "logits": w["dtype"],
            "rule": "strict_top128" if w.get("top128") else "strict"}


def linear_variant(config, rule, lazy, kl, ext, eager=False, resident=False):
    """The rule, schedule and output keys a linear call adds to its config."""
    c = dict(config)
    if ext is not None:
        c["rule"] = "cactus(alpha={alpha},max_rank={max_rank},min_prob={min_prob})".format(**ext)
    if kl:
        c["outputs"] = "tokens, counts and per-position KL(p || q)"
    if resident:
        c["schedule"] = "position-lazy, rows resident in a CTA cluster (each row read once)"
    elif lazy:
        c["schedule"] = "position-lazy (rows 1..n+1 per request)"
    elif eager:
        c["schedule"] = "eager (every row read)"
    return c


def compare_outputs(ref, tokens, accepted, path=None):
    """Whole-batch parity of one call's outputs with the oracle's on the
    same inputs. A request compares bit for bit (tokens, accepted count,
    tree path) unless the oracle flags one of its draws as within 1e-6 of a
    decision boundary; a flagged request compares the output slots before
    the flagged one."""
    import numpy as np
    mism = flagged = 0
    for j, b in enumerate(ref["requests"]):
        fs = int(ref["flag_slot"][j])
        if fs < 0:
            ok = (np.array_equal(tokens[b], ref["tokens"][j])
                  and int(accepted[b]) == int(ref["accepted"][j])
                  and (path is None or np.array_equal(path[b], ref["path"][j])))
        else:
            flagged += 1
            ok = np.array_equal(tokens[b][:fs], ref["tokens"][j][:fs])
        mism += 0 if ok else 1
    return {"requests": int(len(tokens)), "compared": int(len(ref["requests"])),
            "mismatched": mism, "flagged": flagged}


class LinearWork:
    """spec_verify_linear on a linear workload (configs 1, 2, 3, 5)."""
    unit_name = "requests"

    # relaxed rule options: the guard the page recommends (p >= 0.10, top 10)
    CACTUS = {"alpha": 0.5, "max_rank": 10, "min_prob": 0.10}

    def __init__(self, cfg, dev, input_seed=None, B=None, rule=None, lazy=False, kl=False,
                 V=None, eager=False, resident=False, lb=None):
        import torch
        import speculative_decoding_rejection_gb300 as sv
        from speculative_decoding_rejection_gb300 import synthetic as S
        self.sv = sv
        self.cfg = cfg
        if lb is None:
            lb = S.make_linear(cfg, device=dev, input_seed=input_seed, **_overrides(B, V))
        self.lb = lb
        self.rule = sv.SPEC_RULE_STRICT_TOP128 if lb.top128 else sv.SPEC_RULE_STRICT
        self.ext = None
        if rule == "cactus":
            self.rule, self.ext = sv.SPEC_RULE_CACTUS, dict(self.CACTUS)
        self.eager, self.resident_flag = eager, resident
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
        # the top-128 select of bf16 rows with V % 8 == 0 and V >= 4096 runs
        # as a scan launch (which reads the rows) and a finishing launch
        topk_split = (lb.top128 and lb.draft.dtype == torch.bfloat16 and lb.V % 8 == 0
                      and lb.V >= 4096)
        self.kernel = (("k_topk128_scan" if topk_split else "k_topk128") if lb.top128
                       else None)
        # setup, row pass, accept, final draws, + the residual sums (dense
        # drafts) or the top-128 select (truncation); the header memset is
        # not ours
        self.launches = 6 if topk_split else 5
        self.outs = (torch.empty(lb.B, lb.max_k + 1, dtype=torch.int32, device=dev),
                     torch.empty(lb.B, dtype=torch.int32, device=dev), None)
        self.ws = torch.empty(sv.spec_verify_linear_workspace(lb.B, lb.max_k, lb.V, self.rule),
                              dtype=torch.uint8, device=dev)
        self.config = linear_variant(shape_config(cfg, B=B, V=V), rule, lazy, kl, self.ext,
                                     eager, resident)
        # the library's schedule (include/specverify.h): dense bf16 logits
        # with V % 8 == 0 and no KL stream position-lazily in one persistent
        # kernel (setup, streaming verifier, final draws) when asked, and for
        # a plain strict call without per-position outputs; the resident
        # schedule (setup, one cluster kernel that also draws) when asked,
        # under the strict rule with 16384 <= V <= 204800
        bf16 = lb.target.dtype == torch.bfloat16
        streamable = not lb.top128 and not kl and lb.V % 8 == 0 and bf16
        self.resident = (resident and streamable and self.ext is None
                         and 16384 <= lb.V <= 204800)
        plain = not (lazy or resident or eager or kl) and self.ext is None
        self.stream = streamable and not self.resident and (lazy or resident or plain)
        asked_lazy = lazy or resident
        lazy = lazy or resident or self.stream
        self.lazy = lazy
        if lazy:
            # rounds: a row pass and a decision launch per position; around
            # them the setup, the top-128 select or the residual sums, and
            # the final draws
            self.launches = (2 if self.resident else 3 if self.stream
                             else 3 + 2 * (lb.max_k + 1) + (1 if topk_split else 0))
        # small calls of the strict or greedy rule on dense logits or
        # probabilities run as one fused kernel (the library's own test:
        # rows of at most 8192 logits, at most 1 MiB of rows per request and
        # the fused limit in all)
        limit = sv.spec_set_fused_limit(0)
        sv.spec_set_fused_limit(limit)
        esz = lb.target.element_size()
        per_req = (lb.max_k + 1) * lb.V * esz + lb.max_k * lb.V * lb.draft.element_size()
        self.fused = (not (asked_lazy or eager) and not kl and self.ext is None and not lb.top128
                      and lb.V <= 8192 and per_req <= 1 << 20 and lb.B * per_req <= limit)
        # longer bf16 rows in calls of at most 128 requests and 8 drafts whose
        # row slices fit a cluster's shared memory: one cluster per request
        # (one launch; the rows pass through shared-memory buffers)
        slice_ = (lb.V // 8 + 7) // 8 * 8
        self.cluster_small = (not self.fused and not (asked_lazy or eager) and not kl
                              and self.ext is None and not lb.top128 and bf16 and lb.V % 8 == 0
                              and lb.max_k <= 8 and lb.B <= 128 and limit > 0
                              and (2 * lb.max_k + 1) * slice_ * 2 <= 102400)
        if self.fused or self.cluster_small:
            self.launches = 1
            self.kernel = "k_verify_small" if self.fused else "k_verify_cluster_small"
            self.config["schedule"] = ("fused (one block per request)" if self.fused else
                                       "one cluster per request")
            self.stream = self.lazy = False
        elif self.stream and "schedule" not in self.config:
            self.config["schedule"] = "position-lazy streaming (rows 1..n+1 per request)"
        if self.kernel is None:
            self.kernel = ("k_verify_resident" if self.resident
                           else "k_verify_stream" if self.stream
                           else "k_row_pass rounds with k_lazy_decide (one span)" if lazy
                           else "k_row_pass")

    def input_tensors(self):
        lb = self.lb
        return {"target": lb.target, "draft": lb.draft, "draft_tokens": lb.draft_tokens,
                "cu_draft": lb.cu_draft, "temperature": lb.temperature}

    def call(self, inputs=None):
        lb = self.lb
        t = inputs or self.input_tensors()
        if (self.ext is not None or self.kl is not None or self.eager or self.resident_flag
                or (self.lazy and not self.plain_call())):
            self.sv.spec_verify_linear_ext(t["target"], t["draft"], t["draft_tokens"],
                                           t["cu_draft"], t["temperature"], lb.seed,
                                           max_k=lb.max_k, rule=self.rule, workspace=self.ws,
                                           out=self.outs + (None, self.kl),
                                           lazy=self.lazy and not self.resident_flag,
                                           resident=self.resident_flag, eager=self.eager,
                                           **(self.ext or {}))
            return
        self.sv.spec_verify_linear(t["target"], t["draft"], t["draft_tokens"], t["cu_draft"],
                                   t["temperature"], lb.seed, max_k=lb.max_k, rule=self.rule,
                                   workspace=self.ws, out=self.outs)

    def plain_call(self):
        """The workload's own call, spec_verify_linear without options (its
        schedule is the library's choice)."""
        return "schedule" not in self.config or self.config["schedule"].startswith(
            ("position-lazy streaming", "fused", "one cluster per request"))

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

    def host_inputs(self):
        import numpy as np
        if not hasattr(self, "_host"):
            lb = self.lb
            self._host = (lb.target.cpu(), lb.draft.cpu(), lb.draft_tokens.cpu().numpy(),
                          lb.cu_draft.cpu().numpy(), lb.temperature.cpu().numpy())
            self._order = np.random.default_rng(1).permutation(lb.B)
        return self._host

    def oracle_sample(self, units, offset=0):
        """Runs the oracle on `units` requests; returns the draft positions
        done and the oracle's result."""
        import numpy as np
        from oracle import spec_oracle as O
        lb = self.lb
        tgt, drf, toks, cu, T = self.host_inputs()
        req = np.sort(np.roll(self._order, -offset)[:min(units, lb.B)])
        ref = O.verify_linear(tgt, drf, toks, cu, T, lb.seed, rule=self.rule, max_k=lb.max_k,
                              requests=req, **(self.ext or {}))
        return int(sum(cu[b + 1] - cu[b] for b in req)), ref

    def compare(self, ref):
        return compare_outputs(ref, self.outs[0].cpu().numpy(), self.outs[1].cpu().numpy())


class TreeWork:
    """spec_verify_tree on the tree workload (config 4)."""
    unit_name = "trees"

    def __init__(self, cfg, dev, input_seed=None, B=None):
        import torch
        import speculative_decoding_rejection_gb300 as sv
        from speculative_decoding_rejection_gb300 import synthetic as S
        self.sv = sv
        self.cfg = cfg
        self.tb = tb = S.make_tree(cfg, device=dev, input_seed=input_seed, **_overrides(B))
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
        self.config = shape_config(cfg, B=B)

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

    def host_inputs(self):
        if not hasattr(self, "_host"):
            tb = self.tb
            self._host = (tb.target.cpu(), tb.draft.cpu(), tb.node_token.cpu().numpy(),
                          tb.parent.cpu().numpy(), tb.cu_nodes.cpu().numpy(),
                          tb.temperature.cpu().numpy())
        return self._host

    def oracle_sample(self, units, offset=0):
        import numpy as np
        from oracle import spec_oracle as O
        tb = self.tb
        tgt, drf, tok, par, cu, T = self.host_inputs()
        req = np.sort((np.arange(min(units, tb.B)) + offset) % tb.B)
        ref = O.verify_tree(tgt, drf, tok, par, cu, T, tb.seed, tb.max_depth, requests=req)
        return int(sum(cu[b + 1] - cu[b] - 1 for b in req)), ref

    def compare(self, ref):
        return compare_outputs(ref, self.outs[0].cpu().numpy(), self.outs[1].cpu().numpy(),
                               self.outs[2].cpu().numpy())


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
        self.cfg = None
        rb = S.make_rheo(device=dev, input_seed=input_seed, **_overrides(B))
        self.rb = rb
        F, V = rb.draft.shape
        self.positions = F
        self.tgt_bytes = 0
        self.drf_bytes = F * V * rb.draft.element_size()
        self.rowpass_bytes = self.drf_bytes       # the top-128 select reads every row once
        # validate, the top-128 select with the expansion epilogue (bf16 rows
        # with V % 8 == 0 and V >= 4096: a scan launch, which reads the rows,
        # and a finishing launch that also expands), the tree selection
        split = rb.draft.dtype == torch.bfloat16 and V % 8 == 0 and V >= 4096
        self.launches = 4 if split else 3
        self.kernel = "k_topk128_scan" if split else "k_topk128"
        self.outs = (torch.empty(F, rb.K, dtype=torch.int32, device=dev),
                     torch.empty(F, rb.K, dtype=torch.float32, device=dev),
                     torch.empty(F, rb.K, dtype=torch.float32, device=dev),
                     torch.empty(F, rb.K, dtype=torch.float32, device=dev),
                     torch.empty(rb.B, rb.n_keep, dtype=torch.int32, device=dev))
        self.ws = torch.empty(sv.spec_rheo_expand_workspace(F, V), dtype=torch.uint8,
                              device=dev)
        self.config = shape_config(None, rheo=True, B=B)

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
        from oracle import spec_oracle as O
        rb = self.rb
        if not hasattr(self, "_host"):
            self._host = (rb.draft.cpu(), rb.cu_frontier.cpu().numpy(),
                          rb.frontier_score.cpu().numpy(), rb.temperature.cpu().numpy())
        drf, cu, fs, T = self._host
        b0 = offset % rb.B
        b1 = min(rb.B, b0 + units)
        lo, hi = int(cu[b0]), int(cu[b1])
        ref = O.rheo_expand(drf[lo:hi], cu[b0:b1 + 1] - lo, fs[lo:hi], T[b0:b1], rb.seed,
                            rb.level, rb.K, rb.m, rb.eps, rb.n_keep)
        return hi - lo, None

    def compare(self, ref):
        return None


def make_work(cfg, dev, input_seed=None, B=None, rule=None, lazy=False, kl=False, rheo=False,
              V=None, eager=False, resident=False):
    if rheo:
        return RheoWork(dev, input_seed, B)
    if cfg == 4:
        return TreeWork(cfg, dev, input_seed, B)
    return LinearWork(cfg, dev, input_seed, B, rule, lazy, kl, V, eager, resident)


def cpu_baseline(work, n_units):
    """The oracle, as it stands, on a bounded sample of the same workload (the
    whole batch by default). Returns the baseline record and the oracle's
    result on that sample."""
    t0 = time.perf_counter()
    pos, ref = work.oracle_sample(n_units)
    dt = time.perf_counter() - t0
    n = min(n_units, work.config["B"])
    unit = getattr(work, "unit", UNIT)
    return {"value": pos / dt, "unit": unit, "cores": 1, "kind": "oracle",
            "sample": f"{n} of {work.config['B']} {work.unit_name} ({pos} "
                      f"{unit.split('/')[0]}) of the same workload, fp64 numpy, one thread, "
                      f"{dt:.1f} s"}, ref


# --------------------------------------------------------- reference arm
class ReferenceSample:
    """The reference arm's inputs: a batch of `n` requests (trees) drawn on
    the CPU from the workload's own recipe. The arm times the oracle alone,
    so it builds nothing on the GPU and never loads the verifier library."""

    def __init__(self, args, n):
        from speculative_decoding_rejection_gb300 import synthetic as S
        self.rheo = args.rheo
        self.cfg = args.config
        self.ext = LinearWork.CACTUS if args.rule == "cactus" else None
        if args.rheo:
            self.config = shape_config(None, rheo=True, B=args.B)
            self.unit_name = "trees"
            self.rb = S.make_rheo(device="cpu", B=n)
        elif args.config == 4:
            self.config = shape_config(4, B=args.B)
            self.unit_name = "trees"
            self.tb = S.make_tree(4, device="cpu", B=n)
        else:
            self.config = linear_variant(shape_config(args.config, B=args.B, V=args.V),
                                         args.rule, args.lazy, args.kl, self.ext)
            self.unit_name = "requests"
            over = {"B": n}
            if args.V is not None:
                over["V"] = args.V
            self.lb = S.make_linear(args.config, device="cpu", **over)
            # rule ids as include/specverify.h numbers them
            self.rule = 3 if self.ext else 2 if self.lb.top128 else 0
        self.n = n

    def oracle_sample(self, units, offset=0):
        import numpy as np
        from oracle import spec_oracle as O
        if self.rheo:
            rb = self.rb
            b0 = offset % rb.B
            b1 = min(rb.B, b0 + units)
            cu = rb.cu_frontier.numpy()
            lo, hi = int(cu[b0]), int(cu[b1])
            O.rheo_expand(rb.draft[lo:hi], cu[b0:b1 + 1] - lo, rb.frontier_score.numpy()[lo:hi],
                          rb.temperature.numpy()[b0:b1], rb.seed, rb.level, rb.K, rb.m, rb.eps,
                          rb.n_keep)
            return hi - lo
        if self.cfg == 4:
            tb = self.tb
            req = np.sort((np.arange(min(units, tb.B)) + offset) % tb.B)
            cu = tb.cu_nodes.numpy()
            O.verify_tree(tb.target, tb.draft, tb.node_token.numpy(), tb.parent.numpy(), cu,
                          tb.temperature.numpy(), tb.seed, tb.max_depth, requests=req)
            return int(sum(cu[b + 1] - cu[b] - 1 for b in req))
        lb = self.lb
        req = np.sort((np.arange(min(units, lb.B)) + offset) % lb.B)
        cu = lb.cu_draft.numpy()
        O.verify_linear(lb.target, lb.draft, lb.draft_tokens.numpy(), cu, lb.temperature.numpy(),
                        lb.seed, rule=self.rule, max_k=lb.max_k, requests=req, **(self.ext or {}))
        return int(sum(cu[b + 1] - cu[b] for b in req))


# requests (trees) the reference arm draws on the CPU: enough for the steps it
# cycles over, few enough to build in seconds
REFERENCE_SAMPLE = {1: 4, 2: 64, 3: 16, 4: 8, 5: 32, "rheo": 16}


def run_reference(args):
    """Reference arm: the CPU oracle timed as it stands (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    full_B = shape_config(args.config, rheo=args.rheo, B=args.B)["B"]
    n = min(full_B, REFERENCE_SAMPLE["rheo" if args.rheo else args.config])
    work = ReferenceSample(args, n)
    per_step = 1 if args.config == 4 and not args.rheo else 2
    metric, unit = (RheoWork.metric, RheoWork.unit) if args.rheo else (METRIC, UNIT)
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
                                   f"cycling over {n} {work.unit_name} drawn on the CPU from "
                                   "the workload's recipe; fp64 numpy, one thread"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------- measurement
def l2_size(dev):
    import torch
    return int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or 128 << 20


def timed_calls(work, sv, dev, steps, warmup, world):
    """W warm-up calls, then `steps` calls bracketed by a barrier and a
    device synchronisation, timed with CUDA events on the calling stream.
    A second pass of `steps` calls, after the timed one, has the library
    record two more events around the dominant kernel of each call (those
    records would add some microseconds to a short call, so the step time is
    taken without them). Returns the step time (max over ranks), that
    kernel's mean time, whether L2 was flushed, and the clocks sampled
    during the timed calls."""
    import torch
    for _ in range(max(3, warmup)):
        work.call()
    torch.cuda.synchronize()
    if hasattr(work, "settle"):
        work.settle()
    assert sv.spec_get_status(work.ws) == sv.SPEC_OK
    K = steps
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # a call that touches less than twice the L2 would find its rows there
    # on the next call: such workloads write a buffer of twice the L2 before
    # every call, outside the call's own timing
    l2_bytes = l2_size(dev)
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
        work.call()
        if flush:
            ev_e[k].record()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    clocks.stop()
    # the dominant kernel's duration, from the same calls repeated
    for k in range(K):
        sv.spec_profile_row_pass(ev_b[k], ev_a[k])
        if flush:
            scratch.fill_(k & 255)
        work.call()
        if k == 0 and sv.spec_profile_pending():
            raise RuntimeError(f"{work.kernel}: the call recorded no profiling events")
    torch.cuda.synchronize()
    sv.spec_profile_row_pass(None, None)
    if flush:
        ms_step = max_over_ranks(statistics.mean(s_.elapsed_time(e_) for s_, e_ in
                                                 zip(ev_s, ev_e)), world)
    else:
        ms_step = max_over_ranks(e0.elapsed_time(e1) / K, world)
    rp_ms = statistics.mean(b.elapsed_time(a) for b, a in zip(ev_b, ev_a))
    assert sv.spec_get_status(work.ws) == sv.SPEC_OK
    return {"ms_step": ms_step, "rp_ms": rp_ms, "flush": flush, "l2_bytes": l2_bytes,
            "clocks": clocks.summary()}


def traffic_for(work, args):
    """DRAM bytes per launch of the dominant kernel from its committed ncu
    capture, scaled by the algorithmic bytes; None where the capture does not
    hold (other sources, sizes or kernel variants)."""
    kernel = getattr(work, "kernel", None)
    full = args.B is None and args.V is None
    ext = getattr(work, "ext", None)
    if kernel == "k_row_pass" and getattr(work, "kl", None) is None and ext is None:
        if ROWPASS_TRAFFIC["source_sha1"] == source_sha1("rowpass"):
            return ROWPASS_TRAFFIC["dram_per_algorithmic_byte"] * work.rowpass_bytes
    if (kernel == "k_topk128_scan" and full and isinstance(work, RheoWork)
            and RHEO_TRAFFIC["source_sha1"] == source_sha1("topk")):
        return RHEO_TRAFFIC["dram_per_algorithmic_byte"] * work.rowpass_bytes
    if (kernel == "k_topk128_scan" and full and not isinstance(work, RheoWork) and work.cfg == 3
            and TOPK_TRAFFIC["source_sha1"] == source_sha1("topk")):
        return TOPK_TRAFFIC["dram_per_algorithmic_byte"] * work.rowpass_bytes
    if (kernel == "k_tree_walk" and full and work.cfg == 4
            and TREE_TRAFFIC["source_sha1"] == source_sha1("tree")):
        return TREE_TRAFFIC["dram_per_algorithmic_byte"] * work.rowpass_bytes
    if (kernel == "k_verify_stream" and ext is None and full and work.cfg == 5
            and STREAM_TRAFFIC["source_sha1"] == source_sha1("stream")):
        return STREAM_TRAFFIC["dram_per_algorithmic_byte"] * work.rowpass_bytes
    if (kernel == "k_verify_cluster_small" and full and work.cfg == 2
            and CLUSTER_TRAFFIC["source_sha1"] == source_sha1("resident")):
        return CLUSTER_TRAFFIC["dram_per_algorithmic_byte"] * work.rowpass_bytes
    if (kernel == "k_verify_resident" and full and work.cfg == 5
            and RESIDENT_TRAFFIC["source_sha1"] == source_sha1("resident")):
        return RESIDENT_TRAFFIC["dram_per_algorithmic_byte"] * work.rowpass_bytes
    return None


def roofline(work, t, args):
    peaks, peak_src = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    achieved = work.rowpass_bytes / (t["rp_ms"] * 1e-3) / 1e9
    return {"kernel": work.kernel, "bound": "hbm", "achieved": achieved, "peak": peak,
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
            else "fallback", "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic_for(work, args),
            "algorithmic_bytes_per_launch": work.rowpass_bytes, "ms_per_launch": t["rp_ms"]}


def l2_note(work, t):
    algo = work.tgt_bytes + work.drf_bytes
    if t["flush"]:
        return (f"{algo / 1e9:.3f} GB read per step; L2 ({t['l2_bytes'] >> 20} MiB) "
                "flushed before every call by writing twice its size, untimed")
    return f"inputs {algo / 1e9:.2f} GB per step, larger than L2"


def parity_leg(work, n_units):
    """The oracle on `n_units` of the batch (timed: the CPU baseline) and the
    last timed call's outputs compared with it."""
    base, ref = cpu_baseline(work, n_units)
    return base, (work.compare(ref) if ref is not None else None)


def per_config_entry(cfg, dev, args, world, sv):
    """One workload of per_config: timed as the headline, with its roofline,
    clocks and whole-batch parity."""
    import torch
    from speculative_decoding_rejection_gb300 import synthetic as S
    work = make_work(cfg, dev, input_seed=S.INPUT_SEED_BASE + cfg)
    t = timed_calls(work, sv, dev, args.steps, args.warmup, world)
    entry = {"workload": work.config["workload"], "config": dict(work.config, l2=l2_note(work, t)),
             "value": work.positions / (t["ms_step"] * 1e-3),
             "unit": getattr(work, "unit", UNIT), "ms_per_step": t["ms_step"],
             "mean_accepted": work.mean_accepted(),
             "roofline": roofline(work, t, args), "gpu_launches": args.steps * work.launches,
             "clocks": t["clocks"]}
    if not args.no_cpu_baseline:
        entry["cpu_baseline"], entry["parity"] = parity_leg(work, work.config["B"])
    del work
    torch.cuda.empty_cache()
    return entry


def main(argv=None):
    args = parse(argv)
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
                     rule=args.rule, lazy=args.lazy, kl=args.kl, rheo=args.rheo,
                     eager=args.eager, resident=args.resident)
    unit = getattr(work, "unit", UNIT)
    t = timed_calls(work, sv, dev, args.steps, args.warmup, world)
    ms_step = t["ms_step"]

    # end to end through the same API: pinned host inputs copied in, the
    # results read back, every step
    e2e = None
    if not args.no_e2e:
        host = {n: t_.cpu().pin_memory() for n, t_ in work.input_tensors().items()}
        dev_in = {n: torch.empty_like(t_) for n, t_ in work.input_tensors().items()}
        res = work.result_tensors()
        host_out = [torch.empty(r.shape, dtype=r.dtype).pin_memory() for r in res]
        h2d = sum(t_.numel() * t_.element_size() for t_ in host.values())
        d2h = sum(t_.numel() * t_.element_size() for t_ in host_out)

        def e2e_step():
            for n, t_ in host.items():
                dev_in[n].copy_(t_, non_blocking=True)
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
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "impl": "gb300",
        "config": dict(work.config, l2=l2_note(work, t),
                       parallelism=f"replicas x{world} (independent request batches)"),
        "hbm_gbs_whole_call": algo / (ms_step * 1e-3) / 1e9,
        "algorithmic_bytes_per_step": algo,
        "mean_accepted": work.mean_accepted(),
        "roofline": roofline(work, t, args),
        "gpu_launches": args.steps * work.launches,
        "clocks": t["clocks"],
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n = (args.cpu_requests if args.cpu_requests is not None
             else 16 if args.rheo else work.config["B"])
        line["cpu_baseline"], line["parity"] = parity_leg(work, n)
    if isinstance(work, LinearWork) and work.stream and work.plain_call() and world == 1:
        # the same inputs on the eager schedule (every row read), for comparison
        ew = LinearWork(args.config, dev, eager=True, lb=work.lb)
        te = timed_calls(ew, sv, dev, args.steps, args.warmup, world)
        line["eager"] = {"schedule": ew.config["schedule"], "ms_per_step": te["ms_step"],
                         "value": work.positions / (te["ms_step"] * 1e-3),
                         "roofline": roofline(ew, te, args),
                         "algorithmic_bytes_per_step": ew.tgt_bytes + ew.drf_bytes,
                         "clocks": te["clocks"]}
        del ew
    if world == 1 and not args.headline_only:
        # the other workloads, one after another on the same GPU
        del work
        torch.cuda.empty_cache()
        line["per_config"] = {str(c): per_config_entry(c, dev, args, world, sv)
                              for c in (1, 2, 3, 4)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

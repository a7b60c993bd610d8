#!/usr/bin/env python
"""Throughput of the batched speculative-decoding verifier on GB300.

A step is one spec_verify_linear call over one batch of synthetic requests
(default: B=1024 requests x K=4 drafts, V=201088, bf16 target and draft
logits, per-request T ~ U[0, 1.2], greedy below 0.05). The headline value is
verified draft positions per second (sum of K over the batch / step time);
the JSON line also carries the achieved HBM bandwidth of the dominant kernel
(the row-statistics pass) against the measured copy peak, an end-to-end
number through the same C ABI with host buffers, and the CPU oracle timed on
a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--config 1..5]

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

# DRAM traffic of the row pass per algorithmic byte, from an ncu capture of
# a smaller case of the same kernel (dram__bytes_read.sum +
# dram__bytes_write.sum over the algorithmic bytes it streams). Valid only for
# the row-pass source it was taken on.
ROWPASS_TRAFFIC = {"source_sha1": None, "dram_per_algorithmic_byte": None}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", type=int, default=5, choices=[1, 2, 3, 5])
    ap.add_argument("--B", type=int, default=None,
                    help="override the number of requests (small profiling cases)")
    ap.add_argument("--e2e-steps", type=int, default=6)
    ap.add_argument("--cpu-requests", type=int, default=1024,
                    help="requests in the oracle's timed sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


def sha1(path):
    with open(path, "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()


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

    def __init__(self, gpu_index):
        self.gpu = gpu_index
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


def dist_setup(n_gpus):
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


def workload_bytes(lb):
    """Algorithmic bytes of one call: every target row once, plus the dense
    draft rows of sampling requests (read by the row pass, or by the top-128
    select under the truncation rule)."""
    import torch
    K = torch.diff(lb.cu_draft.cpu().long())
    T = lb.temperature.cpu()
    samp = T >= 0.05
    tgt = int((K + 1).sum()) * lb.V * lb.target.element_size()
    drf = int(K[samp].sum()) * lb.V * lb.draft.element_size()
    return tgt, drf, int(K.sum())


def cpu_baseline(lb, n_req, rule):
    """The oracle, as it stands, on a bounded sample of the same workload."""
    import numpy as np
    from oracle import spec_oracle as O
    tgt = lb.target.cpu()
    drf = lb.draft.cpu()
    toks = lb.draft_tokens.cpu().numpy()
    cu = lb.cu_draft.cpu().numpy()
    T = lb.temperature.cpu().numpy()
    req = np.sort(np.random.default_rng(0).choice(lb.B, size=min(n_req, lb.B), replace=False))
    t0 = time.perf_counter()
    O.verify_linear(tgt, drf, toks, cu, T, lb.seed, rule=rule, max_k=lb.max_k, requests=req)
    dt = time.perf_counter() - t0
    pos = int(sum(cu[b + 1] - cu[b] for b in req))
    return {"value": pos / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{len(req)} of {lb.B} requests ({pos} draft positions) of the same "
                      f"workload, fp64 numpy, one thread, {dt:.1f} s"}


def run_reference(args):
    """Reference arm: the CPU oracle timed as it stands (rank 0 only)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np
    import torch
    from oracle import spec_oracle as O
    from speculative_decoding_rejection_gb300 import synthetic as S
    dev = "cuda:0" if torch.cuda.is_available() else "cpu"
    lb = S.make_linear(args.config, device=dev)
    rule = 2 if lb.top128 else 0
    tgt, drf = lb.target.cpu(), lb.draft.cpu()
    toks = lb.draft_tokens.cpu().numpy()
    cu = lb.cu_draft.cpu().numpy()
    T = lb.temperature.cpu().numpy()
    per_step = 2
    order = np.random.default_rng(1).permutation(lb.B)

    def step(k):
        req = np.sort(order[(k * per_step) % lb.B:][:per_step])
        O.verify_linear(tgt, drf, toks, cu, T, lb.seed, rule=rule, max_k=lb.max_k, requests=req)
        return int(sum(cu[b + 1] - cu[b] for b in req))

    for k in range(args.warmup):
        step(k)
    pos = 0
    t0 = time.perf_counter()
    for k in range(args.steps):
        pos += step(args.warmup + k)
    dt = time.perf_counter() - t0
    value = pos / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": lb.meta["workload"], "B": lb.B, "V": lb.V,
                   "step": f"{per_step} requests of the batch per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{per_step} requests per step, {args.steps} steps, "
                                   "fp64 numpy, one thread"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
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

    world, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    sv.lib()
    over = {} if args.B is None else {"B": args.B}
    lb = S.make_linear(args.config, device=dev,
                       input_seed=S.INPUT_SEED_BASE + args.config + 7919 * rank, **over)
    rule = sv.SPEC_RULE_STRICT_TOP128 if lb.top128 else sv.SPEC_RULE_STRICT
    tgt_bytes, drf_bytes, positions = workload_bytes(lb)
    B = lb.B
    outs = (torch.empty(B, lb.max_k + 1, dtype=torch.int32, device=dev),
            torch.empty(B, dtype=torch.int32, device=dev), None)
    ws = torch.empty(sv.spec_verify_linear_workspace(B, lb.max_k, lb.V, rule),
                     dtype=torch.uint8, device=dev)

    def call():
        sv.spec_verify_linear(lb.target, lb.draft, lb.draft_tokens, lb.cu_draft,
                              lb.temperature, lb.seed, max_k=lb.max_k, rule=rule,
                              workspace=ws, out=outs)

    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    assert sv.spec_get_status(ws) == sv.SPEC_OK
    K = args.steps
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else torch.cuda.current_device())
    clocks.start()
    time.sleep(0.25)
    barrier(world)
    torch.cuda.synchronize()
    e0.record()
    for k in range(K):
        sv.spec_profile_row_pass(ev_b[k], ev_a[k])
        call()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    clocks.stop()
    ms_step = max_over_ranks(e0.elapsed_time(e1) / K, world)
    rp_ms = statistics.mean(b.elapsed_time(a) for b, a in zip(ev_b, ev_a))
    mean_acc = float(outs[1].float().mean())

    # dominant kernel: the row pass streams the target rows and the dense
    # draft rows of sampling requests (not under the top-128 rule)
    rp_bytes = tgt_bytes + (0 if lb.top128 else drf_bytes)
    peaks, peak_src = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    achieved = rp_bytes / (rp_ms * 1e-3) / 1e9
    traffic = None
    src = os.path.join(ROOT, "speculative_decoding_rejection_gb300", "csrc", "rowpass.cu")
    if ROWPASS_TRAFFIC["source_sha1"] == sha1(src):
        traffic = ROWPASS_TRAFFIC["dram_per_algorithmic_byte"] * rp_bytes

    # end to end through the same API: pinned host inputs copied in, the
    # result read back, every step
    e2e = None
    if not args.no_e2e:
        host = {n: getattr(lb, n).cpu().pin_memory()
                for n in ("target", "draft", "draft_tokens", "cu_draft", "temperature")}
        dev_in = {n: torch.empty_like(getattr(lb, n)) for n in host}
        h_tok = torch.empty(outs[0].shape, dtype=torch.int32).pin_memory()
        h_acc = torch.empty(outs[1].shape, dtype=torch.int32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = h_tok.numel() * 4 + h_acc.numel() * 4

        def e2e_step():
            for n, t in host.items():
                dev_in[n].copy_(t, non_blocking=True)
            sv.spec_verify_linear(dev_in["target"], dev_in["draft"], dev_in["draft_tokens"],
                                  dev_in["cu_draft"], dev_in["temperature"], lb.seed,
                                  max_k=lb.max_k, rule=rule, workspace=ws, out=outs)
            h_tok.copy_(outs[0], non_blocking=True)
            h_acc.copy_(outs[1], non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record()
        for _ in range(args.e2e_steps):
            e2e_step()
        f1.record()
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(f0.elapsed_time(f1) / args.e2e_steps, world)
        e2e = {"value": world * positions / (e2e_ms * 1e-3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms}
        del host, dev_in

    line = {
        "metric": METRIC,
        "value": world * positions / (ms_step * 1e-3),
        "unit": UNIT,
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
        "config": {
            "workload": lb.meta["workload"], "B": B, "K": lb.max_k, "V": lb.V,
            "logits": "bf16" if lb.target.element_size() == 2 else "f32",
            "rule": {0: "strict", 2: "strict_top128"}[rule],
            "l2": f"inputs {(tgt_bytes + drf_bytes) / 1e9:.2f} GB per step, larger than L2",
            "parallelism": f"replicas x{world} (independent request batches)",
        },
        "hbm_gbs_whole_call": (tgt_bytes + drf_bytes) / (ms_step * 1e-3) / 1e9,
        "algorithmic_bytes_per_step": tgt_bytes + drf_bytes,
        "mean_accepted": mean_acc,
        "roofline": {
            "kernel": "k_row_pass", "bound": "hbm", "achieved": achieved, "peak": peak,
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
            else "fallback", "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
            "algorithmic_bytes_per_launch": rp_bytes, "ms_per_launch": rp_ms,
        },
        # setup, row pass, accept, sampler tiles, sampler final (+ top-128)
        "gpu_launches": K * (6 if lb.top128 else 5),
        "clocks": clocks.summary(),
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(lb, args.cpu_requests, rule)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

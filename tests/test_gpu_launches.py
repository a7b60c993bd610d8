"""The bench's `gpu_launches` claim: for each schedule, the number of the
library's kernels one call launches, counted by the CUDA profiler, equals the
per-call count the bench multiplies by its timed calls."""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)

CASES = [
    ("plain call (streaming)", dict(cfg=5, B=64)),
    ("eager", dict(cfg=5, B=64, eager=True)),
    ("resident", dict(cfg=5, B=64, resident=True)),
    ("top-128", dict(cfg=3, B=16)),
    ("fused", dict(cfg=1)),
    ("cluster per request", dict(cfg=2)),
    ("stream", dict(cfg=5, B=64, lazy=True)),
    ("lazy rounds", dict(cfg=3, B=16, lazy=True)),
    ("cactus", dict(cfg=5, B=64, rule="cactus")),
    ("tree", dict(cfg=4, B=4)),
    ("construction", dict(cfg=5, rheo=True)),
]


def _kernels_of_one_call(work):
    from torch.profiler import ProfilerActivity, profile
    work.call()
    torch.cuda.synchronize()
    for _ in range(2):   # the process's first profiling session may record no kernels
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            work.call()
            torch.cuda.synchronize()
    names = [e.name for e in prof.events()
             if getattr(e, "device_type", None) is not None and "CUDA" in str(e.device_type)]
    return [n for n in names if "k_" in n and "Memset" not in n and "memset" not in n]


@pytest.mark.parametrize("name,case", CASES, ids=[c[0] for c in CASES])
def test_launch_count_matches_the_bench_claim(name, case):
    import bench
    case = dict(case)
    cfg = case.pop("cfg")
    work = bench.make_work(cfg, DEV, **case)
    kernels = _kernels_of_one_call(work)
    if not kernels:
        pytest.skip("the profiler recorded no kernels here")
    assert len(kernels) == work.launches, (name, kernels)


@pytest.mark.parametrize("name,case", CASES, ids=[c[0] for c in CASES])
def test_profiling_events_bracket_a_kernel_of_the_call(name, case):
    """The two events the bench reads its kernel time from are taken and
    recorded by the call itself, inside the call's own interval."""
    import bench
    import speculative_decoding_rejection_gb300 as sv
    case = dict(case)
    cfg = case.pop("cfg")
    work = bench.make_work(cfg, DEV, **case)
    work.call()
    torch.cuda.synchronize()
    e0, e1, eb, ea = (torch.cuda.Event(enable_timing=True) for _ in range(4))
    e0.record()
    sv.spec_profile_row_pass(eb, ea)
    work.call()
    assert not sv.spec_profile_pending(), name
    e1.record()
    torch.cuda.synchronize()
    inner, outer = eb.elapsed_time(ea), e0.elapsed_time(e1)
    assert 0.0 < inner <= outer, (name, inner, outer)

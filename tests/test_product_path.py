"""Host-side checks of the product path's boundaries: the package never
imports the oracle, the binding passes only device tensors, the synthetic
construction inputs have the stated shapes, and the reference arm of the
bench prints one line with the contract's keys."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_package_import_does_not_load_the_oracle():
    code = ("import sys; import speculative_decoding_rejection_gb300 as sv; "
            "from speculative_decoding_rejection_gb300 import synthetic; "
            "print(any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules))")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr[-1000:]
    assert out.stdout.strip() == "False"


def test_binding_rejects_host_tensors():
    import speculative_decoding_rejection_gb300 as sv
    try:
        sv.lib()
    except RuntimeError:
        pytest.skip("library not built")
    t = torch.zeros(4, 8)
    with pytest.raises(ValueError, match="CUDA"):
        sv.spec_verify_linear(t, t, torch.zeros(4, dtype=torch.int32),
                              torch.tensor([0, 4], dtype=torch.int32), torch.ones(1), 1,
                              max_k=4)


def test_construction_inputs_have_the_stated_shapes():
    from speculative_decoding_rejection_gb300 import synthetic as S
    rb = S.make_rheo(B=5, W=(0, 3), V=300, level=2, T=("uniform", 0.0, 1.2))
    F = int(rb.cu_frontier[-1])
    assert rb.draft.shape == (F, 300) and rb.draft.dtype == torch.bfloat16
    assert rb.frontier_score.shape == (F,)
    assert bool((rb.frontier_score <= 0).all()) and bool((rb.frontier_score >= -6).all())
    assert rb.temperature.shape == (5,)
    rb0 = S.make_rheo(B=3, W=2, V=300, level=0)
    assert bool((rb0.frontier_score == 0).all())      # roots at level 0
    again = S.make_rheo(B=5, W=(0, 3), V=300, level=2, T=("uniform", 0.0, 1.2))
    assert torch.equal(rb.draft, again.draft)          # seeded


def test_reference_arm_prints_the_contract_keys():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "0", "--config", "1"], cwd=ROOT, capture_output=True,
                         text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["value"] > 0


def test_reference_arm_never_loads_the_verifier_library():
    """The reference arm times the oracle alone: it builds its sample on the
    CPU and neither loads libspecverify.so nor touches a GPU."""
    code = ("import bench, speculative_decoding_rejection_gb300 as sv\n"
            "bench.main(['--impl', 'reference', '--steps', '1', '--warmup', '0', '--config', '2'])\n"
            "maps = open('/proc/self/maps').read()\n"
            "assert sv._lib is None and 'libspecverify' not in maps\n"
            "print('NOT_LOADED')\n")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                         timeout=600, env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert out.returncode == 0, out.stderr[-2000:]
    assert "NOT_LOADED" in out.stdout


def test_bench_counts_the_fused_schedule_as_one_launch():
    """Small strict calls run as one fused kernel; the bench's launch claim
    and dominant kernel follow the library's own size test."""
    import bench
    import speculative_decoding_rejection_gb300 as sv
    try:
        sv.lib()
    except RuntimeError:
        pytest.skip("library not built")
    cpu = torch.device("cpu")
    w = bench.make_work(1, cpu)
    assert w.fused and w.launches == 1 and w.kernel == "k_verify_small"
    old = sv.spec_set_fused_limit(0)
    try:
        w = bench.make_work(1, cpu)
        assert not w.fused and w.launches == 5
    finally:
        sv.spec_set_fused_limit(old)
    assert not bench.make_work(2, cpu, B=4).fused          # rows above 8192 logits
    assert not bench.make_work(1, cpu, lazy=True).fused

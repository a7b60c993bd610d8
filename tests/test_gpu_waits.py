"""Failure detection without a GPU fault: the kernels' bounded waits give up,
report SPEC_ERR_TIMEOUT through the status word and leave the context usable.

spec_wait_selftest waits with the verifier kernels' own waiting code on
something nothing completes (an mbarrier phase without arrivals, a global
word nothing writes); no kernel is broken and nothing traps or faults."""
import time

import numpy as np
import pytest
import torch

import speculative_decoding_rejection_gb300 as sv
from speculative_decoding_rejection_gb300 import synthetic as S

from parity import gpu_linear, oracle_linear, assert_linear_parity

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("kind", [0, 1])
def test_bounded_wait_times_out_and_the_context_stays_usable(kind):
    limit_ns = 20_000_000   # 20 ms
    t0 = time.perf_counter()
    ws = sv.spec_wait_selftest(kind, limit_ns)
    status = sv.spec_get_status(ws)
    elapsed = time.perf_counter() - t0
    assert status == sv.SPEC_ERR_TIMEOUT
    assert 0.015 < elapsed < 5.0
    # the same context verifies correctly afterwards, on the same workspace too
    lb = S.make_linear(1, device=DEV, input_seed=71)
    g = gpu_linear(lb)
    assert g["status"] == sv.SPEC_OK
    assert_linear_parity(g, oracle_linear(lb), lb.cu_draft.cpu(), min_compared=3)
    big = torch.zeros(sv.spec_verify_linear_workspace(lb.B, lb.max_k, lb.V), dtype=torch.uint8,
                      device=DEV)
    big[:256] = ws
    _, acc, _, ws2 = sv.spec_verify_linear(lb.target, lb.draft, lb.draft_tokens, lb.cu_draft,
                                           lb.temperature, lb.seed, max_k=lb.max_k, workspace=big)
    assert sv.spec_get_status(ws2) == sv.SPEC_OK
    assert np.array_equal(acc.cpu().numpy(), g["accepted"])

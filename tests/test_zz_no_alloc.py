"""spec_verify_linear_noalloc: the entry point for callers that cannot give
the library device scratch (engines that keep nearly all of HBM for their KV
cache, decode loops where cudaMalloc/cudaFree would synchronise the device).
It must give the same results as spec_verify_linear with a workspace.

Two calls in a row with different batches: the second finds the first one's
contents in the library's fixed scratch array and must not be affected.
This file sorts last so a run that stops at the first failure has already
run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_rejection_gb300 as sv
from speculative_decoding_rejection_gb300 import synthetic as S

from parity import assert_probs_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(lb):
    """Calls the no-allocation entry point through the C ABI."""
    B = lb.B
    tokens = torch.full((B, lb.max_k + 1), -7, dtype=torch.int32, device=DEV)
    acc = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    pq = torch.empty(lb.draft_tokens.numel(), 2, dtype=torch.float32, device=DEV)
    status = torch.full((1,), 99, dtype=torch.int32, device=DEV)
    dt = sv.SPEC_BF16 if lb.target.dtype == torch.bfloat16 else sv.SPEC_F32
    code = sv.lib().spec_verify_linear_noalloc(
        _p(lb.target), dt, _p(lb.draft), dt, sv.SPEC_DRAFT_LOGITS, None,
        _p(lb.draft_tokens), _p(lb.cu_draft), _p(lb.temperature), B, lb.V, lb.max_k,
        ctypes.c_uint64(lb.seed), sv.SPEC_RULE_STRICT, _p(tokens), _p(acc), _p(pq),
        _p(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == sv.SPEC_OK, sv.spec_status_string(code)
    torch.cuda.synchronize()
    return tokens.cpu().numpy(), acc.cpu().numpy(), pq.cpu().numpy(), int(status.item())


def _with_workspace(lb):
    tokens, acc, pq, ws = sv.spec_verify_linear(
        lb.target, lb.draft, lb.draft_tokens, lb.cu_draft, lb.temperature, lb.seed,
        max_k=lb.max_k, want_pq=True)
    assert sv.spec_get_status(ws) == sv.SPEC_OK
    return tokens.cpu().numpy(), acc.cpu().numpy(), pq.cpu().numpy()


def test_noalloc_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    batches = [S.make_linear(2, device=DEV, B=48, V=32000, input_seed=101),
               S.make_linear(1, device=DEV, B=7, K=6, V=5003, dtype="bf16", input_seed=202)]
    for lb in batches:
        t, a, pq, status = _noalloc(lb)
        rt, ra, rpq = _with_workspace(lb)
        assert status == sv.SPEC_OK
        assert np.array_equal(t, rt)
        assert np.array_equal(a, ra)
        assert_probs_close(pq, rpq, "p(d), q(d) of the no-allocation call")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    need = sv.spec_verify_linear_workspace(8192, 8, 201088)
    assert need > (16 << 20)
    code = sv.lib().spec_verify_linear_noalloc(
        None, 1, None, 1, 0, None, None, None, None, 8192, 201088, 8, ctypes.c_uint64(1), 0,
        None, None, None, None, None)
    assert code == sv.SPEC_ERR_UNSUPPORTED

"""GB300-native batched speculative-decoding verifier.

Thin Python binding over the C ABI in include/specverify.h: the functions here
only marshal arguments (device pointers of torch tensors, the current CUDA
stream) and raise on a non-zero return code. Every step of the verification
runs in the CUDA kernels of libspecverify.so; there is no CPU fallback. If
the library is not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from pathlib import Path

__all__ = [
    "SPEC_OK", "SPEC_F32", "SPEC_BF16", "SPEC_DRAFT_LOGITS", "SPEC_DRAFT_PROBS",
    "SPEC_DRAFT_SPARSE128", "SPEC_RULE_STRICT", "SPEC_RULE_GREEDY",
    "SPEC_RULE_STRICT_TOP128", "SPEC_RULE_CACTUS", "SPEC_TOPK", "lib", "spec_status_string",
    "spec_verify_linear", "spec_verify_linear_ext", "spec_verify_linear_workspace", "spec_verify_tree",
    "spec_verify_tree_workspace", "spec_verify_tree_ext", "draft_topk_softmax",
    "draft_topk_softmax_workspace", "spec_get_status", "spec_uniforms",
    "spec_profile_row_pass", "spec_profile_pending", "spec_rheo_expand", "spec_rheo_expand_workspace",
    "spec_set_fused_limit", "SpecError", "use_checked_library", "spec_check_selftest",
]

SPEC_OK = 0
SPEC_ERR_INVALID_ARG = -1
SPEC_ERR_UNSUPPORTED = -2
SPEC_ERR_WORKSPACE = -3
SPEC_ERR_CUDA = -4
SPEC_ERR_TIMEOUT = -5
SPEC_ERR_BOUNDS = -6
SPEC_F32, SPEC_BF16 = 0, 1
SPEC_DRAFT_LOGITS, SPEC_DRAFT_PROBS, SPEC_DRAFT_SPARSE128 = 0, 1, 2
SPEC_RULE_STRICT, SPEC_RULE_GREEDY, SPEC_RULE_STRICT_TOP128, SPEC_RULE_CACTUS = 0, 1, 2, 3
SPEC_TOPK = 128
SPEC_EXT_LAZY = 1
SPEC_EXT_RESIDENT = 2
SPEC_EXT_EAGER = 4
SPEC_RHEO_MAX_CANDIDATES = 8192

LIB_PATH = Path(__file__).resolve().parent / "libspecverify.so"
# The same library built with SPEC_CHECKED: every global access of the
# kernels checked against the call's buffers (include/specverify.h,
# SPEC_ERR_BOUNDS); a test build.
CHECKED_LIB_PATH = Path(__file__).resolve().parent / "libspecverify_checked.so"
HEADER = Path(__file__).resolve().parent.parent / "include" / "specverify.h"

_lib = None
_lib_path = LIB_PATH
_vp, _i32, _u64, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t
class SpecLinearExt(ctypes.Structure):
    """spec_linear_ext of include/specverify.h."""
    _fields_ = [("alpha", ctypes.c_float), ("max_rank", ctypes.c_int32),
                ("min_prob", ctypes.c_float), ("flags", ctypes.c_int32),
                ("out_rank", ctypes.c_void_p), ("out_kl", ctypes.c_void_p),
                ("seed_dev", ctypes.c_void_p)]


_SIGS = {
    "spec_status_string": (ctypes.c_char_p, [_i32]),
    "spec_verify_linear_workspace": (_sz, [_i32, _i32, _i32, _i32]),
    "spec_verify_linear": (_i32, [_vp, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _i32,
                                  _i32, _u64, _i32, _vp, _vp, _vp, _vp, _sz, _vp]),
    "spec_verify_linear_ext": (_i32, [_vp, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _i32,
                                      _i32, _i32, _u64, _i32, ctypes.POINTER(SpecLinearExt),
                                      _vp, _vp, _vp, _vp, _sz, _vp]),
    "spec_verify_tree_workspace": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "spec_verify_tree": (_i32, [_vp, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _i32,
                                _i32, _i32, _i32, _u64, _vp, _vp, _vp, _vp, _sz, _vp]),
    "spec_verify_tree_ext": (_i32, [_vp, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _i32,
                                    _i32, _i32, _i32, _i32, _u64, _vp, _vp, _vp, _vp, _vp, _sz,
                                    _vp]),
    "draft_topk_softmax_workspace": (_sz, [_i32, _i32]),
    "draft_topk_softmax": (_i32, [_vp, _i32, _i32, _i32, _vp, _vp, _i32, _i32, _vp, _vp, _vp,
                                  _sz, _vp]),
    "spec_rheo_expand_workspace": (_sz, [_i32, _i32]),
    "spec_rheo_expand": (_i32, [_vp, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                ctypes.c_float, _i32, _u64, _i32, _vp, _vp, _vp, _vp, _vp,
                                _vp, _sz, _vp]),
    "spec_get_status": (_i32, [_vp, _vp, ctypes.POINTER(_i32)]),
    "spec_set_fused_limit": (_sz, [_sz]),
    "spec_uniforms": (_i32, [_u64, _vp, _vp, _vp, _i32, _vp, _vp]),
    "spec_profile_row_pass": (_i32, [_vp, _vp]),
    "spec_profile_pending": (_i32, []),
    "spec_wait_selftest": (_i32, [_i32, ctypes.c_ulonglong, _vp, _vp]),
    "spec_check_selftest": (_i32, [_vp, _sz, _vp]),
    "spec_verify_linear_noalloc": (_i32, [_vp, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _i32,
                                          _i32, _i32, _u64, _i32, _vp, _vp, _vp, _vp, _vp]),
}


class SpecError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {spec_status_string(code)} ({code})")
        self.code = code


def use_checked_library(on: bool) -> None:
    """Routes every call of this module to the bounds-checked build (on) or
    to the product library (off). The first call after a switch loads the
    chosen library."""
    global _lib, _lib_path
    path = CHECKED_LIB_PATH if on else LIB_PATH
    if path != _lib_path:
        _lib_path, _lib = path, None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not _lib_path.exists():
            raise RuntimeError(f"{_lib_path.name} is not built; run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(str(_lib_path))
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/specverify.h declares."""
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(\w+)\s*\(", text, flags=re.M)


def spec_status_string(code: int) -> str:
    return lib().spec_status_string(int(code)).decode()


# ------------------------------------------------------------ marshalling
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to the verifier must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the verifier must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(code: int, where: str):
    if code != SPEC_OK:
        raise SpecError(code, where)


def _workspace(nbytes: int, device, workspace=None):
    torch = _torch()
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def spec_verify_linear_workspace(B: int, max_k: int, V: int, rule: int = SPEC_RULE_STRICT) -> int:
    return int(lib().spec_verify_linear_workspace(B, max_k, V, rule))


def _linear_workspace(B, max_k, V, rule, device, workspace):
    # a caller's workspace goes to the library as it is: the call checks its
    # size (SPEC_ERR_WORKSPACE) without a second query on this path
    if workspace is not None:
        return workspace
    ws_bytes = spec_verify_linear_workspace(B, max_k, V, rule)
    if ws_bytes == 0:
        raise SpecError(SPEC_ERR_INVALID_ARG, "spec_verify_linear_workspace")
    return _workspace(ws_bytes, device)


def spec_verify_linear(target, draft, draft_tokens, cu_draft, temperature, seed: int, *,
                       max_k: int, rule: int = SPEC_RULE_STRICT,
                       draft_kind: int = SPEC_DRAFT_LOGITS, draft_idx=None, want_pq=False,
                       workspace=None, out=None, stream=None):
    """Verifies a batch of linear drafts on the GPU.

    Returns (tokens [B, max_k+1] int32, accepted [B] int32, pq [R_d, 2] or
    None, workspace). See include/specverify.h for the semantics.
    """
    torch = _torch()
    B = cu_draft.numel() - 1
    V = target.shape[1]
    dev = target.device
    ws = _linear_workspace(B, max_k, V, rule, dev, workspace)
    if out is None:
        tokens = torch.empty(B, max_k + 1, dtype=torch.int32, device=dev)
        accepted = torch.empty(B, dtype=torch.int32, device=dev)
        pq = torch.empty(draft_tokens.numel(), 2, dtype=torch.float32, device=dev) if want_pq else None
    else:
        tokens, accepted, pq = out
    ddt = _dtype_code(draft) if draft is not None else SPEC_BF16
    code = lib().spec_verify_linear(
        _ptr(target), _dtype_code(target), _ptr(draft), ddt, draft_kind, _ptr(draft_idx),
        _ptr(draft_tokens), _ptr(cu_draft), _ptr(temperature), B, V, max_k,
        ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF), rule, _ptr(tokens), _ptr(accepted),
        _ptr(pq), _ptr(ws), ctypes.c_size_t(ws.numel() * ws.element_size()), _stream(stream))
    _check(code, "spec_verify_linear")
    return tokens, accepted, pq, ws


def spec_verify_linear_ext(target, draft, draft_tokens, cu_draft, temperature, seed: int, *,
                           max_k: int, rule: int = SPEC_RULE_STRICT,
                           draft_kind: int = SPEC_DRAFT_LOGITS, draft_idx=None, alpha=0.0,
                           max_rank=0, min_prob=0.0, lazy=False, resident=False, eager=False,
                           want_pq=False, want_rank=False, want_kl=False, seed_dev=None,
                           workspace=None, out=None, stream=None):
    """spec_verify_linear with the relaxed CACTUS rule's options and target
    ranks. `lazy`, `resident` and `eager` set SPEC_EXT_LAZY,
    SPEC_EXT_RESIDENT and SPEC_EXT_EAGER (the schedules of
    include/specverify.h).

    Returns (tokens, accepted, pq or None, rank [R_d] int32 or None,
    kl [R_d] f32 or None, workspace).
    """
    torch = _torch()
    B = cu_draft.numel() - 1
    V = target.shape[1]
    dev = target.device
    ws = _linear_workspace(B, max_k, V, rule, dev, workspace)
    if out is None:
        tokens = torch.empty(B, max_k + 1, dtype=torch.int32, device=dev)
        accepted = torch.empty(B, dtype=torch.int32, device=dev)
        pq = torch.empty(draft_tokens.numel(), 2, dtype=torch.float32, device=dev) if want_pq else None
        rank = torch.empty(draft_tokens.numel(), dtype=torch.int32, device=dev) if want_rank else None
        kl = torch.empty(draft_tokens.numel(), dtype=torch.float32, device=dev) if want_kl else None
    else:
        tokens, accepted, pq, rank, kl = out
    flags = ((SPEC_EXT_LAZY if lazy else 0) | (SPEC_EXT_RESIDENT if resident else 0)
             | (SPEC_EXT_EAGER if eager else 0))
    ext = SpecLinearExt(float(alpha), int(max_rank), float(min_prob), flags, _ptr(rank),
                        _ptr(kl), _ptr(seed_dev))
    ddt = _dtype_code(draft) if draft is not None else SPEC_BF16
    code = lib().spec_verify_linear_ext(
        _ptr(target), _dtype_code(target), _ptr(draft), ddt, draft_kind, _ptr(draft_idx),
        _ptr(draft_tokens), _ptr(cu_draft), _ptr(temperature), B, V, max_k,
        ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF), rule, ctypes.byref(ext), _ptr(tokens),
        _ptr(accepted), _ptr(pq), _ptr(ws), ctypes.c_size_t(ws.numel() * ws.element_size()), _stream(stream))
    _check(code, "spec_verify_linear_ext")
    return tokens, accepted, pq, rank, kl, ws


def spec_verify_tree_workspace(B: int, n_nodes: int, V: int, max_depth: int, max_branch: int) -> int:
    return int(lib().spec_verify_tree_workspace(B, n_nodes, V, max_depth, max_branch))


def spec_verify_tree(target, draft, node_token, parent, cu_nodes, temperature, seed: int, *,
                     max_depth: int, max_branch: int, draft_kind: int = SPEC_DRAFT_LOGITS,
                     node_fixed=None, seed_dev=None, workspace=None, out=None, stream=None):
    """Verifies a batch of draft trees (RRSw) on the GPU. With `node_fixed`
    ([n_nodes] int32, nonzero = a point-mass child) or `seed_dev` (a device
    uint64 tensor read as the seed when the walk runs) the call goes through
    spec_verify_tree_ext.

    Returns (tokens [B, max_depth+1], accepted [B], path [B, max_depth+1],
    workspace).
    """
    torch = _torch()
    B = cu_nodes.numel() - 1
    n_nodes, V = target.shape
    dev = target.device
    ws_bytes = spec_verify_tree_workspace(B, n_nodes, V, max_depth, max_branch)
    if ws_bytes == 0:
        raise SpecError(SPEC_ERR_INVALID_ARG, "spec_verify_tree_workspace")
    ws = _workspace(ws_bytes, dev, workspace)
    if out is None:
        tokens = torch.empty(B, max_depth + 1, dtype=torch.int32, device=dev)
        accepted = torch.empty(B, dtype=torch.int32, device=dev)
        path = torch.empty(B, max_depth + 1, dtype=torch.int32, device=dev)
    else:
        tokens, accepted, path = out
    ddt = _dtype_code(draft) if draft is not None else SPEC_BF16
    head = (_ptr(target), _dtype_code(target), _ptr(draft), ddt, draft_kind, _ptr(node_token),
            _ptr(parent))
    mid = (_ptr(cu_nodes), _ptr(temperature), B, n_nodes, V, max_depth, max_branch,
           ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF))
    tail = (_ptr(tokens), _ptr(accepted), _ptr(path), _ptr(ws), ctypes.c_size_t(ws.numel() * ws.element_size()),
            _stream(stream))
    if node_fixed is None and seed_dev is None:
        code = lib().spec_verify_tree(*head, *mid, *tail)
        _check(code, "spec_verify_tree")
    else:
        code = lib().spec_verify_tree_ext(*head, _ptr(node_fixed), *mid, _ptr(seed_dev), *tail)
        _check(code, "spec_verify_tree_ext")
    return tokens, accepted, path, ws


def draft_topk_softmax_workspace(rows: int, V: int) -> int:
    return int(lib().draft_topk_softmax_workspace(rows, V))


def draft_topk_softmax(draft_logits, cu_rows, temperature, *, workspace=None, out=None,
                       stream=None):
    """Top-128 ids (ascending) and softmax(z/T) over them for every row.
    Returns (idx [rows, 128] int32, prob [rows, 128] f32, workspace)."""
    torch = _torch()
    rows, V = draft_logits.shape
    B = cu_rows.numel() - 1
    dev = draft_logits.device
    ws = _workspace(draft_topk_softmax_workspace(rows, V), dev, workspace)
    if out is None:
        idx = torch.empty(rows, SPEC_TOPK, dtype=torch.int32, device=dev)
        prob = torch.empty(rows, SPEC_TOPK, dtype=torch.float32, device=dev)
    else:
        idx, prob = out
    code = lib().draft_topk_softmax(
        _ptr(draft_logits), _dtype_code(draft_logits), rows, V, _ptr(cu_rows),
        _ptr(temperature), B, SPEC_TOPK, _ptr(idx), _ptr(prob), _ptr(ws),
        ctypes.c_size_t(ws.numel() * ws.element_size()), _stream(stream))
    _check(code, "draft_topk_softmax")
    return idx, prob, ws


def spec_rheo_expand_workspace(F: int, V: int) -> int:
    return int(lib().spec_rheo_expand_workspace(F, V))


def spec_rheo_expand(draft, cu_frontier, frontier_score, temperature, seed: int, level: int,
                     *, K: int, m: int = 1, eps: float = 1e-6, n_keep: int = 0,
                     want_qproxy=True, want_qtrue=True, workspace=None, out=None,
                     stream=None):
    """One level of RheoSampling tree expansion (see spec_rheo_expand in
    include/specverify.h). Returns (child_token [F, K] int32, child_qproxy
    [F, K] f32 or None, child_qtrue [F, K] f32 or None, child_score [F, K] f32,
    keep [B, n_keep] int32, workspace)."""
    torch = _torch()
    F, V = draft.shape
    B = cu_frontier.numel() - 1
    dev = draft.device
    ws = _workspace(spec_rheo_expand_workspace(F, V), dev, workspace)
    if out is None:
        token = torch.empty(F, K, dtype=torch.int32, device=dev)
        qproxy = torch.empty(F, K, dtype=torch.float32, device=dev) if want_qproxy else None
        qtrue = torch.empty(F, K, dtype=torch.float32, device=dev) if want_qtrue else None
        score = torch.empty(F, K, dtype=torch.float32, device=dev)
        keep = torch.empty(B, n_keep, dtype=torch.int32, device=dev)
    else:
        token, qproxy, qtrue, score, keep = out
    code = lib().spec_rheo_expand(
        _ptr(draft), _dtype_code(draft), _ptr(cu_frontier), _ptr(frontier_score),
        _ptr(temperature), B, F, V, K, m, ctypes.c_float(eps), n_keep, ctypes.c_uint64(seed),
        level, _ptr(token), _ptr(qproxy), _ptr(qtrue), _ptr(score),
        _ptr(keep) if n_keep > 0 else None, _ptr(ws), ctypes.c_size_t(ws.numel() * ws.element_size()),
        _stream(stream))
    _check(code, "spec_rheo_expand")
    return token, qproxy, qtrue, score, keep, ws


def spec_set_fused_limit(nbytes: int) -> int:
    """Sets the largest call (bytes of rows) the fused small-batch kernel
    takes (0: never); returns the previous limit."""
    return int(lib().spec_set_fused_limit(ctypes.c_size_t(nbytes)))


def spec_get_status(workspace, stream=None) -> int:
    """Synchronises the stream and returns the device status word."""
    v = ctypes.c_int(0)
    _check(lib().spec_get_status(_ptr(workspace), _stream(stream), ctypes.byref(v)),
           "spec_get_status")
    return v.value


def spec_uniforms(seed: int, b, pos, stream_id, stream=None):
    """The verifier's uniforms u(seed, b[i], pos[i], stream_id[i])."""
    torch = _torch()
    out = torch.empty(b.numel(), dtype=torch.float32, device=b.device)
    _check(lib().spec_uniforms(ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF), _ptr(b), _ptr(pos),
                               _ptr(stream_id), b.numel(), _ptr(out), _stream(stream)),
           "spec_uniforms")
    return out


def spec_wait_selftest(kind: int, limit_ns: int, workspace=None, stream=None):
    """Runs the bounded-wait self-test (kind 0: mbarrier, 1: global word);
    returns the workspace, whose status word then reads SPEC_ERR_TIMEOUT."""
    torch = _torch()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda") if workspace is None else workspace
    _check(lib().spec_wait_selftest(int(kind), ctypes.c_ulonglong(limit_ns), _ptr(ws),
                                    _stream(stream)), "spec_wait_selftest")
    return ws


def spec_check_selftest(workspace=None, stream=None):
    """Runs the bounds-checked build's self-test (use_checked_library(True)
    first); returns the 512-byte workspace, whose status word then reads
    SPEC_ERR_BOUNDS. The product library raises SPEC_ERR_UNSUPPORTED."""
    torch = _torch()
    ws = torch.zeros(512, dtype=torch.uint8, device="cuda") if workspace is None else workspace
    _check(lib().spec_check_selftest(_ptr(ws), ctypes.c_size_t(ws.numel() * ws.element_size()), _stream(stream)),
           "spec_check_selftest")
    return ws


def spec_profile_row_pass(before=None, after=None):
    """Registers two torch.cuda.Event objects (enable_timing=True) that the
    next verify call on this thread records around its row-statistics pass."""
    def ev(e):
        if e is None:
            return None
        if not e.cuda_event:     # torch creates the CUDA event on first record
            e.record()
        return ctypes.c_void_p(e.cuda_event)
    _check(lib().spec_profile_row_pass(ev(before), ev(after)), "spec_profile_row_pass")


def spec_profile_pending() -> bool:
    """True while events registered with spec_profile_row_pass have not been
    taken by a call: after a call, whether that call recorded them."""
    return bool(lib().spec_profile_pending())

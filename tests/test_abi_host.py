"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function the header declares, sizes its workspaces, and rejects bad
arguments before launching anything."""
import ctypes

import pytest

import speculative_decoding_rejection_gb300 as sv


@pytest.fixture(scope="module")
def L():
    try:
        return sv.lib()
    except RuntimeError as e:
        pytest.fail(f"library not built: {e}")


def test_exports_every_declared_function(L):
    names = sv.header_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(sv._SIGS)


def test_status_strings(L):
    for code, name in [(0, "SPEC_OK"), (-1, "SPEC_ERR_INVALID_ARG"), (-3, "SPEC_ERR_WORKSPACE"),
                       (-5, "SPEC_ERR_TIMEOUT"), (7, "SPEC_ERR_UNKNOWN")]:
        assert sv.spec_status_string(code) == name


def test_workspace_sizes():
    assert sv.spec_verify_linear_workspace(1024, 4, 201088) > 0
    assert sv.spec_verify_linear_workspace(4, 4, 1024, sv.SPEC_RULE_STRICT_TOP128) > \
        sv.spec_verify_linear_workspace(4, 4, 1024, sv.SPEC_RULE_STRICT)
    assert sv.spec_verify_linear_workspace(-1, 4, 100) == 0
    assert sv.spec_verify_linear_workspace(4, 4, 0) == 0
    assert sv.spec_verify_linear_workspace(4, 100000, 100) == 0
    assert sv.draft_topk_softmax_workspace(10, 1000) > 0
    assert sv.draft_topk_softmax_workspace(10, 0) == 0


def _align256(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("rows,V", [(10, 4096), (1792, 151936), (7, 4088), (7, 4095),
                                    (3, 100)])
def test_top128_workspace_holds_the_candidate_lists(rows, V):
    """The two-launch select (V % 8 == 0, V >= 4096) keeps per row a list of
    512 eight-byte keys and one count word after the 256-byte header; other
    shapes take the one-launch select and need the header only."""
    lists = V % 8 == 0 and V >= 4096
    want = 256 + ((_align256(rows * 512 * 8) + _align256(rows * 4)) if lists else 0)
    assert sv.draft_topk_softmax_workspace(rows, V) == want


@pytest.mark.parametrize("F,V", [(640, 128256), (8, 1000), (8, 4100)])
def test_construction_workspace_holds_the_candidate_lists(F, V):
    """spec_rheo_expand's workspace: the 256-byte header, and the candidate
    lists of the two-launch select when its rows take it."""
    lists = V % 8 == 0 and V >= 4096
    want = 256 + ((_align256(F * 512 * 8) + _align256(F * 4)) if lists else 0)
    assert sv.spec_rheo_expand_workspace(F, V) == want


def test_top128_workload_fits_the_no_alloc_scratch():
    """B=256, K=7, V=151936 under the top-128 rule (its candidate lists
    included) fits the 16 MiB the no-alloc entry point holds."""
    need = sv.spec_verify_linear_workspace(256, 7, 151936, sv.SPEC_RULE_STRICT_TOP128)
    assert 0 < need <= 16 << 20
    # the lists are part of it: 1792 rows x 4 KB
    assert need - sv.spec_verify_linear_workspace(256, 7, 151936, sv.SPEC_RULE_STRICT) > 1792 * 4096


FAKE = 1 << 20   # a 256-byte-aligned non-null value; never dereferenced


def lin_args(**kw):
    args = dict(target=FAKE, tdt=1, draft=FAKE, ddt=1, dk=0, draft_idx=None, tokens=FAKE,
                cu=FAKE, temp=FAKE, B=4, V=1000, max_k=4, seed=1, rule=0, out_tokens=FAKE,
                out_acc=FAKE, out_pq=None, ws=FAKE, ws_bytes=1 << 30, stream=None)
    args.update(kw)
    return args


def lin(L, **kw):
    return L.spec_verify_linear(*lin_args(**kw).values())


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), sv.SPEC_ERR_INVALID_ARG),
    (dict(V=0), sv.SPEC_ERR_INVALID_ARG),
    (dict(V=(1 << 24) + 1), sv.SPEC_ERR_INVALID_ARG),
    (dict(max_k=-1), sv.SPEC_ERR_INVALID_ARG),
    (dict(max_k=257), sv.SPEC_ERR_UNSUPPORTED),
    (dict(tdt=5), sv.SPEC_ERR_INVALID_ARG),
    (dict(dk=3), sv.SPEC_ERR_INVALID_ARG),
    (dict(rule=9), sv.SPEC_ERR_INVALID_ARG),
    (dict(rule=2, dk=1), sv.SPEC_ERR_INVALID_ARG),
    (dict(dk=2, ddt=1, draft_idx=FAKE), sv.SPEC_ERR_INVALID_ARG),
    (dict(dk=2, ddt=0, draft_idx=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(target=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(tokens=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(target=FAKE + 8), sv.SPEC_ERR_INVALID_ARG),
    (dict(out_pq=FAKE + 2), sv.SPEC_ERR_INVALID_ARG),
    (dict(ws=None), sv.SPEC_ERR_WORKSPACE),
    (dict(ws=FAKE + 128), sv.SPEC_ERR_WORKSPACE),
    (dict(ws_bytes=100), sv.SPEC_ERR_WORKSPACE),
])
def test_linear_rejects_bad_arguments_on_the_host(L, kw, code):
    assert lin(L, **kw) == code


@pytest.mark.parametrize("flags", [sv.SPEC_EXT_EAGER | sv.SPEC_EXT_LAZY,
                                   sv.SPEC_EXT_EAGER | sv.SPEC_EXT_RESIDENT, 8, -1])
def test_linear_ext_rejects_bad_schedule_flags_on_the_host(L, flags):
    """The eager schedule combines with neither position-lazy one; unknown
    flag bits are invalid. Nothing is launched (the pointers are fake)."""
    import ctypes
    ext = sv.SpecLinearExt(0.0, 0, 0.0, flags, None, None, None)
    a = lin_args()
    code = L.spec_verify_linear_ext(*list(a.values())[:14], ctypes.byref(ext),
                                    *list(a.values())[14:])
    assert code == sv.SPEC_ERR_INVALID_ARG


def test_topk_rejects_bad_arguments_on_the_host(L):
    f = L.draft_topk_softmax
    ok = dict(logits=FAKE, dt=1, rows=8, V=1000, cu=FAKE, temp=FAKE, B=2, k=128, idx=FAKE,
              prob=FAKE, ws=FAKE, ws_bytes=256, stream=None)
    for kw, code in [(dict(k=64), sv.SPEC_ERR_UNSUPPORTED), (dict(V=0), sv.SPEC_ERR_INVALID_ARG),
                     (dict(dt=4), sv.SPEC_ERR_INVALID_ARG), (dict(cu=None), sv.SPEC_ERR_INVALID_ARG),
                     (dict(logits=FAKE + 4), sv.SPEC_ERR_INVALID_ARG),
                     (dict(ws=None), sv.SPEC_ERR_WORKSPACE), (dict(ws_bytes=8), sv.SPEC_ERR_WORKSPACE),
                     # rows the two-launch select takes need their candidate lists too
                     (dict(V=4096, ws_bytes=256), sv.SPEC_ERR_WORKSPACE)]:
        a = dict(ok)
        a.update(kw)
        assert f(*a.values()) == code, kw


def test_status_and_uniform_argument_checks(L):
    v = ctypes.c_int(0)
    assert L.spec_get_status(None, None, ctypes.byref(v)) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_get_status(FAKE + 4, None, ctypes.byref(v)) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_uniforms(1, None, None, None, -1, None, None) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_uniforms(1, None, None, None, 0, None, None) == sv.SPEC_OK


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(sv, "_lib", None)
    monkeypatch.setattr(sv, "_lib_path", tmp_path / "missing.so")
    with pytest.raises(RuntimeError, match="not built"):
        sv.lib()


def test_wait_selftest_rejects_bad_arguments(L):
    assert L.spec_wait_selftest(2, 1000, FAKE, None) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_wait_selftest(0, 0, FAKE, None) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_wait_selftest(0, 20 * 10 ** 9, FAKE, None) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_wait_selftest(1, 1000, None, None) == sv.SPEC_ERR_WORKSPACE
    assert L.spec_wait_selftest(1, 1000, FAKE + 16, None) == sv.SPEC_ERR_WORKSPACE


def test_rheo_expand_rejects_bad_arguments_on_the_host(L):
    f = L.spec_rheo_expand
    ws = sv.spec_rheo_expand_workspace(8, 1000)
    assert ws >= 256
    assert sv.spec_rheo_expand_workspace(-1, 1000) == 0
    assert sv.spec_rheo_expand_workspace(8, 0) == 0
    ok = dict(draft=FAKE, ddt=1, cu=FAKE, fscore=FAKE, temp=FAKE, B=2, F=8, V=1000, K=10, m=1,
              eps=1e-6, n_keep=10, seed=1, level=0, token=FAKE, qproxy=None, qtrue=None,
              score=FAKE, keep=FAKE, ws=FAKE, ws_bytes=ws, stream=None)
    for kw, code in [(dict(K=0), sv.SPEC_ERR_INVALID_ARG), (dict(K=129), sv.SPEC_ERR_INVALID_ARG),
                     (dict(V=5, K=6), sv.SPEC_ERR_INVALID_ARG),
                     (dict(m=10), sv.SPEC_ERR_INVALID_ARG), (dict(m=-1), sv.SPEC_ERR_INVALID_ARG),
                     (dict(eps=-1.0), sv.SPEC_ERR_INVALID_ARG),
                     (dict(eps=float("inf")), sv.SPEC_ERR_INVALID_ARG),
                     (dict(level=1 << 24), sv.SPEC_ERR_INVALID_ARG),
                     (dict(n_keep=-1), sv.SPEC_ERR_INVALID_ARG),
                     (dict(n_keep=sv.SPEC_RHEO_MAX_CANDIDATES + 1), sv.SPEC_ERR_UNSUPPORTED),
                     (dict(ddt=3), sv.SPEC_ERR_INVALID_ARG),
                     (dict(draft=FAKE + 8), sv.SPEC_ERR_INVALID_ARG),
                     (dict(keep=None), sv.SPEC_ERR_INVALID_ARG),
                     (dict(score=None), sv.SPEC_ERR_INVALID_ARG),
                     (dict(cu=None), sv.SPEC_ERR_INVALID_ARG),
                     (dict(ws=None), sv.SPEC_ERR_WORKSPACE),
                     (dict(ws_bytes=ws - 1), sv.SPEC_ERR_WORKSPACE)]:
        a = dict(ok)
        a.update(kw)
        assert f(*a.values()) == code, kw


def test_tree_ext_rejects_a_misaligned_flag_array(L):
    args = [FAKE, 1, FAKE, 1, 0, FAKE, FAKE, FAKE + 2, FAKE, FAKE, 2, 128, 1000, 6, 4, 1,
            None, FAKE, FAKE, None, FAKE, 1 << 20, None]
    assert L.spec_verify_tree_ext(*args) == sv.SPEC_ERR_INVALID_ARG
    args[7], args[16] = FAKE, FAKE + 4                     # a misaligned seed pointer
    assert L.spec_verify_tree_ext(*args) == sv.SPEC_ERR_INVALID_ARG

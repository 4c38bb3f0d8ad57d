"""Host-only checks of the C ABI: the library builds for sm_103a, loads, exports
every function include/dsa.h declares, and rejects bad arguments before any
launch (so none of these calls touches a GPU)."""
import ctypes

import pytest

from long_context_sparse_dsa_gb300 import build as dsa_build

dsa = pytest.importorskip("long_context_sparse_dsa_gb300")


@pytest.fixture(scope="module")
def lib():
    dsa_build.build()
    return dsa.library()


def test_every_declared_symbol_is_exported(lib):
    names = dsa.header_functions()
    assert {"dsa_pool_keys", "dsa_indexer_score", "dsa_topk", "dsa_sparse_attn_fwd", "dsa_sparse_attn_bwd",
            "dsa_layer_fwd", "dsa_layer_bwd", "dsa_check_device_error", "dsa_workspace_bytes"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for s in range(7):
        assert dsa.status_string(s) not in ("", "unknown status")
    assert dsa.status_string(99) == "unknown status"


def _dims(**kw):
    base = dict(L=4096, Hq=16, d=128, Hi=8, di=64, k=512, q_chunk=1024, dtype="bf16")
    base.update(kw)
    return dsa.make_dims(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(), dsa.DSA_OK),
    (dict(L=4094), dsa.DSA_ERR_INVALID_ARG),
    (dict(L=0), dsa.DSA_ERR_INVALID_ARG),
    (dict(k=0), dsa.DSA_ERR_INVALID_ARG),
    (dict(q_chunk=0), dsa.DSA_ERR_INVALID_ARG),
    (dict(d=96), dsa.DSA_ERR_UNSUPPORTED),
    (dict(di=32), dsa.DSA_ERR_UNSUPPORTED),
    (dict(Hq=8), dsa.DSA_ERR_UNSUPPORTED),          # bf16 needs 16 or 32 heads: no silent fallback
    (dict(Hi=6), dsa.DSA_ERR_UNSUPPORTED),
    (dict(k=2048), dsa.DSA_ERR_UNSUPPORTED),
    (dict(pool=8), dsa.DSA_ERR_UNSUPPORTED),
    (dict(Hq=8, dtype="fp32"), dsa.DSA_OK),
    (dict(Hq=3, Hi=3, dtype="fp32"), dsa.DSA_OK),
])
def test_validate_dims(lib, kw, status):
    assert dsa.validate_dims(_dims(**kw)) == status


def test_fp32_backward_is_rejected_not_faked(lib):
    assert dsa.validate_dims(_dims(Hq=8, dtype="fp32"), with_backward=True) == dsa.DSA_ERR_UNSUPPORTED


def test_bwd_workspace_bytes(lib):
    assert dsa.bwd_workspace_bytes(_dims(L=131072)) == 131072 * 16 * 4
    assert dsa.bwd_workspace_bytes(_dims(Hq=8, dtype="fp32")) == 0     # no fp32 backward


def _fused_ws(C, P):
    """The documented parts of the fused indexer + top-k workspace, each rounded up to 256 bytes."""
    a = lambda b: (b + 255) // 256 * 256
    nb = (C + 31) // 32
    nseg = (P + 2047) // 2048
    stride = max(4096, 64 * nseg)
    return (a(C * P * 4) + a(C * ((P + 31) // 32) * 4) + a(C * stride * 8) + a(C * nseg * 16)
            + 2 * a(C * 4) + 2 * a(nb * 4) + a(16))   # scores, samples, candidates, lengths, tau, row list, blocks


def test_workspace_bytes(lib):
    assert dsa.workspace_bytes(_dims(L=131072, q_chunk=8192)) == _fused_ws(8192, 32768)
    assert dsa.workspace_bytes(_dims(L=4096, q_chunk=100)) == _fused_ws(100, 1024)
    assert dsa.indexer_topk_workspace_bytes(_dims(L=4096, q_chunk=100), 37) == _fused_ws(37, 1024)
    # fp32 layers run the unfused pair: the score block only
    assert dsa.workspace_bytes(_dims(L=4096, q_chunk=100, Hq=8, dtype="fp32")) == (100 * 1024 * 4 + 255) // 256 * 256
    assert dsa.workspace_bytes(_dims(L=4094)) == 0
    assert dsa.indexer_topk_workspace_bytes(_dims(L=4096), 0) == 0
    assert dsa.indexer_topk_workspace_bytes(_dims(L=4096), 4097) == 0


def test_null_and_misaligned_pointers_fail_before_launch(lib):
    d = _dims()
    assert lib.dsa_pool_keys(ctypes.byref(d), None, ctypes.c_void_p(256), None) == dsa.DSA_ERR_INVALID_ARG
    assert b"k_idx" in lib.dsa_last_error_message()
    assert lib.dsa_pool_keys(ctypes.byref(d), ctypes.c_void_p(264), ctypes.c_void_p(256), None) == \
        dsa.DSA_ERR_INVALID_ARG
    assert b"aligned" in lib.dsa_last_error_message()
    assert lib.dsa_indexer_score(ctypes.byref(d), 256, 256, 256, 4000, 200, 256, None) == dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_topk(ctypes.byref(d), 256, -1, 10, 256, None) == dsa.DSA_ERR_INVALID_ARG
    # an empty query range is an error, not a silent no-op
    assert lib.dsa_topk(ctypes.byref(d), 256, 0, 0, 256, None) == dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_indexer_score(ctypes.byref(d), 256, 256, 256, 8, 0, 256, None) == dsa.DSA_ERR_INVALID_ARG
    # the fused indexer + top-k: range, pointers and workspace are checked before any launch
    p = ctypes.c_void_p(256)
    assert lib.dsa_indexer_topk(ctypes.byref(d), p, p, p, 4000, 200, p, p, 1 << 40, None) == dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_indexer_topk(ctypes.byref(d), p, None, p, 0, 200, p, p, 1 << 40, None) == dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_indexer_topk(ctypes.byref(d), p, p, p, 0, 200, p, p, 16, None) == dsa.DSA_ERR_WORKSPACE
    assert lib.dsa_indexer_topk(ctypes.byref(d), p, p, p, 0, 200, p, None, 1 << 40, None) == dsa.DSA_ERR_WORKSPACE
    assert lib.dsa_indexer_topk(ctypes.byref(d), p, p, p, 0, 200, p, ctypes.c_void_p(264), 1 << 40, None) == \
        dsa.DSA_ERR_INVALID_ARG
    # too small a workspace is reported as such
    p = ctypes.c_void_p(256)
    assert lib.dsa_layer_fwd(ctypes.byref(d), p, p, p, p, p, p, p, p, None, p, p, p, 16, None) == \
        dsa.DSA_ERR_WORKSPACE
    assert lib.dsa_layer_fwd(ctypes.byref(d), p, p, p, p, p, p, p, p, None, p, p, None, 1 << 40, None) == \
        dsa.DSA_ERR_WORKSPACE
    # the optional fp32 output is checked only when given
    odd = ctypes.c_void_p(264)          # 8 mod 16
    assert lib.dsa_layer_fwd(ctypes.byref(d), p, p, p, p, p, p, p, p, odd, p, p, p, 16, None) == \
        dsa.DSA_ERR_INVALID_ARG
    assert b"o_acc" in lib.dsa_last_error_message()
    assert lib.dsa_sparse_attn_fwd(ctypes.byref(d), p, p, p, p, p, p, odd, None) == dsa.DSA_ERR_INVALID_ARG
    # aliased gradient outputs
    assert lib.dsa_sparse_attn_bwd(ctypes.byref(d), p, p, p, p, p, p, None, p, p, p, p, None, 0, None) == \
        dsa.DSA_ERR_INVALID_ARG
    # without o_acc the backward needs its D workspace; with a misaligned one it fails on that
    q = ctypes.c_void_p(512)
    assert lib.dsa_sparse_attn_bwd(ctypes.byref(d), p, p, p, p, p, p, None, p, p, p, q, None, 0, None) == \
        dsa.DSA_ERR_WORKSPACE
    assert lib.dsa_sparse_attn_bwd(ctypes.byref(d), p, p, p, p, p, p, odd, p, p, p, q, None, 0, None) == \
        dsa.DSA_ERR_INVALID_ARG
    assert b"o_acc" in lib.dsa_last_error_message()
    assert lib.dsa_selftest_bounded_wait(0, None) == dsa.DSA_ERR_INVALID_ARG


def test_noalloc_checks_every_pointer_before_anything_is_enqueued(lib):
    """dsa_layer_fwd_noalloc rejects a NULL or misaligned tensor pointer with
    DSA_ERR_INVALID_ARG before it touches the GPU: on a host without a GPU any
    CUDA call it made first (the scratch array's address, a launch) would
    report DSA_ERR_CUDA instead."""
    d = _dims()
    p = ctypes.c_void_p(256)
    names = ["q", "k", "v", "q_idx", "k_idx", "w", "o", "lse", "idx", "kpool"]
    for i, name in enumerate(names):
        for bad in (None, ctypes.c_void_p(264)):
            args = [p] * len(names)
            args[i] = bad
            assert lib.dsa_layer_fwd_noalloc(ctypes.byref(d), *args, None) == dsa.DSA_ERR_INVALID_ARG, name
            assert name.encode() in lib.dsa_last_error_message()


def test_deterministic_backward_validates_before_launch(lib):
    d = _dims()
    p, q, odd = ctypes.c_void_p(256), ctypes.c_void_p(512), ctypes.c_void_p(264)
    f = lib.dsa_sparse_attn_bwd_det
    need = dsa.bwd_det_workspace_bytes(d)
    assert need > 4096 * 512 * 4          # at least the inverted selection's query lists
    #        q  k  v  idx o  lse o_acc dout dq dk dv ws ws_bytes
    assert f(ctypes.byref(d), p, p, p, p, p, p, None, p, p, p, q, None, 0, None) == dsa.DSA_ERR_WORKSPACE
    assert f(ctypes.byref(d), p, p, p, p, p, p, None, p, p, p, q, p, need - 1, None) == dsa.DSA_ERR_WORKSPACE
    assert f(ctypes.byref(d), p, p, p, p, p, p, None, p, p, p, q, odd, need, None) == dsa.DSA_ERR_INVALID_ARG
    assert f(ctypes.byref(d), p, p, p, None, p, p, None, p, p, p, q, p, need, None) == dsa.DSA_ERR_INVALID_ARG
    assert f(ctypes.byref(d), p, p, p, p, p, p, None, p, p, p, p, p, need, None) == dsa.DSA_ERR_INVALID_ARG  # dk == dv
    assert f(ctypes.byref(d), p, p, p, p, p, p, odd, p, p, p, q, p, need, None) == dsa.DSA_ERR_INVALID_ARG
    assert f(ctypes.byref(_dims(Hq=8, dtype="fp32")), p, p, p, p, p, p, None, p, p, p, q, p, need, None) == \
        dsa.DSA_ERR_UNSUPPORTED
    assert dsa.bwd_det_workspace_bytes(_dims(L=1 << 22, k=1024)) == 0     # L * (k + 1) >= 2^31


def test_probe_validates_before_launch(lib):
    p, odd = ctypes.c_void_p(256), ctypes.c_void_p(264)
    f = lib.dsa_probe_traffic
    d = _dims()
    assert f(ctypes.byref(_dims(d=96)), p, p, p, None, None, None) == dsa.DSA_ERR_UNSUPPORTED
    assert f(ctypes.byref(_dims(Hq=8, dtype="fp32")), p, p, p, None, None, None) == dsa.DSA_ERR_UNSUPPORTED
    assert f(ctypes.byref(_dims(L=4094)), p, p, p, None, None, None) == dsa.DSA_ERR_INVALID_ARG
    assert f(ctypes.byref(d), None, p, p, None, None, None) == dsa.DSA_ERR_INVALID_ARG
    assert f(ctypes.byref(d), p, odd, p, None, None, None) == dsa.DSA_ERR_INVALID_ARG
    assert f(ctypes.byref(d), p, p, None, None, None, None) == dsa.DSA_ERR_INVALID_ARG
    assert f(ctypes.byref(d), p, p, p, p, None, None) == dsa.DSA_ERR_INVALID_ARG      # only one of dk/dv
    assert f(ctypes.byref(d), p, p, p, p, odd, None) == dsa.DSA_ERR_INVALID_ARG


def test_binding_has_no_cpu_path():
    import inspect
    src = inspect.getsource(dsa)
    assert "oracle" not in src and "numpy" not in src


def test_route_setters_accept_only_their_routes(lib):
    """The two route hooks take 0 or 1 and nothing else; they only set a host
    variable (nothing is launched), and are left at their documented defaults
    (indexer + top-k: 1, attention forward: 0)."""
    for setter, default in ((lib.dsa_set_indexer_topk_route, 1), (lib.dsa_set_attn_fwd_route, 0)):
        assert setter(2) == 1 and setter(-1) == 1          # DSA_ERR_INVALID_ARG
        assert setter(0) == 0 and setter(1) == 0
        assert setter(default) == 0


def test_gated_pool_keys_validates_before_launch(lib):
    """NULL or misaligned pointers are rejected before anything is enqueued
    (the pointers below are never dereferenced: validation fails first)."""
    dims = dsa.make_dims(1024, 16, 128, 8, 64, 64)
    good = ctypes.c_void_p(1 << 20)
    for k, g, out in ((None, good, good), (good, None, good), (good, good, None),
                      (good, ctypes.c_void_p((1 << 20) + 4), good)):
        assert lib.dsa_pool_keys_gated(ctypes.byref(dims), k, g, out, None) == 1   # DSA_ERR_INVALID_ARG

"""GB300 (sm_103a) DeepSeek Sparse Attention layer: thin Python binding.

Every computation runs in the CUDA kernels of ``libdsa_gb300.so`` (built by
``build.py``); this module only marshals arguments through the C ABI of
``include/dsa.h``.  Tensors are torch CUDA tensors (torch provides device
memory and streams only).  There is no CPU path: if the library is missing
or no GPU is present, calls raise.

Entry points (same names as the C ABI, without the ``dsa_`` prefix):
pool_keys, indexer_score, topk, indexer_topk, sparse_attn_fwd, sparse_attn_bwd, sparse_attn_bwd_det,
layer_fwd, layer_bwd, check_device_error, workspace_bytes, indexer_topk_workspace_bytes,
bwd_workspace_bytes,
validate_dims, layer_fwd_noalloc; and the measurement probe probe_traffic
(``include/dsa_probe.h``).
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa_gb300.so")
INCLUDE_DIR = os.path.join(os.path.dirname(_HERE), "include")
HEADER_PATH = os.path.join(INCLUDE_DIR, "dsa.h")

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_WORKSPACE = 0, 1, 2, 3
DSA_ERR_CUDA, DSA_ERR_TIMEOUT, DSA_ERR_BAD_INDEX = 4, 5, 6
DSA_FP32, DSA_BF16 = 0, 1


class DSAError(RuntimeError):
    def __init__(self, status: int, func: str, message: str):
        self.status = status
        super().__init__(f"{func}: status {status} ({message})")


class Dims(ctypes.Structure):
    """Mirror of ``dsa_dims``."""
    _fields_ = [("L", ctypes.c_int64), ("Hq", ctypes.c_int32), ("d", ctypes.c_int32), ("Hi", ctypes.c_int32),
                ("di", ctypes.c_int32), ("pool", ctypes.c_int32), ("k", ctypes.c_int32),
                ("q_chunk", ctypes.c_int32), ("scale", ctypes.c_float), ("dtype", ctypes.c_int32)]


def make_dims(L, Hq, d, Hi, di, k, q_chunk=None, scale=None, dtype="bf16", pool=4) -> Dims:
    return Dims(int(L), int(Hq), int(d), int(Hi), int(di), int(pool), int(k), int(L if q_chunk is None else q_chunk),
                float(scale if scale is not None else d ** -0.5), DSA_BF16 if dtype == "bf16" else DSA_FP32)


_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with long_context_sparse_dsa_gb300.build.build() "
                              "(nvcc, sm_103a). There is no CPU fallback.")
        lib = ctypes.CDLL(LIB_PATH)
        P, i64, i32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32
        D = ctypes.POINTER(Dims)
        sig = {
            "dsa_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "dsa_last_error_message": ([], ctypes.c_char_p),
            "dsa_validate_dims": ([D, i32], ctypes.c_int),
            "dsa_workspace_bytes": ([D], ctypes.c_size_t),
            "dsa_bwd_workspace_bytes": ([D], ctypes.c_size_t),
            "dsa_pool_keys": ([D, P, P, P], ctypes.c_int),
            "dsa_pool_keys_gated": ([D, P, P, P, P], ctypes.c_int),
            "dsa_indexer_score": ([D, P, P, P, i64, i64, P, P], ctypes.c_int),
            "dsa_topk": ([D, P, i64, i64, P, P], ctypes.c_int),
            "dsa_indexer_topk": ([D, P, P, P, i64, i64, P, P, ctypes.c_size_t, P], ctypes.c_int),
            "dsa_indexer_topk_workspace_bytes": ([D, i64], ctypes.c_size_t),
            "dsa_sparse_attn_fwd": ([D, P, P, P, P, P, P, P, P], ctypes.c_int),
            "dsa_sparse_attn_bwd": ([D, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P], ctypes.c_int),
            "dsa_layer_fwd": ([D, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P], ctypes.c_int),
            "dsa_layer_bwd": ([D, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P], ctypes.c_int),
            "dsa_sparse_attn_bwd_det": ([D, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P], ctypes.c_int),
            "dsa_bwd_det_workspace_bytes": ([D], ctypes.c_size_t),
            "dsa_layer_fwd_noalloc": ([D, P, P, P, P, P, P, P, P, P, P, P], ctypes.c_int),
            "dsa_check_device_error": ([P], ctypes.c_int),
            "dsa_set_wait_limit": ([u32], None),
            "dsa_set_indexer_topk_route": ([i32], ctypes.c_int),
            "dsa_set_attn_fwd_route": ([i32], ctypes.c_int),
            "dsa_selftest_bounded_wait": ([u32, P], ctypes.c_int),
            "dsa_probe_traffic": ([D, P, P, P, P, P, P], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
    return _lib


def library():
    """The loaded ctypes library (raises if it was not built)."""
    return _load()


def header_functions():
    """Names of the functions the headers under ``include/`` declare."""
    names = set()
    for fn in sorted(os.listdir(INCLUDE_DIR)):
        if fn.endswith(".h"):
            src = open(os.path.join(INCLUDE_DIR, fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names.update(re.findall(r"\b(dsa_[a-z_0-9]+)\s*\(", src))
    return sorted(names)


def status_string(status: int) -> str:
    return _load().dsa_status_string(status).decode()


def _check(status: int, func: str):
    if status != DSA_OK:
        msg = _load().dsa_last_error_message().decode() or status_string(status)
        raise DSAError(status, func, msg)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def validate_dims(dims: Dims, with_backward: bool = False) -> int:
    return _load().dsa_validate_dims(ctypes.byref(dims), int(bool(with_backward)))


def workspace_bytes(dims: Dims) -> int:
    return int(_load().dsa_workspace_bytes(ctypes.byref(dims)))


def bwd_workspace_bytes(dims: Dims) -> int:
    return int(_load().dsa_bwd_workspace_bytes(ctypes.byref(dims)))


def pool_keys(dims, k_idx, kpool, stream=None):
    _check(_load().dsa_pool_keys(ctypes.byref(dims), _ptr(k_idx), _ptr(kpool), _stream(stream)), "dsa_pool_keys")


def pool_keys_gated(dims, k_idx, gate, kpool, stream=None):
    """kpool[p] = sum_j gate[4p+j] * k_idx[4p+j] (gate: [L] fp32)."""
    _check(_load().dsa_pool_keys_gated(ctypes.byref(dims), _ptr(k_idx), _ptr(gate), _ptr(kpool), _stream(stream)),
           "dsa_pool_keys_gated")


def indexer_score(dims, q_idx, kpool, w, q_begin, q_count, scores, stream=None):
    _check(_load().dsa_indexer_score(ctypes.byref(dims), _ptr(q_idx), _ptr(kpool), _ptr(w), int(q_begin),
                                     int(q_count), _ptr(scores), _stream(stream)), "dsa_indexer_score")


def topk(dims, scores, q_begin, q_count, idx, stream=None):
    _check(_load().dsa_topk(ctypes.byref(dims), _ptr(scores), int(q_begin), int(q_count), _ptr(idx),
                            _stream(stream)), "dsa_topk")


def indexer_topk_workspace_bytes(dims, q_count) -> int:
    return int(_load().dsa_indexer_topk_workspace_bytes(ctypes.byref(dims), int(q_count)))


def indexer_topk(dims, q_idx, kpool, w, q_begin, q_count, idx, ws, ws_bytes=None, stream=None):
    """Indexer + top-k of one query range in one call; for bf16 layers route 1 (default) uses the score
    block in ws, route 0 the candidate lists (set_indexer_topk_route)."""
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(_load().dsa_indexer_topk(ctypes.byref(dims), _ptr(q_idx), _ptr(kpool), _ptr(w), int(q_begin), int(q_count),
                                    _ptr(idx), _ptr(ws), int(ws_bytes), _stream(stream)), "dsa_indexer_topk")


def sparse_attn_fwd(dims, q, k, v, idx, o, lse, stream=None, o_acc=None):
    """o_acc: optional fp32 [L, Hq, d] output (O with P carried beyond bf16)."""
    _check(_load().dsa_sparse_attn_fwd(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(o), _ptr(lse),
                                       _ptr(o_acc), _stream(stream)), "dsa_sparse_attn_fwd")


def sparse_attn_bwd(dims, q, k, v, idx, o, lse, dout, dq, dk, dv, ws=None, ws_bytes=None, stream=None, o_acc=None):
    """With o_acc (the forward's) the workspace is not needed."""
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(_load().dsa_sparse_attn_bwd(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(o), _ptr(lse),
                                       _ptr(o_acc), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), int(ws_bytes),
                                       _stream(stream)), "dsa_sparse_attn_bwd")


def bwd_det_workspace_bytes(dims) -> int:
    return int(_load().dsa_bwd_det_workspace_bytes(ctypes.byref(dims)))


def alloc_bwd_det_workspace(dims, device="cuda"):
    import torch
    n = bwd_det_workspace_bytes(dims)
    if n == 0:
        _check(validate_dims(dims, True), "dsa_bwd_det_workspace_bytes")
        raise DSAError(DSA_ERR_UNSUPPORTED, "dsa_bwd_det_workspace_bytes", "L * (k + 1) >= 2^31")
    return torch.empty((n,), dtype=torch.uint8, device=device)


def sparse_attn_bwd_det(dims, q, k, v, idx, o, lse, dout, dq, dk, dv, ws, ws_bytes=None, stream=None, o_acc=None):
    """Deterministic backward: dK/dV summed in a fixed order (bitwise reproducible)."""
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(_load().dsa_sparse_attn_bwd_det(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(o),
                                           _ptr(lse), _ptr(o_acc), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                                           int(ws_bytes), _stream(stream)), "dsa_sparse_attn_bwd_det")


def layer_fwd(dims, q, k, v, q_idx, k_idx, w, o, lse, idx, kpool, ws, ws_bytes=None, stream=None, o_acc=None):
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(_load().dsa_layer_fwd(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(q_idx), _ptr(k_idx), _ptr(w),
                                 _ptr(o), _ptr(lse), _ptr(o_acc), _ptr(idx), _ptr(kpool), _ptr(ws), int(ws_bytes),
                                 _stream(stream)), "dsa_layer_fwd")


def layer_fwd_noalloc(dims, q, k, v, q_idx, k_idx, w, o, lse, idx, kpool, stream=None):
    """dsa_layer_fwd with the score block in the library's fixed device array (no workspace)."""
    _check(_load().dsa_layer_fwd_noalloc(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(q_idx), _ptr(k_idx),
                                         _ptr(w), _ptr(o), _ptr(lse), _ptr(idx), _ptr(kpool), _stream(stream)),
           "dsa_layer_fwd_noalloc")


def layer_bwd(dims, q, k, v, idx, o, lse, dout, dq, dk, dv, ws=None, ws_bytes=None, stream=None, o_acc=None):
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(_load().dsa_layer_bwd(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(o), _ptr(lse),
                                 _ptr(o_acc), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), int(ws_bytes),
                                 _stream(stream)), "dsa_layer_bwd")


def check_device_error(stream=None):
    _check(_load().dsa_check_device_error(_stream(stream)), "dsa_check_device_error")


def probe_traffic(dims, k, v, idx, dk=None, dv=None, stream=None):
    """Replay the attention kernels' memory traffic for a selection, with no arithmetic (include/dsa_probe.h)."""
    _check(_load().dsa_probe_traffic(ctypes.byref(dims), _ptr(k), _ptr(v), _ptr(idx), _ptr(dk), _ptr(dv),
                                     _stream(stream)), "dsa_probe_traffic")


def set_indexer_topk_route(route: int):
    """Route of the bf16 indexer + top-k: 1 score block + row-wise top-k (default), 0 candidate lists."""
    _check(_load().dsa_set_indexer_topk_route(int(route)), "dsa_set_indexer_topk_route")


def set_attn_fwd_route(route: int):
    """Kernel of the bf16 attention forward: 0 warp-level m16n8k16 (default), 1 tcgen05 (d = 128)."""
    _check(_load().dsa_set_attn_fwd_route(int(route)), "dsa_set_attn_fwd_route")


def set_wait_limit(spins: int):
    _load().dsa_set_wait_limit(int(spins))


def selftest_bounded_wait(spins: int, stream=None):
    _check(_load().dsa_selftest_bounded_wait(int(spins), _stream(stream)), "dsa_selftest_bounded_wait")


@dataclass
class LayerBuffers:
    """Device buffers of one layer call (allocated by torch, owned by the caller)."""
    o: object
    lse: object
    idx: object
    kpool: object
    ws: object
    o_acc: object = None


def alloc_backward_workspace(dims: Dims, device="cuda"):
    import torch
    n = bwd_workspace_bytes(dims)
    if n == 0:
        _check(validate_dims(dims, True), "dsa_bwd_workspace_bytes")
    return torch.empty((n,), dtype=torch.uint8, device=device)


def alloc_forward_buffers(dims: Dims, device="cuda", o_acc: bool = False) -> LayerBuffers:
    """o_acc=True adds the fp32 [L, Hq, d] output the backward can take in place of its D pass."""
    import torch
    dt = torch.bfloat16 if dims.dtype == DSA_BF16 else torch.float32
    ws_bytes = workspace_bytes(dims)
    if ws_bytes == 0:
        _check(validate_dims(dims), "dsa_workspace_bytes")
    return LayerBuffers(
        o=torch.empty((dims.L, dims.Hq, dims.d), dtype=dt, device=device),
        lse=torch.empty((dims.L, dims.Hq), dtype=torch.float32, device=device),
        idx=torch.empty((dims.L, dims.k), dtype=torch.int32, device=device),
        kpool=torch.empty((dims.L // 4, dims.di), dtype=dt, device=device),
        ws=torch.empty((ws_bytes,), dtype=torch.uint8, device=device),
        o_acc=torch.empty((dims.L, dims.Hq, dims.d), dtype=torch.float32, device=device) if o_acc else None,
    )

"""CPU oracle for one DeepSeek Sparse Attention (DSA) layer, fp64.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product path never imports this
package.  The arithmetic lives in ``dsa_oracle.c`` (plain single-threaded C);
this module only builds it with gcc and marshals numpy arrays through ctypes.

Parity pins: see ``tests/test_oracle_pins.py``.  Every function is pinned by
at least one test that does not re-type its formula (closed forms, invariants,
brute force on tiny inputs, torch library routines on a different
formulation).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libdsa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32, f64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_double
            lib.oracle_round_bf16.argtypes = [ctypes.c_float]
            lib.oracle_round_bf16.restype = ctypes.c_float
            lib.oracle_pool_keys.argtypes = [i64, i32, i32, P, P]
            lib.oracle_pool_keys.restype = None
            lib.oracle_pool_keys_gated.argtypes = [i64, i32, i32, P, P, P]
            lib.oracle_pool_keys_gated.restype = None
            lib.oracle_indexer_scores.argtypes = [i64, i32, i32, P, P, P, P, i64, P]
            lib.oracle_indexer_scores.restype = None
            lib.oracle_topk.argtypes = [i64, i32, P, P, i64, P]
            lib.oracle_topk.restype = ctypes.c_int
            lib.oracle_key_set.argtypes = [i64, P, i32, P]
            lib.oracle_key_set.restype = i64
            lib.oracle_attn_fwd.argtypes = [i64, i32, i32, f64, P, i32, P, P, P, i32, P, i64, P, P]
            lib.oracle_attn_fwd.restype = ctypes.c_int
            lib.oracle_attn_bwd.argtypes = [i64, i32, i32, f64, P, i32, P, P, P, i32, P, P, i64, P, P, P]
            lib.oracle_attn_bwd.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _rows(rows, L):
    r = np.ascontiguousarray(np.arange(L, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64))
    if r.size and (r.min() < 0 or r.max() >= L):
        raise ValueError("row index out of range")
    return r


def elig(t):
    """Number of complete pools at or before token t."""
    return (np.asarray(t) + 1) // 4


def round_bf16(x: float) -> float:
    return float(_load().oracle_round_bf16(float(x)))


def pool_keys(k_I, round_to_bf16: bool) -> np.ndarray:
    """kpool[p] = k_I[4p] + k_I[4p+1] + k_I[4p+2] + k_I[4p+3] (fp32, then bf16 if asked)."""
    k_I = _f32(k_I)
    L, di = k_I.shape
    assert L % 4 == 0
    out = np.empty((L // 4, di), np.float32)
    _load().oracle_pool_keys(L, di, int(bool(round_to_bf16)), _ptr(k_I), _ptr(out))
    return out


def pool_keys_gated(k_I, gate, round_to_bf16: bool) -> np.ndarray:
    """kpool[p] = sum_j gate[4p+j] * k_I[4p+j] (fp32 fma chain in token order, then bf16 if asked)."""
    k_I = _f32(k_I)
    gate = _f32(gate)
    L, di = k_I.shape
    assert L % 4 == 0 and gate.shape == (L,)
    out = np.empty((L // 4, di), np.float32)
    _load().oracle_pool_keys_gated(L, di, int(bool(round_to_bf16)), _ptr(k_I), _ptr(gate), _ptr(out))
    return out


def indexer_scores(q_I, kpool, w, rows=None) -> np.ndarray:
    """fp64 scores [len(rows), P]; entries of pools a query may not see are NaN."""
    q_I, kpool, w = _f32(q_I), _f32(kpool), _f32(w)
    L, Hi, di = q_I.shape
    r = _rows(rows, L)
    out = np.empty((r.size, L // 4), np.float64)
    _load().oracle_indexer_scores(L, Hi, di, _ptr(q_I), _ptr(kpool), _ptr(w), _ptr(r), r.size, _ptr(out))
    return out


def topk(scores, L: int, k: int, rows=None) -> np.ndarray:
    """Selected pools per listed row, ascending, padded with -1: int32 [len(rows), k]."""
    s = np.ascontiguousarray(scores, dtype=np.float64)
    r = _rows(rows, L)
    assert s.shape == (r.size, L // 4)
    out = np.empty((r.size, k), np.int32)
    rc = _load().oracle_topk(L, k, _ptr(s), _ptr(r), r.size, _ptr(out))
    if rc:
        raise RuntimeError(f"oracle_topk failed ({rc})")
    return out


def key_set(t: int, idx_row, k: int) -> np.ndarray:
    row = np.ascontiguousarray(idx_row, dtype=np.int32)
    keys = np.empty(4 * k + 4, np.int64)
    n = _load().oracle_key_set(int(t), _ptr(row), k, _ptr(keys))
    if n < 0:
        raise ValueError("idx names a pool the query may not see")
    return keys[:n].copy()


def attn_fwd(Q, K, V, idx, scale: float, rows=None, q_compact: bool = False):
    """O [len(rows), Hq, d] and LSE [len(rows), Hq], fp64.  idx: full [L, k].

    With q_compact, Q holds only the listed rows ([len(rows), Hq, d])."""
    Q, K, V = _f32(Q), _f32(K), _f32(V)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    L = K.shape[0]
    Hq, d = Q.shape[1], Q.shape[2]
    k = idx.shape[1]
    r = _rows(rows, L)
    if q_compact:
        assert Q.shape[0] == r.size
    else:
        assert Q.shape[0] == L
    O = np.empty((r.size, Hq, d), np.float64)
    LSE = np.empty((r.size, Hq), np.float64)
    rc = _load().oracle_attn_fwd(L, Hq, d, float(scale), _ptr(Q), int(q_compact), _ptr(K), _ptr(V), _ptr(idx), k,
                                 _ptr(r), r.size, _ptr(O), _ptr(LSE))
    if rc:
        raise RuntimeError(f"oracle_attn_fwd failed ({rc})")
    return O, LSE


def attn_bwd(Q, K, V, idx, dO, scale: float, rows=None, with_dkv: bool = True, threads: int = 1,
             q_compact: bool = False):
    """dQ [len(rows), Hq, d]; dK, dV [L, d] summed over the listed rows (fp64).

    With threads > 1 the rows are split into `threads` contiguous shards, each
    run by the same single-threaded routine into private dK/dV buffers that
    are then added in shard order.
    """
    Q, K, V, dO = _f32(Q), _f32(K), _f32(V), _f32(dO)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    L = K.shape[0]
    Hq, d = Q.shape[1], Q.shape[2]
    k = idx.shape[1]
    r = _rows(rows, L)
    if q_compact:
        assert Q.shape[0] == r.size and dO.shape[0] == r.size
    lib = _load()
    dQ = np.zeros((r.size, Hq, d), np.float64)
    nshard = max(1, min(int(threads), r.size if r.size else 1))
    bounds = np.linspace(0, r.size, nshard + 1).astype(np.int64)
    dKs = [np.zeros((L, d), np.float64) if with_dkv else None for _ in range(nshard)]
    dVs = [np.zeros((L, d), np.float64) if with_dkv else None for _ in range(nshard)]

    def run(s):
        a, b = int(bounds[s]), int(bounds[s + 1])
        rr = np.ascontiguousarray(r[a:b])
        dq = np.zeros((b - a, Hq, d), np.float64)
        Qs = np.ascontiguousarray(Q[a:b]) if q_compact else Q
        dOs = np.ascontiguousarray(dO[a:b]) if q_compact else dO
        rc = lib.oracle_attn_bwd(L, Hq, d, float(scale), _ptr(Qs), int(q_compact), _ptr(K), _ptr(V), _ptr(idx), k,
                                 _ptr(dOs),
                                 _ptr(rr), rr.size, _ptr(dq),
                                 _ptr(dKs[s]) if with_dkv else None, _ptr(dVs[s]) if with_dkv else None)
        if rc:
            raise RuntimeError(f"oracle_attn_bwd failed ({rc})")
        dQ[a:b] = dq

    if nshard == 1:
        run(0)
    else:
        with ThreadPoolExecutor(nshard) as ex:
            list(ex.map(run, range(nshard)))
    if not with_dkv:
        return dQ, None, None
    dK, dV = dKs[0], dVs[0]
    for s in range(1, nshard):
        dK += dKs[s]
        dV += dVs[s]
    return dQ, dK, dV


def layer_fwd(Q, K, V, q_I, k_I, w, k: int, scale: float, round_to_bf16: bool, rows=None):
    """The whole forward for the listed rows: pool, score, select, attend.

    Returns (kpool, idx [len(rows), k], O, LSE).  Selection rows are computed
    only for the listed rows; attention runs on those rows' selections.
    """
    L = Q.shape[0]
    r = _rows(rows, L)
    kpool = pool_keys(k_I, round_to_bf16)
    s = indexer_scores(q_I, kpool, w, r)
    idx_rows = topk(s, L, k, r)
    idx_full = np.full((L, k), -1, np.int32)
    idx_full[r] = idx_rows
    O, LSE = attn_fwd(Q, K, V, idx_full, scale, r)
    return kpool, idx_rows, O, LSE


def select_rows(q_I, kpool, w, k: int, rows, threads: int = 1, block: int = 128) -> np.ndarray:
    """Top-k selection for the listed rows, scored and selected block by block
    (bounded memory), optionally over several threads.  Pure orchestration of
    indexer_scores and topk."""
    q_I, kpool, w = _f32(q_I), _f32(kpool), _f32(w)
    L = q_I.shape[0]
    r = _rows(rows, L)
    out = np.empty((r.size, k), np.int32)
    starts = list(range(0, r.size, block))

    def run(a):
        rr = r[a:a + block]
        out[a:a + rr.size] = topk(indexer_scores(q_I, kpool, w, rr), L, k, rr)

    if threads <= 1:
        for a in starts:
            run(a)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(run, starts))
    return out


def scores_for(q_I, kpool, w, rows) -> np.ndarray:
    """fp64 indexer scores for the listed rows (alias kept for readability at call sites)."""
    return indexer_scores(q_I, kpool, w, rows)

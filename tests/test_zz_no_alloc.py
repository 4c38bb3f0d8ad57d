"""dsa_layer_fwd_noalloc: the layer forward for callers that cannot allocate.

Some callers cannot hand the library a workspace: a plugin inside a framework
whose caching allocator owns the device memory and whose operator interface
has no workspace argument, or a code path where cudaMalloc (which may
synchronise the device) is not allowed.  dsa_layer_fwd_noalloc keeps the
indexer's score block in one fixed device array inside the library instead.
These tests call it through the C ABI and check that it gives what
dsa_layer_fwd gives, on two calls in a row (the array keeps the previous
call's contents, which must not leak into the next result).

This file is collected last on purpose, so that a stop-at-first-failure run
has already run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import dsa_inputs
import long_context_sparse_dsa_gb300 as dsa

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = {"bf16": 2e-2, "fp32": 1e-4}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_sparse_dsa_gb300 import build
    build.build()
    dsa.library()


def _inputs(wl):
    host = dsa_inputs.make(wl, ("Q", "K", "V", "q_I", "k_I", "w"))
    return {n: t.to(DEV) for n, t in host.items()}


@pytest.mark.parametrize("wl", [
    dsa_inputs.WORKLOADS["bf16_32k"].with_(name="bf16_64k", L=65536),   # 1024-query chunks in the array
    dsa_inputs.WORKLOADS["tiny_fp32_fwd"],
], ids=lambda w: w.name)
def test_noalloc_forward_matches_layer_fwd_twice(wl):
    x = _inputs(wl)
    dims = dsa.make_dims(wl.L, wl.Hq, wl.d, wl.Hi, wl.di, wl.k, q_chunk=wl.q_chunk, scale=wl.scale, dtype=wl.dtype)
    ref = dsa.alloc_forward_buffers(dims, DEV)
    dsa.layer_fwd(dims, x["Q"], x["K"], x["V"], x["q_I"], x["k_I"], x["w"], ref.o, ref.lse, ref.idx, ref.kpool,
                  ref.ws)
    dsa.check_device_error()
    for call in range(2):
        got = dsa.alloc_forward_buffers(dims, DEV)
        got.idx.fill_(-5)
        got.o.fill_(7.0)
        got.lse.fill_(7.0)
        dsa.layer_fwd_noalloc(dims, x["Q"], x["K"], x["V"], x["q_I"], x["k_I"], x["w"], got.o, got.lse, got.idx,
                              got.kpool)
        dsa.check_device_error()
        assert torch.equal(got.idx, ref.idx), call
        assert torch.equal(got.kpool.view(torch.uint8), ref.kpool.view(torch.uint8)), call
        assert float((got.o.float() - ref.o.float()).abs().max()) <= TOL[wl.dtype], call
        assert float((got.lse - ref.lse).abs().max()) <= TOL[wl.dtype], call


def test_noalloc_rejects_rows_larger_than_its_array():
    # one score row of L/4 fp32 values must fit the fixed array; this is checked
    # before any pointer is used, so placeholder pointers are safe here
    lib = dsa.library()
    L = 1 << 27                              # 2^25 pools -> a 128 MiB row
    dims = dsa.make_dims(L, 16, 128, 8, 64, 512, q_chunk=4096)
    p = ctypes.c_void_p(256)
    st = lib.dsa_layer_fwd_noalloc(ctypes.byref(dims), p, p, p, p, p, p, p, p, p, p, None)
    assert st == dsa.DSA_ERR_UNSUPPORTED
    assert b"scratch" in lib.dsa_last_error_message()

"""The end-to-end leg of bench.py does the layer's work: the outputs its
pipelined schedule copies back to pinned host memory equal those of a direct
dsa_layer_fwd + dsa_layer_bwd on the same inputs.

O, LSE and dQ are computed without atomics and must match bit for bit; dK and
dV are sums of fp32 reductions whose order varies between runs, so they are
held to the rounding of those sums."""
import pytest
import torch

import bench
import dsa_inputs
import long_context_sparse_dsa_gb300 as dsa

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_sparse_dsa_gb300 import build
    build.build()
    dsa.library()


@pytest.mark.parametrize("steps", [1, 3])
def test_pipelined_outputs_equal_the_direct_layer(steps):
    wl = dsa_inputs.WORKLOADS["bf16_32k"].with_(name="bf16_e2e_8k", L=8192, q_chunk=3000)
    names = ["Q", "K", "V", "q_I", "k_I", "w", "dO"]
    host = dsa_inputs.make(wl, tuple(names), pin=True)
    d_in = {n: host[n].to(DEV) for n in names}
    dims = dsa.make_dims(wl.L, wl.Hq, wl.d, wl.Hi, wl.di, wl.k, q_chunk=wl.q_chunk, scale=wl.scale, dtype=wl.dtype)
    bufs = dsa.alloc_forward_buffers(dims, DEV, o_acc=True)
    grads = [torch.empty((wl.L, wl.Hq, wl.d), device=DEV), torch.empty((wl.L, wl.d), device=DEV),
             torch.empty((wl.L, wl.d), device=DEV)]
    outs = [bufs.o, bufs.lse] + grads

    # the direct calls
    dsa.layer_fwd(dims, d_in["Q"], d_in["K"], d_in["V"], d_in["q_I"], d_in["k_I"], d_in["w"], bufs.o, bufs.lse,
                  bufs.idx, bufs.kpool, bufs.ws, o_acc=bufs.o_acc)
    dsa.layer_bwd(dims, d_in["Q"], d_in["K"], d_in["V"], bufs.idx, bufs.o, bufs.lse, d_in["dO"], *grads, None,
                  o_acc=bufs.o_acc)
    dsa.check_device_error()
    ref = [t.cpu().clone() for t in outs]
    for t in outs:
        t.fill_(float("nan"))

    phases = bench.layer_phases(dsa, dims, wl, bufs, None, with_bwd=True)
    sink = []
    ms, overlap = bench._e2e_pipelined(host, d_in, outs, phases, steps, DEV, sink=sink)
    dsa.check_device_error()
    got = sink[0]
    assert ms > 0 and overlap["layer_ms_mean"] > 0
    for name, g, r in zip(("O", "LSE", "dQ"), got[:3], ref[:3]):
        assert torch.equal(g, r), name
    for name, g, r in zip(("dK", "dV"), got[3:], ref[3:]):
        assert torch.isfinite(g).all(), name
        assert (g - r).abs().max().item() <= 1e-5 * max(1.0, r.abs().max().item()), name

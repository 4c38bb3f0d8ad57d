"""GPU parity of the whole layer (dsa_layer_fwd / dsa_layer_bwd) against the oracle.

* the tiny fp32 workload (L=4096) in full: selection bit-exact, O/LSE 1e-4;
* a bf16 layer with several indexer chunks, integer indexer inputs: selection
  bit-exact for every row, O on sampled rows and dQ/dK/dV everywhere within 2e-2,
  for the backward with its own D pass and with the forward's fp32 o_acc;
* chunk-size invariance and run-to-run bitwise determinism of the forward;
* the full-size workloads on sampled rows, with near-tie tolerance for the
  selection where scores come from N(0,1) inputs (fp32 scores are not
  bit-reproducible against fp64 there), and closed-form invariants of dV/dK;
* the gradients of the 32k and 128k-needle workloads element by element over
  every row, dK and dV included (the oracle sharded over the host's cores, on
  the GPU's own selection);
* integer twins of the 128k-needle and 256k workloads: the selection bit for
  bit on sampled rows of 32768 and 65536 pools;
* the tcgen05 forward (route 1) at full size against the warp-level forward on
  every row and against the oracle on sampled rows;
* the two indexer + top-k routes against each other over every row at full size;
* the deterministic backward at 256k against itself and the atomic backward.
"""
import math
import os

import numpy as np
import pytest
import torch

import dsa_inputs
import oracle
import long_context_sparse_dsa_gb300 as dsa

pytestmark = pytest.mark.gpu
DEV = "cuda"
NTHREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_sparse_dsa_gb300 import build
    build.build()
    dsa.library()


def _f32(t):
    return t.detach().to("cpu", torch.float32).numpy()


def _run_layer(wl, host, with_bwd, q_chunk=None, o_acc=False):
    """o_acc=True: the forward also writes the fp32 output and the backward takes
    D from it (no workspace, no D pass), as the benchmark runs the layer."""
    dims = dsa.make_dims(wl.L, wl.Hq, wl.d, wl.Hi, wl.di, wl.k, q_chunk=q_chunk or wl.q_chunk, scale=wl.scale,
                         dtype=wl.dtype)
    dev = {n: t.to(DEV) for n, t in host.items()}
    bufs = dsa.alloc_forward_buffers(dims, DEV, o_acc=o_acc)
    dsa.layer_fwd(dims, dev["Q"], dev["K"], dev["V"], dev["q_I"], dev["k_I"], dev["w"], bufs.o, bufs.lse, bufs.idx,
                  bufs.kpool, bufs.ws, o_acc=bufs.o_acc)
    out = {"o": bufs.o, "lse": bufs.lse, "idx": bufs.idx, "kpool": bufs.kpool, "o_acc": bufs.o_acc}
    if with_bwd:
        dq = torch.empty((wl.L, wl.Hq, wl.d), device=DEV)
        dk = torch.empty((wl.L, wl.d), device=DEV)
        dv = torch.empty((wl.L, wl.d), device=DEV)
        ws = None if o_acc else dsa.alloc_backward_workspace(dims, DEV)
        dsa.layer_bwd(dims, dev["Q"], dev["K"], dev["V"], bufs.idx, bufs.o, bufs.lse, dev["dO"], dq, dk, dv, ws,
                      o_acc=bufs.o_acc)
        out.update(dq=dq, dk=dk, dv=dv)
    dsa.check_device_error()
    return out


def test_tiny_fp32_forward_in_full():
    wl = dsa_inputs.WORKLOADS["tiny_fp32_fwd"]
    host = dsa_inputs.make(wl, ("Q", "K", "V", "q_I", "k_I", "w"))
    out = _run_layer(wl, host, with_bwd=False)
    f = {n: _f32(t) for n, t in host.items()}
    kp = oracle.pool_keys(f["k_I"], False)
    assert np.array_equal(_f32(out["kpool"]), kp)
    idx = oracle.select_rows(f["q_I"], kp, f["w"], wl.k, None, threads=NTHREADS)
    assert np.array_equal(out["idx"].cpu().numpy(), idx)
    O, LSE = oracle.attn_fwd(f["Q"], f["K"], f["V"], idx, wl.scale)
    assert np.abs(_f32(out["o"]) - O).max() <= 1e-4
    assert np.abs(out["lse"].cpu().numpy() - LSE).max() <= 1e-4


@pytest.mark.parametrize("L", [4, 8, 12, 16, 132])
@pytest.mark.parametrize("k", [1, 512])
def test_tiny_sequences_fwd_bwd(L, k):
    """Degenerate lengths: a single pool (L=4), score rows narrower than one
    score tile or TMA box, a ragged last pool tile; k above and below the
    number of eligible pools.  Compared in full with the oracle."""
    wl = dsa_inputs.WORKLOADS["bf16_32k"].with_(name=f"bf16_tiny_{L}", L=L, k=k, q_chunk=L, indexer="int3",
                                                  weights="int1_4")
    host = dsa_inputs.make(wl)
    f = {n: _f32(t) for n, t in host.items()}
    kp = oracle.pool_keys(f["k_I"], True)
    idx = oracle.select_rows(f["q_I"], kp, f["w"], k, None, threads=1)
    O, LSE = oracle.attn_fwd(f["Q"], f["K"], f["V"], idx, wl.scale)
    dQ, dK, dV = oracle.attn_bwd(f["Q"], f["K"], f["V"], idx, f["dO"], wl.scale, threads=1)
    out = _run_layer(wl, host, with_bwd=True, o_acc=True)
    assert np.array_equal(_f32(out["kpool"]).view(np.uint32), kp.view(np.uint32))
    assert np.array_equal(out["idx"].cpu().numpy(), idx)
    assert np.abs(_f32(out["o"]) - O).max() <= 2e-2
    assert np.abs(out["o_acc"].cpu().numpy() - O).max() <= 1e-4
    assert np.abs(out["lse"].cpu().numpy() - LSE).max() <= 1e-3
    for n, ref in (("dq", dQ), ("dk", dK), ("dv", dV)):
        assert np.abs(out[n].cpu().numpy() - ref).max() <= 2e-2, n


@pytest.mark.parametrize("L", [4, 8, 132])
def test_tiny_sequences_fp32_forward(L):
    wl = dsa_inputs.WORKLOADS["tiny_fp32_fwd"].with_(name=f"fp32_tiny_{L}", L=L, q_chunk=L)
    host = dsa_inputs.make(wl, ("Q", "K", "V", "q_I", "k_I", "w"))
    f = {n: _f32(t) for n, t in host.items()}
    kp = oracle.pool_keys(f["k_I"], False)
    idx = oracle.select_rows(f["q_I"], kp, f["w"], wl.k, None, threads=1)
    O, LSE = oracle.attn_fwd(f["Q"], f["K"], f["V"], idx, wl.scale)
    out = _run_layer(wl, host, with_bwd=False, o_acc=True)
    assert np.array_equal(out["idx"].cpu().numpy(), idx)
    assert np.abs(_f32(out["o"]) - O).max() <= 1e-4
    assert torch.equal(out["o_acc"], out["o"])
    assert np.abs(out["lse"].cpu().numpy() - LSE).max() <= 1e-4


def _bf16_multichunk():
    return dsa_inputs.WORKLOADS["bf16_32k"].with_(name="bf16_8k_int", L=8192, q_chunk=3000, indexer="int3",
                                                  weights="int1_4")


def test_bf16_layer_fwd_bwd_multichunk_integer_indexer():
    wl = _bf16_multichunk()
    host = dsa_inputs.make(wl)
    f = {n: _f32(t) for n, t in host.items()}
    kp = oracle.pool_keys(f["k_I"], True)
    idx = oracle.select_rows(f["q_I"], kp, f["w"], wl.k, None, threads=NTHREADS)
    rows = dsa_inputs.sample_rows(wl, 192)
    O, LSE = oracle.attn_fwd(f["Q"], f["K"], f["V"], idx, wl.scale, rows)
    dQ, dK, dV = oracle.attn_bwd(f["Q"], f["K"], f["V"], idx, f["dO"], wl.scale, threads=NTHREADS)
    for o_acc in (False, True):
        out = _run_layer(wl, host, with_bwd=True, o_acc=o_acc)
        assert np.array_equal(_f32(out["kpool"]).view(np.uint32), kp.view(np.uint32))
        assert np.array_equal(out["idx"].cpu().numpy(), idx)
        assert np.abs(_f32(out["o"])[rows] - O).max() <= 2e-2
        assert np.abs(out["lse"].cpu().numpy()[rows] - LSE).max() <= 1e-3
        if o_acc:
            assert np.abs(out["o_acc"].cpu().numpy()[rows] - O).max() <= 1e-4
        errs = {n: float(np.abs(out[n].cpu().numpy() - ref).max()) for n, ref in (("dq", dQ), ("dk", dK), ("dv", dV))}
        assert max(errs.values()) <= 2e-2, (o_acc, errs)


def test_forward_is_chunk_invariant_and_deterministic():
    wl = dsa_inputs.WORKLOADS["bf16_32k"].with_(name="bf16_6k", L=6144)
    host = dsa_inputs.make(wl, ("Q", "K", "V", "q_I", "k_I", "w"))
    ref = _run_layer(wl, host, False, q_chunk=wl.L)
    for qc in (wl.L, 1000, 256, 4096 + 13):
        out = _run_layer(wl, host, False, q_chunk=qc)
        for n in ("idx", "o", "lse", "kpool"):
            assert torch.equal(out[n].view(torch.uint8), ref[n].view(torch.uint8)), (qc, n)


def _score_bound(f_qI, kp, f_w, rows, di, Hi):
    absdot = np.einsum("thi,pi->thp", np.abs(f_qI[rows]).astype(np.float64), np.abs(kp).astype(np.float64))
    return 4 * (di + Hi + 2) * 2.0 ** -24 * np.einsum("th,thp->tp", np.abs(f_w[rows]).astype(np.float64), absdot)


def _check_selection(wl, f, kp, got_idx, rows, exact):
    """Compare GPU idx rows with the oracle.  Returns the rows whose sets agree."""
    ref = oracle.select_rows(f["q_I"], kp, f["w"], wl.k, rows, threads=NTHREADS)
    same = np.all(got_idx == ref, axis=1)
    if exact:
        assert same.all(), np.argwhere(~same)[:5]
        return np.asarray(rows), ref
    bad = np.nonzero(~same)[0]
    if bad.size:
        sc = oracle.indexer_scores(f["q_I"], kp, f["w"], np.asarray(rows)[bad])
        bnd = _score_bound(f["q_I"], kp, f["w"], np.asarray(rows)[bad], wl.di, wl.Hi)
        for j, r in enumerate(bad):
            g_set, o_set = set(got_idx[r][got_idx[r] >= 0]), set(ref[r][ref[r] >= 0])
            assert len(g_set) == len(o_set)
            kth = np.min(sc[j][list(o_set)])
            for p in g_set ^ o_set:                 # every disagreement is a near-tie at the threshold
                assert abs(sc[j][p] - kth) <= bnd[j][p] + bnd[j].max(), (rows[r], p)
    assert bad.size <= max(2, len(rows) // 50)
    return np.asarray(rows)[same], ref[same]


@pytest.mark.parametrize("name", ["bf16_32k", "bf16_128k_needle", "bf16_256k", "bf16_1m_ties"])
def test_full_size_workload_sampled(name):
    wl = dsa_inputs.WORKLOADS[name]
    with_bwd = wl.passes == "fwd+bwd"
    host = dsa_inputs.make(wl, ("Q", "K", "V", "q_I", "k_I", "w") + (("dO",) if with_bwd else ()))
    out = _run_layer(wl, host, with_bwd, o_acc=with_bwd)
    rows = np.asarray(dsa_inputs.sample_rows(wl, 96))
    f = {n: _f32(host[n]) for n in ("K", "V", "q_I", "k_I", "w")}
    kp = oracle.pool_keys(f["k_I"], True)
    assert np.array_equal(_f32(out["kpool"]).view(np.uint32), kp.view(np.uint32))
    got_idx = out["idx"].cpu().numpy()[rows]
    agree, ref_idx = _check_selection(wl, f, kp, got_idx, rows, exact=wl.indexer != "normal")
    # attention on the rows whose selection agrees, with the oracle's own idx
    idx_full = np.full((wl.L, wl.k), -1, np.int32)
    idx_full[agree] = ref_idx
    Qr = _f32(host["Q"][agree])
    O, LSE = oracle.attn_fwd(Qr, f["K"], f["V"], idx_full, wl.scale, agree, q_compact=True)
    assert np.abs(_f32(out["o"][agree]) - O).max() <= 2e-2
    assert np.abs(out["lse"][agree].cpu().numpy() - LSE).max() <= 1e-3
    if with_bwd:
        assert np.abs(out["o_acc"][agree].cpu().numpy() - O).max() <= 1e-4
        dOr = _f32(host["dO"][agree])
        dQ, _, _ = oracle.attn_bwd(Qr, f["K"], f["V"], idx_full, dOr, wl.scale, agree, with_dkv=False,
                                   threads=NTHREADS, q_compact=True)
        assert np.abs(out["dq"][agree].cpu().numpy() - dQ).max() <= 2e-2
        # closed forms valid at any size: sum_j dV[j] = sum_{t,h} dO[t,h] (softmax rows sum to 1) and
        # sum_j dK[j] = 0 (sum_j dS = dO.O - D = 0), up to rounding
        dv_sum = out["dv"].double().sum(0).cpu().numpy()
        do_sum = host["dO"].to(torch.float64).sum((0, 1)).numpy()
        assert np.abs(dv_sum - do_sum).max() <= 1e-5 * wl.L * wl.Hq ** 0.5
        dk_sum = out["dk"].double().sum(0).cpu().numpy()
        assert np.abs(dk_sum).max() <= 2e-3 * math.sqrt(wl.L * wl.Hq)


@pytest.mark.parametrize("name", ["bf16_32k", "bf16_128k_needle"])
def test_full_size_gradients_elementwise(name, record_property):
    """dQ, dK and dV of a full-size workload compared element by element with
    the oracle over all rows.  The oracle runs on the GPU's selection (so
    near-tie selection differences cannot leak into the gradients), sharded
    over the host's cores into private fp64 dK/dV that are summed in shard
    order.  The keys selected by the most queries -- with the needle, a few
    needle keys collect contributions from a large share of the sequence --
    are where fp32 accumulation error would concentrate; their error is
    recorded."""
    wl = dsa_inputs.WORKLOADS[name]
    host = dsa_inputs.make(wl)
    out = _run_layer(wl, host, with_bwd=True, o_acc=True)
    idx = out["idx"].cpu().numpy()
    f = {n: _f32(host[n]) for n in ("Q", "K", "V", "dO")}
    threads = max(1, os.cpu_count() or 1)
    dQ, dK, dV = oracle.attn_bwd(f["Q"], f["K"], f["V"], idx, f["dO"], wl.scale, threads=threads)
    del f
    gq = out["dq"].cpu().numpy()
    eq = float(np.abs(gq - dQ).max())
    del gq, dQ
    # the deterministic backward on the same forward: the same bits twice, and
    # the same oracle bound
    dims = dsa.make_dims(wl.L, wl.Hq, wl.d, wl.Hi, wl.di, wl.k, q_chunk=wl.q_chunk, scale=wl.scale, dtype=wl.dtype)
    dev = {n: host[n].to(DEV) for n in ("Q", "K", "V", "dO")}
    ws = dsa.alloc_bwd_det_workspace(dims, DEV)
    det = []
    for _ in range(2):
        g = [torch.empty_like(out["dq"]), torch.empty_like(out["dk"]), torch.empty_like(out["dv"])]
        dsa.sparse_attn_bwd_det(dims, dev["Q"], dev["K"], dev["V"], out["idx"], out["o"], out["lse"], dev["dO"], *g,
                                ws, o_acc=out["o_acc"])
        det.append(g)
    dsa.check_device_error()
    for a, b in zip(det[0], det[1]):
        assert torch.equal(a, b)
    assert torch.equal(det[0][0], out["dq"])
    del dev, ws
    gk, gv = out["dk"].cpu().numpy(), out["dv"].cpu().numpy()
    errk, errv = np.abs(gk - dK), np.abs(gv - dV)
    dk_det, dv_det = det[0][1].cpu().numpy(), det[0][2].cpu().numpy()
    err_det = max(float(np.abs(dk_det - dK).max()), float(np.abs(dv_det - dV).max()))
    del det
    counts = np.bincount(idx[idx >= 0].ravel(), minlength=wl.P)
    top = int(np.argmax(counts))
    keys = slice(4 * top, 4 * top + 4)
    rec = {"max_err_dq": eq, "max_err_dk": float(errk.max()), "max_err_dv": float(errv.max()),
           "most_selected_pool": top, "its_queries": int(counts[top]),
           "its_err_dk": float(errk[keys].max()), "its_err_dv": float(errv[keys].max()),
           "its_max_abs_dv": float(np.abs(dV[keys]).max()), "max_err_dkdv_deterministic": err_det}
    record_property("gradient_errors", rec)
    print(name, rec)
    assert eq <= 2e-2, rec
    assert errk.max() <= 2e-2 and errv.max() <= 2e-2, rec
    assert err_det <= 2e-2, rec


@pytest.mark.parametrize("name", ["bf16_128k_needle", "bf16_256k"])
def test_full_size_integer_twin_selection_bitexact(name):
    """The integer-input twin of a full-size workload (same shapes; indexer
    inputs and weights small integers, so every fp32 score is exact): the
    selection of sampled rows with 32768 (128k) or 65536 (256k) pools is
    compared bit for bit with the oracle, including every indexer-chunk
    boundary +-1 and the last rows."""
    wl = dsa_inputs.WORKLOADS[name].integer_twin()
    host = dsa_inputs.make(wl, ("Q", "K", "V", "q_I", "k_I", "w"))
    out = _run_layer(wl, host, with_bwd=False)
    f = {n: _f32(host[n]) for n in ("q_I", "k_I", "w")}
    kp = oracle.pool_keys(f["k_I"], True)
    assert np.array_equal(_f32(out["kpool"]).view(np.uint32), kp.view(np.uint32))
    rows = np.asarray(dsa_inputs.sample_rows(wl, 512))
    got = out["idx"].cpu().numpy()[rows]
    ref = oracle.select_rows(f["q_I"], kp, f["w"], wl.k, rows, threads=NTHREADS, block=32)
    bad = np.nonzero(~np.all(got == ref, axis=1))[0]
    assert bad.size == 0, rows[bad[:5]]


@pytest.mark.parametrize("name", ["bf16_128k_needle", "bf16_256k"])
def test_full_size_tcgen05_forward(name):
    """The tcgen05 forward (route 1) at full size, on the layer's own selection:
    every row against the warp-level forward (route 0) -- O within 2e-2, LSE
    within 1e-4, o_acc within 1e-4 -- and sampled rows (early padded rows,
    needle rows and a spread of the rest) against the oracle."""
    wl = dsa_inputs.WORKLOADS[name]
    host = dsa_inputs.make(wl, ("Q", "K", "V", "q_I", "k_I", "w"))
    dims = dsa.make_dims(wl.L, wl.Hq, wl.d, wl.Hi, wl.di, wl.k, q_chunk=wl.q_chunk, scale=wl.scale, dtype=wl.dtype)
    dev = {n: t.to(DEV) for n, t in host.items()}
    bufs = dsa.alloc_forward_buffers(dims, DEV, o_acc=True)
    outs = {}
    try:
        for route in (0, 1):
            dsa.set_attn_fwd_route(route)
            if route == 0:
                dsa.layer_fwd(dims, dev["Q"], dev["K"], dev["V"], dev["q_I"], dev["k_I"], dev["w"], bufs.o, bufs.lse,
                              bufs.idx, bufs.kpool, bufs.ws, o_acc=bufs.o_acc)
                outs[0] = (bufs.o, bufs.lse, bufs.o_acc)
            else:
                o, lse, acc = torch.empty_like(bufs.o), torch.empty_like(bufs.lse), torch.empty_like(bufs.o_acc)
                dsa.sparse_attn_fwd(dims, dev["Q"], dev["K"], dev["V"], bufs.idx, o, lse, o_acc=acc)
                outs[1] = (o, lse, acc)
            dsa.check_device_error()
    finally:
        dsa.set_attn_fwd_route(0)
    (o0, l0, a0), (o1, l1, a1) = outs[0], outs[1]
    assert (o1.float() - o0.float()).abs().max().item() <= 2e-2
    assert (l1 - l0).abs().max().item() <= 1e-4
    assert (a1 - a0).abs().max().item() <= 1e-4
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([np.arange(0, 12), rng.integers(12, wl.L, 48), [wl.L - 1]]))
    idx = bufs.idx.cpu().numpy()
    Qr = _f32(host["Q"][torch.from_numpy(rows)])   # only the sampled rows of Q
    O, LSE = oracle.attn_fwd(Qr, _f32(host["K"]), _f32(host["V"]), idx, wl.scale, rows=rows, q_compact=True)
    assert np.abs(_f32(o1)[rows] - O).max() <= 2e-2
    assert np.abs(a1.cpu().numpy()[rows] - O).max() <= 1e-4
    assert np.abs(l1.cpu().numpy()[rows] - LSE).max() <= 1e-3


@pytest.mark.parametrize("name", ["bf16_128k_needle", "bf16_1m_ties"])
def test_full_size_indexer_routes_agree(name):
    """The two indexer + top-k routes of dsa_indexer_topk select the same pools
    bit for bit over every row of a full-size workload: route 1 (the score
    block and the row-wise top-k, checked against the oracle on sampled rows
    above) and route 0 (candidate lists, no score block).  At 1M the integer
    indexer inputs make thousands of exact ties per row, which overflow route
    0's candidate lists and send rows through its fallback."""
    wl = dsa_inputs.WORKLOADS[name]
    host = dsa_inputs.make(wl, ("q_I", "k_I", "w"))
    dims = dsa.make_dims(wl.L, wl.Hq, wl.d, wl.Hi, wl.di, wl.k, q_chunk=wl.q_chunk, scale=wl.scale, dtype=wl.dtype)
    dev = {n: t.to(DEV) for n, t in host.items()}
    kpool = torch.empty((wl.L // 4, wl.di), dtype=dev["k_I"].dtype, device=DEV)
    dsa.pool_keys(dims, dev["k_I"], kpool)
    ws = torch.empty(dsa.indexer_topk_workspace_bytes(dims, wl.q_chunk), dtype=torch.uint8, device=DEV)
    out = {}
    try:
        for route in (1, 0):
            dsa.set_indexer_topk_route(route)
            idx = torch.full((wl.L, wl.k), -7, dtype=torch.int32, device=DEV)
            for q0 in range(0, wl.L, wl.q_chunk):
                n = min(wl.q_chunk, wl.L - q0)
                dsa.indexer_topk(dims, dev["q_I"], kpool, dev["w"], q0, n, idx, ws)
            dsa.check_device_error()
            out[route] = idx
    finally:
        dsa.set_indexer_topk_route(1)
    same = (out[0] == out[1]).all(dim=1)
    assert bool(same.all()), torch.nonzero(~same)[:5].flatten().tolist()
    assert int((out[1] == -7).sum()) == 0


def test_full_size_deterministic_backward_256k():
    """The deterministic backward at the 256k workload (Hq = 32: two head
    groups per query) on the layer's own forward: two runs give the same bits,
    its dQ is bit-identical to the atomic backward's (the same query-major
    arithmetic), and its dK/dV agree with the atomic backward's (which the
    closed forms above hold at this size) within 2e-2 everywhere."""
    wl = dsa_inputs.WORKLOADS["bf16_256k"]
    host = dsa_inputs.make(wl)
    out = _run_layer(wl, host, with_bwd=True, o_acc=True)
    dims = dsa.make_dims(wl.L, wl.Hq, wl.d, wl.Hi, wl.di, wl.k, q_chunk=wl.q_chunk, scale=wl.scale, dtype=wl.dtype)
    dev = {n: host[n].to(DEV) for n in ("Q", "K", "V", "dO")}
    ws = dsa.alloc_bwd_det_workspace(dims, DEV)
    det = []
    for _ in range(2):
        g = [torch.empty_like(out["dq"]), torch.empty_like(out["dk"]), torch.empty_like(out["dv"])]
        dsa.sparse_attn_bwd_det(dims, dev["Q"], dev["K"], dev["V"], out["idx"], out["o"], out["lse"], dev["dO"], *g,
                                ws, o_acc=out["o_acc"])
        det.append(g)
    dsa.check_device_error()
    for a, b in zip(det[0], det[1]):
        assert torch.equal(a, b)
    assert torch.equal(det[0][0], out["dq"])
    ek = (det[0][1] - out["dk"]).abs().max().item()
    ev = (det[0][2] - out["dv"]).abs().max().item()
    assert ek <= 2e-2 and ev <= 2e-2, (ek, ev)

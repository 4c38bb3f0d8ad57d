"""GPU parity of each kernel against the CPU oracle (through the C ABI).

Sizes span several tiles and a ragged tail: pool counts that are not a
multiple of the 128-pool MMA tile, query ranges that start and end off the
32-query block, score rows on both sides of the top-k shared-memory staging
limit, keys sets below k.  Integer-valued indexer inputs make every fp32 score
exact, so pool keys, scores and top-k are compared bit for bit; attention is
compared by max-abs error against the fp64 oracle (2e-2 bf16, 1e-4 fp32).
"""
import math

import numpy as np
import pytest
import torch

import dsa_inputs
import oracle
import long_context_sparse_dsa_gb300 as dsa

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = {"bf16": 2e-2, "fp32": 1e-4}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_sparse_dsa_gb300 import build
    build.build()
    dsa.library()


def _tdt(dtype):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def _f32(t):
    return t.detach().to("cpu", torch.float32).numpy()


def _int_inputs(g, L, Hi, di, dtype):
    q = torch.randint(-3, 4, (L, Hi, di), generator=g).to(_tdt(dtype))
    k = torch.randint(-3, 4, (L, di), generator=g).to(_tdt(dtype))
    w = torch.randint(1, 5, (L, Hi), generator=g).to(torch.float32)
    return q, k, w


def _sentinel(shape):
    return torch.full(shape, 0x7fc0dead, dtype=torch.int32, device=DEV).view(torch.float32)


# ---------------------------------------------------------------- selftest
def test_bounded_wait_gives_up_and_stream_survives():
    dsa.check_device_error()
    dsa.selftest_bounded_wait(2000)
    with pytest.raises(dsa.DSAError) as e:
        dsa.check_device_error()
    assert e.value.status == dsa.DSA_ERR_TIMEOUT
    x = torch.arange(16, device=DEV, dtype=torch.float32)
    assert float((x * 2).sum()) == 240.0
    dsa.check_device_error()


# ---------------------------------------------------------------- traffic probe
@pytest.mark.parametrize("Hq,d", [(16, 64), (32, 128)])
def test_probe_traffic_does_its_reductions(Hq, d):
    """The traffic replay behind the attention kernels' roofline does the work
    it claims: every (query, 16-head group) adds each of its attended keys'
    rows (d values) once into dK and once into dV, so their sums grow by
    exactly the attended-key count x head groups x d times the added value,
    and only attended rows are touched."""
    L, k = 3000, 32
    Q, K, V, _, idx = _attn_case(L, Hq, d, k, "bf16", seed=41)
    dims = dsa.make_dims(L, Hq, d, 8, 64, k)
    kd, vd, idx_d = K.to(DEV), V.to(DEV), torch.from_numpy(idx).to(DEV)
    dk = torch.zeros(L, d, device=DEV)
    dv = torch.zeros(L, d, device=DEV)
    dsa.probe_traffic(dims, kd, vd, idx_d)
    dsa.probe_traffic(dims, kd, vd, idx_d, dk, dv)
    dsa.check_device_error()
    hits = np.zeros(L, np.int64)
    for t in range(L):
        keys = oracle.key_set(t, idx[t], k)
        np.add.at(hits, keys, 1)
    want = float(hits.sum()) * (Hq // 16) * d * 1e-30
    for tns in (dk, dv):
        got = float(tns.double().sum())
        assert abs(got - want) <= 1e-3 * want, (got, want)
        touched = (tns != 0).any(1).cpu().numpy()
        assert np.array_equal(touched, hits > 0)


# ---------------------------------------------------------------- pool keys
@pytest.mark.parametrize("dtype,di", [("bf16", 64), ("bf16", 128), ("fp32", 64), ("fp32", 128)])
def test_pool_keys_bitexact(dtype, di):
    g = torch.Generator().manual_seed(1)
    L = 4 * 1331
    k_I = (torch.randn(L, di, generator=g) * 3).to(_tdt(dtype))
    dims = dsa.make_dims(L, 16 if dtype == "bf16" else 8, 128, 8, di, 8, dtype=dtype)
    kp = torch.empty((L // 4, di), dtype=_tdt(dtype), device=DEV)
    dsa.pool_keys(dims, k_I.to(DEV), kp)
    ref = oracle.pool_keys(_f32(k_I), dtype == "bf16")
    assert np.array_equal(_f32(kp).view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("dtype,di", [("bf16", 64), ("bf16", 128), ("fp32", 64), ("fp32", 128)])
def test_pool_keys_gated_bitexact(dtype, di):
    """Gated pooling against the oracle bit for bit (N(0,1)-scale keys, gates
    of both signs and assorted magnitudes), and all-one gates against the plain
    pool."""
    g = torch.Generator().manual_seed(31)
    L = 4 * 1331
    k_I = (torch.randn(L, di, generator=g) * 3).to(_tdt(dtype))
    gate = torch.randn(L, generator=g) * torch.exp2(torch.randint(-6, 7, (L,), generator=g).float())
    dims = dsa.make_dims(L, 16 if dtype == "bf16" else 8, 128, 8, di, 8, dtype=dtype)
    kp = torch.empty((L // 4, di), dtype=_tdt(dtype), device=DEV)
    dsa.pool_keys_gated(dims, k_I.to(DEV), gate.to(DEV), kp)
    ref = oracle.pool_keys_gated(_f32(k_I), gate.numpy(), dtype == "bf16")
    assert np.array_equal(_f32(kp).view(np.uint32), ref.view(np.uint32))
    ones = torch.ones(L, device=DEV)
    kp1, kp0 = torch.empty_like(kp), torch.empty_like(kp)
    dsa.pool_keys_gated(dims, k_I.to(DEV), ones, kp1)
    dsa.pool_keys(dims, k_I.to(DEV), kp0)
    dsa.check_device_error()
    assert torch.equal(kp1.view(torch.uint8), kp0.view(torch.uint8))


@pytest.mark.parametrize("name", ["bf16_128k_needle", "bf16_1m_ties"])
def test_pool_keys_full_size_bitexact(name):
    """Plain and gated pool keys of a full-size workload's own k_I, every pool,
    against the oracle bit for bit (gates of both signs, zeros and assorted
    magnitudes)."""
    wl = dsa_inputs.WORKLOADS[name]
    k_I = dsa_inputs.make(wl, ("k_I",))["k_I"]
    g = torch.Generator().manual_seed(33)
    gate = torch.randn(wl.L, generator=g) * torch.exp2(torch.randint(-6, 7, (wl.L,), generator=g).float())
    gate[::17] = 0.0
    dims = dsa.make_dims(wl.L, wl.Hq, wl.d, wl.Hi, wl.di, wl.k, q_chunk=wl.q_chunk, dtype=wl.dtype)
    kp = torch.empty((wl.L // 4, wl.di), dtype=torch.bfloat16, device=DEV)
    kg = torch.empty_like(kp)
    kd = k_I.to(DEV)
    dsa.pool_keys(dims, kd, kp)
    dsa.pool_keys_gated(dims, kd, gate.to(DEV), kg)
    dsa.check_device_error()
    kf = _f32(k_I)
    assert np.array_equal(_f32(kp).view(np.uint32), oracle.pool_keys(kf, True).view(np.uint32))
    assert np.array_equal(_f32(kg).view(np.uint32), oracle.pool_keys_gated(kf, gate.numpy(), True).view(np.uint32))


def test_gated_pools_feed_the_selection_bitexact():
    """The gated pool keys through the indexer and top-k (dsa_indexer_topk, both
    routes): with integer keys and gates every score is an exact integer, so the
    selection equals the oracle's bit for bit."""
    g = torch.Generator().manual_seed(32)
    L, Hi, di, k = 4096, 8, 64, 64
    q_I, k_I, w = _int_inputs(g, L, Hi, di, "bf16")
    gate = torch.randint(-1, 3, (L,), generator=g).float()
    dims = dsa.make_dims(L, 16, 128, Hi, di, k, q_chunk=1500, dtype="bf16")
    kp = torch.empty((L // 4, di), dtype=torch.bfloat16, device=DEV)
    dsa.pool_keys_gated(dims, k_I.to(DEV), gate.to(DEV), kp)
    kp_ref = oracle.pool_keys_gated(_f32(k_I), gate.numpy(), True)
    assert np.array_equal(_f32(kp).view(np.uint32), kp_ref.view(np.uint32))
    idx_ref = oracle.topk(oracle.indexer_scores(_f32(q_I), kp_ref, _f32(w)), L, k)
    ws = torch.empty(dsa.workspace_bytes(dims), dtype=torch.uint8, device=DEV)
    try:
        for route in (1, 0):
            dsa.set_indexer_topk_route(route)
            idx = torch.full((L, k), -7, dtype=torch.int32, device=DEV)
            for q0 in range(0, L, 1500):
                dsa.indexer_topk(dims, q_I.to(DEV), kp, w.to(DEV), q0, min(1500, L - q0), idx, ws)
            dsa.check_device_error()
            assert np.array_equal(idx.cpu().numpy(), idx_ref), route
    finally:
        dsa.set_indexer_topk_route(1)


# ---------------------------------------------------------------- indexer
@pytest.mark.parametrize("dtype,Hi,di", [("bf16", 8, 64), ("bf16", 8, 128), ("bf16", 4, 64), ("bf16", 4, 128),
                                         ("fp32", 4, 64), ("fp32", 3, 128)])
@pytest.mark.parametrize("q_begin,q_count", [(0, None), (37, 701)])
def test_indexer_integer_inputs_bitexact(dtype, Hi, di, q_begin, q_count):
    g = torch.Generator().manual_seed(2)
    L = 4 * 330 + 4 * 200   # P = 530: four full 128-pool tiles and a ragged one
    q_count = L - q_begin if q_count is None else q_count
    q_I, k_I, w = _int_inputs(g, L, Hi, di, dtype)
    dims = dsa.make_dims(L, 16 if dtype == "bf16" else 8, 128, Hi, di, 16, dtype=dtype)
    P = L // 4
    kp = torch.empty((P, di), dtype=_tdt(dtype), device=DEV)
    dsa.pool_keys(dims, k_I.to(DEV), kp)
    sc = _sentinel((q_count, P))
    dsa.indexer_score(dims, q_I.to(DEV), kp, w.to(DEV), q_begin, q_count, sc)
    dsa.check_device_error()
    rows = np.arange(q_begin, q_begin + q_count)
    ref = oracle.indexer_scores(_f32(q_I), oracle.pool_keys(_f32(k_I), dtype == "bf16"), _f32(w), rows)
    got = sc.cpu().numpy()
    e = (rows + 1) // 4
    mask = np.arange(P)[None, :] < e[:, None]
    assert np.array_equal(got[mask].astype(np.float64), ref[mask])
    # beyond the causal prefix only the diagonal 128-pool tile of a 32-query block may be written
    blk_end = np.minimum(((rows - q_begin) // 32) * 32 + 31 + q_begin, q_begin + q_count - 1)
    reach = ((blk_end + 1) // 4 + 127) // 128 * 128
    far = np.arange(P)[None, :] >= reach[:, None]
    assert np.all(got.view(np.uint32)[far] == 0x7fc0dead)


def test_indexer_normal_inputs_within_fp32_bound():
    g = torch.Generator().manual_seed(3)
    L, Hi, di = 4096, 8, 64
    q_I = torch.randn(L, Hi, di, generator=g).to(torch.bfloat16)
    k_I = torch.randn(L, di, generator=g).to(torch.bfloat16)
    w = torch.rand(L, Hi, generator=g)
    dims = dsa.make_dims(L, 16, 128, Hi, di, 512)
    kp = torch.empty((L // 4, di), dtype=torch.bfloat16, device=DEV)
    dsa.pool_keys(dims, k_I.to(DEV), kp)
    sc = torch.zeros((L, L // 4), device=DEV)
    dsa.indexer_score(dims, q_I.to(DEV), kp, w.to(DEV), 0, L, sc)
    rows = np.arange(0, L, 7)
    kpn = oracle.pool_keys(_f32(k_I), True)
    ref = oracle.indexer_scores(_f32(q_I), kpn, _f32(w), rows)
    # |error| <= (di + Hi + 2) u sum_h |w| sum_i |q_i kp_i|, u = 2^-24 (products of bf16 are exact in fp32)
    absdot = np.einsum("thi,pi->thp", np.abs(_f32(q_I)[rows]).astype(np.float64), np.abs(kpn).astype(np.float64))
    bound = (di + Hi + 2) * 2.0 ** -24 * np.einsum("th,thp->tp", np.abs(_f32(w)[rows]), absdot)
    got = sc.cpu().numpy()[rows].astype(np.float64)
    e = (rows + 1) // 4
    mask = np.arange(L // 4)[None, :] < e[:, None]
    err = np.abs(got - ref)
    assert np.all(err[mask] <= 4 * bound[mask] + 1e-30), float((err[mask] / (bound[mask] + 1e-30)).max())


# ---------------------------------------------------------------- top-k
def _topk_case(P, rows, k, kind, seed):
    g = torch.Generator().manual_seed(seed)
    n = len(rows)
    if kind == "ties":
        s = torch.randint(-3, 4, (n, P), generator=g).to(torch.float32)
    elif kind == "ties_spikes":
        # integer scores plus a few larger ones per row: the k-th score has
        # thousands of ties and some scores lie above it
        s = torch.randint(-3, 4, (n, P), generator=g).to(torch.float32)
        pos = torch.randint(0, P, (n, 40), generator=g)
        s.scatter_(1, pos, 10.0)
    elif kind == "signed_zero":
        s = torch.randint(-1, 2, (n, P), generator=g).to(torch.float32) * 0.0   # +0 and -0 only
        s[:, ::17] = -1.5
    else:
        s = torch.randn(n, P, generator=g) * 10
    return s


@pytest.mark.parametrize("kind", ["normal", "ties", "ties_spikes", "signed_zero"])
@pytest.mark.parametrize("k", [64, 512, 1024])
def test_topk_bitexact(kind, k):
    # rows of fewer than k pools (all kept), of up to 4096 pools (every score a
    # candidate) and of up to 14000 pools (sampled threshold); k = 1024 is the
    # largest k the library accepts
    L = 4 * 14000
    P = L // 4
    dims = dsa.make_dims(L, 16, 128, 8, 64, k)
    for (q_begin, q_count) in ((0, 300), (2000, 97), (L - 40, 40), (4 * 12288 - 20, 40)):
        rows = np.arange(q_begin, q_begin + q_count)
        s = _topk_case(P, rows, k, kind, seed=q_begin + k)
        idx = torch.full((L, k), -7, dtype=torch.int32, device=DEV)
        dsa.topk(dims, s.to(DEV), q_begin, q_count, idx)
        got = idx.cpu().numpy()[rows]
        sn = s.numpy().astype(np.float64)
        e = (rows + 1) // 4
        sn[np.arange(P)[None, :] >= e[:, None]] = np.nan
        ref = oracle.topk(sn, L, k, rows)
        assert np.array_equal(got, ref), (q_begin, np.argwhere(got != ref)[:5])
        untouched = np.setdiff1d(np.arange(L), rows)[:50]
        assert np.all(idx.cpu().numpy()[untouched] == -7)


# ---------------------------------------------------------------- fused indexer + top-k
def _fused_vs_unfused(L, Hi, di, k, q_I, k_I, w, q_begin, q_count):
    """idx rows from dsa_indexer_topk and from dsa_indexer_score + dsa_topk."""
    dims = dsa.make_dims(L, 16, 128, Hi, di, k, q_chunk=q_count)
    kp = torch.empty((L // 4, di), dtype=torch.bfloat16, device=DEV)
    qd, wd = q_I.to(DEV), w.to(DEV)
    dsa.pool_keys(dims, k_I.to(DEV), kp)
    sc = torch.empty((q_count, L // 4), device=DEV)
    ref = torch.full((L, k), -7, dtype=torch.int32, device=DEV)
    dsa.indexer_score(dims, qd, kp, wd, q_begin, q_count, sc)
    dsa.topk(dims, sc, q_begin, q_count, ref)
    ws = torch.empty(dsa.indexer_topk_workspace_bytes(dims, q_count), dtype=torch.uint8, device=DEV)
    ws.fill_(0xA5)                                  # nothing in the workspace may need to start at zero
    outs = []
    try:
        for route in (0, 1):                        # candidate lists; score block + sampled thresholds
            dsa.set_indexer_topk_route(route)
            for _ in range(2):                      # the second call runs on a used workspace
                got = torch.full((L, k), -7, dtype=torch.int32, device=DEV)
                dsa.indexer_topk(dims, qd, kp, wd, q_begin, q_count, got, ws)
                outs.append(got)
    finally:
        dsa.set_indexer_topk_route(1)
    dsa.check_device_error()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    return outs[0].cpu().numpy(), ref.cpu().numpy(), kp


@pytest.mark.parametrize("inputs", ["normal", "int"])
@pytest.mark.parametrize("Hi,di,k", [(8, 64, 512), (4, 128, 64), (8, 128, 1024), (4, 64, 1)])
def test_indexer_topk_equals_unfused(inputs, Hi, di, k):
    """The fused indexer + top-k gives the unfused pair's idx bit for bit:
    rows of every kind (elig <= k, kept whole, thresholded), a range that
    starts and ends off the 32-query block, rows outside it untouched; with
    integer inputs also the oracle's selection."""
    g = torch.Generator().manual_seed(7 + Hi + di + k)
    L = 4 * 9000 + 4 * 77
    if inputs == "int":
        q_I, k_I, w = _int_inputs(g, L, Hi, di, "bf16")
    else:
        q_I = torch.randn(L, Hi, di, generator=g).to(torch.bfloat16)
        k_I = torch.randn(L, di, generator=g).to(torch.bfloat16)
        w = torch.rand(L, Hi, generator=g)
    for q_begin, q_count in ((0, 3000), (L - 5037, 5037)):
        got, ref, kp = _fused_vs_unfused(L, Hi, di, k, q_I, k_I, w, q_begin, q_count)
        assert np.array_equal(got, ref), (q_begin, np.argwhere(got != ref)[:5])
        rows = np.arange(q_begin, q_begin + q_count)
        outside = np.setdiff1d(np.arange(L), rows)
        assert np.all(got[outside] == -7)
        if inputs == "int":
            sample = rows[:: max(1, q_count // 200)]
            orc = oracle.topk(oracle.indexer_scores(_f32(q_I), _f32(kp), _f32(w), sample), L, k, sample)
            assert np.array_equal(got[sample], orc)


@pytest.mark.parametrize("case", ["all_tied", "threshold_misses"])
def test_indexer_topk_fallback_rows(case):
    """Rows the candidate lists cannot settle go through the score rows and
    the row-wise top-k, with the same result.  all_tied: every score is 0, so
    every eligible pool is a candidate and long rows overflow their lists
    (the answer is pools 0..k-1).  threshold_misses: the sampled pools (every
    32nd) score far above the rest, so the sampled threshold lets fewer than
    k candidates through."""
    L, Hi, di, k = 4 * 12000, 8, 64, 512
    g = torch.Generator().manual_seed(99)
    if case == "all_tied":
        q_I = torch.zeros(L, Hi, di).to(torch.bfloat16)
        k_I = torch.randint(-3, 4, (L, di), generator=g).to(torch.bfloat16)
        w = torch.ones(L, Hi)
    else:
        q_I = torch.randint(1, 3, (L, Hi, di), generator=g).to(torch.bfloat16)
        k_I = torch.randint(0, 2, (L, di), generator=g).to(torch.float32)
        pool_of = torch.arange(L) // 4
        k_I[(pool_of % 32) == 0] += 3.0
        k_I = k_I.to(torch.bfloat16)
        w = torch.randint(1, 5, (L, Hi), generator=g).to(torch.float32)
    q_begin, q_count = L - 4096, 4096
    got, ref, kp = _fused_vs_unfused(L, Hi, di, k, q_I, k_I, w, q_begin, q_count)
    assert np.array_equal(got, ref)
    rows = np.arange(q_begin, q_begin + q_count)[::97]
    orc = oracle.topk(oracle.indexer_scores(_f32(q_I), _f32(kp), _f32(w), rows), L, k, rows)
    assert np.array_equal(got[rows], orc)
    if case == "all_tied":
        assert np.array_equal(got[rows], np.tile(np.arange(k, dtype=np.int32), (rows.size, 1)))


# ---------------------------------------------------------------- attention
def _attn_case(L, Hq, d, k, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    dt = _tdt(dtype)
    Q = torch.randn(L, Hq, d, generator=g).to(dt)
    K = torch.randn(L, d, generator=g).to(dt)
    V = torch.randn(L, d, generator=g).to(dt)
    dO = torch.randn(L, Hq, d, generator=g).to(dt)
    q_I, k_I, w = _int_inputs(g, L, 2, 16, "fp32")
    idx = oracle.topk(oracle.indexer_scores(_f32(q_I), oracle.pool_keys(_f32(k_I), False), _f32(w)), L, k)
    return Q, K, V, dO, idx


@pytest.fixture(params=[1, 0], ids=["tcgen05", "warp"])
def fwd_route(request):
    """Run the test under each bf16 forward kernel (d = 64 always takes the
    warp-level one); the library default (0) is restored afterwards."""
    dsa.set_attn_fwd_route(request.param)
    yield request.param
    dsa.set_attn_fwd_route(0)


@pytest.mark.parametrize("dtype,Hq,d", [("bf16", 16, 128), ("bf16", 32, 128), ("bf16", 16, 64), ("fp32", 8, 64),
                                        ("fp32", 5, 128)])
@pytest.mark.parametrize("k", [1, 5, 32])
def test_attn_fwd_matches_oracle(dtype, Hq, d, k, fwd_route):
    L = 1000
    Q, K, V, _, idx = _attn_case(L, Hq, d, k, dtype, seed=10 + k)
    scale = 1 / math.sqrt(d)
    dims = dsa.make_dims(L, Hq, d, 8, 64, k, scale=scale, dtype=dtype)
    O = torch.empty((L, Hq, d), dtype=_tdt(dtype), device=DEV)
    lse = torch.empty((L, Hq), device=DEV)
    dsa.sparse_attn_fwd(dims, Q.to(DEV), K.to(DEV), V.to(DEV), torch.from_numpy(idx).to(DEV), O, lse)
    dsa.check_device_error()
    Or, LSEr = oracle.attn_fwd(_f32(Q), _f32(K), _f32(V), idx, scale)
    assert np.abs(_f32(O) - Or).max() <= TOL[dtype]
    assert np.abs(lse.cpu().numpy() - LSEr).max() <= (1e-3 if dtype == "bf16" else 1e-4)
    # with the fp32 output: O and LSE unchanged bit for bit (fp32 layers) or within
    # tolerance (bf16: P.V now carries the low part of P), o_acc within 1e-4
    O2, lse2 = torch.empty_like(O), torch.empty_like(lse)
    o_acc = torch.full((L, Hq, d), float("nan"), device=DEV)
    dsa.sparse_attn_fwd(dims, Q.to(DEV), K.to(DEV), V.to(DEV), torch.from_numpy(idx).to(DEV), O2, lse2, o_acc=o_acc)
    dsa.check_device_error()
    assert torch.equal(lse2, lse)
    assert np.abs(_f32(O2) - Or).max() <= TOL[dtype]
    assert np.abs(o_acc.cpu().numpy() - Or).max() <= 1e-4
    if dtype == "fp32":
        assert torch.equal(O2, O) and torch.equal(o_acc, O)


@pytest.mark.parametrize("Hq", [16, 32])
@pytest.mark.parametrize("spiky", [False, True])
def test_attn_fwd_tc_many_tiles_and_queries(Hq, spiky):
    """The tcgen05 forward at L = 8192, k = 512: 16 key tiles per query and
    tens of queries per persistent CTA, so every stage ring, accumulator and
    barrier phase wraps many times.  `spiky` scales Q by 6, so the scores
    span ~2^9 and the softmax base moves (rescaling O in tensor memory) on
    many tiles.  Sampled rows (the first 40, whose selections are padded with
    -1, and a spread of later ones) against the oracle, with and without
    o_acc; every row against the warp-level kernel."""
    L, d, k = 8192, 128, 512
    Q, K, V, _, idx = _attn_case(L, Hq, d, k, "bf16", seed=90 + Hq)
    if spiky:
        Q = (Q.float() * 6).to(torch.bfloat16)
    scale = 1 / math.sqrt(d)
    dims = dsa.make_dims(L, Hq, d, 8, 64, k, scale=scale, dtype="bf16")
    dev = [t.to(DEV) for t in (Q, K, V)]
    idx_d = torch.from_numpy(idx).to(DEV)
    out = {}
    try:
        for route in (1, 0):
            dsa.set_attn_fwd_route(route)
            O = torch.empty((L, Hq, d), dtype=torch.bfloat16, device=DEV)
            lse = torch.empty((L, Hq), device=DEV)
            o_acc = torch.full((L, Hq, d), float("nan"), device=DEV)
            dsa.sparse_attn_fwd(dims, *dev, idx_d, O, lse, o_acc=o_acc)
            O2 = torch.empty_like(O)
            lse2 = torch.empty_like(lse)
            dsa.sparse_attn_fwd(dims, *dev, idx_d, O2, lse2)
            dsa.check_device_error()
            out[route] = (O, lse, o_acc, O2, lse2)
    finally:
        dsa.set_attn_fwd_route(0)
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([np.arange(40), rng.integers(40, L, 88), [L - 4, L - 3, L - 2, L - 1]]))
    Or, LSEr = oracle.attn_fwd(_f32(Q), _f32(K), _f32(V), idx, scale, rows=rows)
    O, lse, o_acc, O2, lse2 = out[1]
    assert torch.equal(lse2, lse)
    assert np.abs(_f32(O)[rows] - Or).max() <= 2e-2
    assert np.abs(_f32(O2)[rows] - Or).max() <= 2e-2
    assert np.abs(lse.cpu().numpy()[rows] - LSEr).max() <= 1e-3
    assert np.abs(o_acc.cpu().numpy()[rows] - Or).max() <= 1e-4
    Ow, lsew, accw, _, _ = out[0]
    assert (O.float() - Ow.float()).abs().max().item() <= 2e-2
    assert (lse - lsew).abs().max().item() <= 1e-4
    assert (o_acc - accw).abs().max().item() <= 1e-4


def _bwd(det, dims, dev, idx_d, O, lse, dq, dk, dv, o_acc):
    """The atomic backward (det=False) or the deterministic one (det=True)."""
    if det:
        ws = dsa.alloc_bwd_det_workspace(dims, DEV)
        ws.fill_(0x5A)                              # nothing in it may need to start at zero
        dsa.sparse_attn_bwd_det(dims, dev[0], dev[1], dev[2], idx_d, O, lse, dev[3], dq, dk, dv, ws, o_acc=o_acc)
    else:
        ws = None if o_acc is not None else dsa.alloc_backward_workspace(dims, DEV)
        dsa.sparse_attn_bwd(dims, dev[0], dev[1], dev[2], idx_d, O, lse, dev[3], dq, dk, dv, ws, o_acc=o_acc)


@pytest.mark.parametrize("Hq,d", [(16, 128), (32, 128), (16, 64), (32, 64)])
@pytest.mark.parametrize("k", [3, 32])
@pytest.mark.parametrize("use_o_acc", [False, True])
def test_attn_bwd_det_matches_oracle_and_repeats(Hq, d, k, use_o_acc):
    """The deterministic backward: dQ, dK, dV within 2e-2 of the oracle, the
    same bits on a second call (on a dirty workspace), and dQ bit-identical to
    the atomic backward's (the same query-major arithmetic)."""
    L = 1000
    Q, K, V, dO, idx = _attn_case(L, Hq, d, k, "bf16", seed=60 + k)
    scale = 1 / math.sqrt(d)
    dims = dsa.make_dims(L, Hq, d, 8, 64, k, scale=scale)
    dev = [t.to(DEV) for t in (Q, K, V, dO)]
    idx_d = torch.from_numpy(idx).to(DEV)
    O = torch.empty((L, Hq, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((L, Hq), device=DEV)
    o_acc = torch.empty((L, Hq, d), device=DEV) if use_o_acc else None
    dsa.sparse_attn_fwd(dims, dev[0], dev[1], dev[2], idx_d, O, lse, o_acc=o_acc)
    runs = []
    for _ in range(2):
        dq = torch.full((L, Hq, d), 3.0, device=DEV)
        dk = torch.full((L, d), 5.0, device=DEV)    # overwritten, not accumulated into
        dv = torch.full((L, d), 5.0, device=DEV)
        _bwd(True, dims, dev, idx_d, O, lse, dq, dk, dv, o_acc)
        runs.append((dq, dk, dv))
    dsa.check_device_error()
    for a, b in zip(runs[0], runs[1]):
        assert torch.equal(a, b)
    dq_a = torch.empty((L, Hq, d), device=DEV)
    dk_a, dv_a = torch.empty((L, d), device=DEV), torch.empty((L, d), device=DEV)
    _bwd(False, dims, dev, idx_d, O, lse, dq_a, dk_a, dv_a, o_acc)
    dsa.check_device_error()
    assert torch.equal(runs[0][0], dq_a)
    dQr, dKr, dVr = oracle.attn_bwd(_f32(Q), _f32(K), _f32(V), idx, _f32(dO), scale, threads=8)
    errs = {name: float(np.abs(got.cpu().numpy() - ref).max())
            for name, got, ref in (("dQ", runs[0][0], dQr), ("dK", runs[0][1], dKr), ("dV", runs[0][2], dVr))}
    assert max(errs.values()) <= 2e-2, errs


@pytest.mark.parametrize("Hq,d", [(16, 128), (32, 128), (16, 64), (32, 64)])
@pytest.mark.parametrize("k", [3, 32])
@pytest.mark.parametrize("use_o_acc", [False, True])
def test_attn_bwd_matches_oracle(Hq, d, k, use_o_acc):
    L = 1000
    Q, K, V, dO, idx = _attn_case(L, Hq, d, k, "bf16", seed=20 + k)
    scale = 1 / math.sqrt(d)
    dims = dsa.make_dims(L, Hq, d, 8, 64, k, scale=scale)
    dev = [t.to(DEV) for t in (Q, K, V, dO)]
    idx_d = torch.from_numpy(idx).to(DEV)
    O = torch.empty((L, Hq, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((L, Hq), device=DEV)
    o_acc = torch.empty((L, Hq, d), device=DEV) if use_o_acc else None
    dsa.sparse_attn_fwd(dims, dev[0], dev[1], dev[2], idx_d, O, lse, o_acc=o_acc)
    dq = torch.empty((L, Hq, d), device=DEV)
    dk = torch.full((L, d), 5.0, device=DEV)     # must be overwritten, not accumulated into
    dv = torch.full((L, d), 5.0, device=DEV)
    ws = None if use_o_acc else dsa.alloc_backward_workspace(dims, DEV)
    dsa.sparse_attn_bwd(dims, dev[0], dev[1], dev[2], idx_d, O, lse, dev[3], dq, dk, dv, ws, o_acc=o_acc)
    dsa.check_device_error()
    dQr, dKr, dVr = oracle.attn_bwd(_f32(Q), _f32(K), _f32(V), idx, _f32(dO), scale, threads=8)
    errs = {name: float(np.abs(got.cpu().numpy() - ref).max())
            for name, got, ref in (("dQ", dq, dQr), ("dK", dk, dKr), ("dV", dv, dVr))}
    assert max(errs.values()) <= 2e-2, errs


@pytest.mark.parametrize("case", ["dO_times_1e-6", "beyond_fp16_range", "unit_scale"])
@pytest.mark.parametrize("use_o_acc", [False, True])
@pytest.mark.parametrize("det", [False, True])
def test_attn_bwd_scaled_inputs(case, use_o_acc, det):
    """Inputs far from unit scale, compared element by element with the oracle.

    A loss-scaled upstream gradient (dO ~ 1e-6 per element) and Q / dO entries
    above 65504 (fp16's largest finite value, with K scaled down by the same
    power of two so the softmax stays unsaturated) are legal bf16 inputs.  The
    gradients scale with the inputs: dV with dO, dK with dO * Q, dQ with dO * K,
    so each is held to the 2e-2 bound times its own scale."""
    L, Hq, d, k = 1000, 16, 128, 32
    Q, K, V, dO, idx = _attn_case(L, Hq, d, k, "bf16", seed=31)
    sQ = sK = sdO = 1.0
    if case == "dO_times_1e-6":
        sdO = 1e-6
    elif case == "beyond_fp16_range":
        sQ, sK, sdO = 2.0 ** 17, 2.0 ** -17, 2.0 ** 17
    Q = (Q.float() * sQ).to(torch.bfloat16)
    K = (K.float() * sK).to(torch.bfloat16)
    dO = (dO.float() * sdO).to(torch.bfloat16)
    if case == "beyond_fp16_range":
        assert float(Q.float().abs().max()) > 65504 and float(dO.float().abs().max()) > 65504
    scale = 1 / math.sqrt(d)
    dims = dsa.make_dims(L, Hq, d, 8, 64, k, scale=scale)
    dev = [t.to(DEV) for t in (Q, K, V, dO)]
    idx_d = torch.from_numpy(idx).to(DEV)
    O = torch.empty((L, Hq, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((L, Hq), device=DEV)
    o_acc = torch.empty((L, Hq, d), device=DEV) if use_o_acc else None
    dsa.sparse_attn_fwd(dims, dev[0], dev[1], dev[2], idx_d, O, lse, o_acc=o_acc)
    dq = torch.empty((L, Hq, d), device=DEV)
    dk = torch.empty((L, d), device=DEV)
    dv = torch.empty((L, d), device=DEV)
    _bwd(det, dims, dev, idx_d, O, lse, dq, dk, dv, o_acc)
    dsa.check_device_error()
    dQr, dKr, dVr = oracle.attn_bwd(_f32(Q), _f32(K), _f32(V), idx, _f32(dO), scale, threads=8)
    grad_scale = {"dQ": sdO * sK, "dK": sdO * sQ, "dV": sdO}
    for name, got, ref in (("dQ", dq, dQr), ("dK", dk, dKr), ("dV", dv, dVr)):
        g = got.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(g)), name
        err = float(np.abs(g - ref).max()) / grad_scale[name]
        assert err <= 2e-2, (name, err)
        # not flushed to zero: the gradient carries the reference's magnitude
        assert np.abs(g).max() >= 0.5 * np.abs(ref).max(), name


def test_attn_bad_index_is_skipped_and_reported(fwd_route):
    L, Hq, d, k = 256, 16, 128, 4
    Q, K, V, _, idx = _attn_case(L, Hq, d, k, "bf16", seed=5)
    idx = idx.copy()
    idx[200, 0] = 10_000          # beyond the sequence
    idx[100, 1] = 30              # pool 30 ends at token 123 > 100: the future
    dims = dsa.make_dims(L, Hq, d, 8, 64, k)
    O = torch.empty((L, Hq, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((L, Hq), device=DEV)
    dsa.sparse_attn_fwd(dims, Q.to(DEV), K.to(DEV), V.to(DEV), torch.from_numpy(idx).to(DEV), O, lse)
    with pytest.raises(dsa.DSAError) as e:
        dsa.check_device_error()
    assert e.value.status == dsa.DSA_ERR_BAD_INDEX
    clean = idx.copy()
    clean[200, 0] = -1
    clean[100, 1] = -1
    Or, _ = oracle.attn_fwd(_f32(Q), _f32(K), _f32(V), clean, 1 / math.sqrt(d), rows=[100, 200])
    assert np.abs(_f32(O)[[100, 200]] - Or).max() <= 2e-2


@pytest.mark.parametrize("use_o_acc", [False, True])
def test_attn_bwd_two_head_groups_long_rows(use_o_acc):
    """Hq = 32: the two 16-head groups of a query are a warp pair that sums its
    dK/dV tiles before one reduction per key.  L = 4096 with k = 256 gives rows
    of up to 65 key steps (so the pair's barriers and shared stages cycle many
    times), compared element by element with the oracle."""
    L, Hq, d, k = 4096, 32, 128, 256
    Q, K, V, dO, idx = _attn_case(L, Hq, d, k, "bf16", seed=77)
    scale = 1 / math.sqrt(d)
    dims = dsa.make_dims(L, Hq, d, 8, 64, k, scale=scale, dtype="bf16")
    dev = [t.to(DEV) for t in (Q, K, V, dO)]
    idx_d = torch.from_numpy(idx).to(DEV)
    O = torch.empty((L, Hq, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((L, Hq), device=DEV)
    o_acc = torch.empty((L, Hq, d), device=DEV) if use_o_acc else None
    dsa.sparse_attn_fwd(dims, dev[0], dev[1], dev[2], idx_d, O, lse, o_acc=o_acc)
    dq = torch.empty((L, Hq, d), device=DEV)
    dk = torch.empty((L, d), device=DEV)
    dv = torch.empty((L, d), device=DEV)
    _bwd(False, dims, dev, idx_d, O, lse, dq, dk, dv, o_acc)
    dsa.check_device_error()
    dQr, dKr, dVr = oracle.attn_bwd(_f32(Q), _f32(K), _f32(V), idx, _f32(dO), scale, threads=8)
    errs = {name: float(np.abs(got.cpu().numpy() - ref).max())
            for name, got, ref in (("dQ", dq, dQr), ("dK", dk, dKr), ("dV", dv, dVr))}
    assert max(errs.values()) <= 2e-2, errs

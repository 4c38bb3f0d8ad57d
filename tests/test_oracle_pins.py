"""Pins for the CPU oracle, checked against things other than itself.

Each test ties one oracle function to a closed form, an invariant, a brute
force on tiny inputs, a torch library routine on a different formulation, or
a number the pages print ("SkyRL extends GLM-5.3-Flash training context to 1
million tokens": about 2048 keys per query, exactly 2051 in the Flash
variant; one pool per 4 tokens).  The tests are chosen so that a plausible
mistake in the oracle (a dropped term, a wrong sign or index, a transposed
operand, a wrong tie rule) fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------- bf16
def test_round_bf16_matches_torch_rne():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * 10.0,
        (rng.integers(-(1 << 20), 1 << 20, 2000) / 1024.0).astype(np.float32),
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130, 3.0e38, -0.0, 0.0], np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    got = np.array([oracle.round_bf16(float(v)) for v in x], np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_round_bf16_ties_to_even():
    # halfway between 1 and 1+2^-7 -> 1 (even); halfway between 1+2^-7 and 1+2^-6 -> 1+2^-6
    assert oracle.round_bf16(1 + 2 ** -8) == 1.0
    assert oracle.round_bf16(1 + 3 * 2 ** -8) == 1 + 2 ** -6
    assert oracle.round_bf16(1 + 2 ** -8 + 2 ** -20) == 1 + 2 ** -7


# ---------------------------------------------------------------- pool keys
def test_pool_keys_integer_inputs_equal_block_sum():
    rng = np.random.default_rng(1)
    k_I = rng.integers(-3, 4, size=(64, 16)).astype(np.float32)
    expect = k_I.reshape(16, 4, 16).sum(axis=1)          # numpy reduction, exact for small integers
    for rnd in (False, True):
        assert np.array_equal(oracle.pool_keys(k_I, rnd), expect)


def test_pool_keys_fp32_order_and_single_rounding():
    # ((1 + 2^-24) + 2^-24) + 2^-24 in fp32 stays 1.0 (each add is a tie to even);
    # the exact sum 1 + 3*2^-24 would round to 1 + 2^-22.
    e = 2.0 ** -24
    k_I = np.array([[1.0], [e], [e], [e]], np.float32)
    assert oracle.pool_keys(k_I, False)[0, 0] == np.float32(1.0)
    # bf16 pool: fp32 sum 1 + 2^-8 + 2^-20 (exact in fp32) rounds once, up to 1 + 2^-7;
    # rounding after every add would give 1.0.
    k_I = np.array([[1.0], [2 ** -8], [2 ** -20], [0.0]], np.float32)
    assert oracle.pool_keys(k_I, True)[0, 0] == np.float32(1 + 2 ** -7)


def test_pool_keys_gated_unit_gates_are_the_plain_sum():
    # fma(1, k, acc) rounds exactly like acc + k, so all-one gates give the plain pool bit for bit
    rng = np.random.default_rng(21)
    k_I = rng.standard_normal((256, 32)).astype(np.float32)
    g = np.ones(256, np.float32)
    for rnd in (False, True):
        assert np.array_equal(oracle.pool_keys_gated(k_I, g, rnd).view(np.uint32),
                              oracle.pool_keys(k_I, rnd).view(np.uint32))


def test_pool_keys_gated_one_hot_gates_pick_one_token():
    rng = np.random.default_rng(22)
    L, di = 64, 16
    k_I = rng.standard_normal((L, di)).astype(np.float32)
    pick = rng.integers(0, 4, size=L // 4)
    g = np.zeros(L, np.float32)
    g[4 * np.arange(L // 4) + pick] = 1.0
    expect = k_I[4 * np.arange(L // 4) + pick]
    assert np.array_equal(oracle.pool_keys_gated(k_I, g, False), expect)
    assert np.array_equal(oracle.pool_keys_gated(k_I, np.zeros(L, np.float32), False), np.zeros((L // 4, di)))


def test_pool_keys_gated_integer_inputs_equal_weighted_block_sum():
    # small integers: every product and partial sum is exact in fp32, so the result is the
    # exact weighted sum, computed here in int64 by numpy
    rng = np.random.default_rng(23)
    L, di = 128, 8
    k_I = rng.integers(-3, 4, size=(L, di))
    g = rng.integers(-2, 5, size=L)
    expect = (g[:, None] * k_I).reshape(L // 4, 4, di).sum(axis=1)
    for rnd in (False, True):   # |sum| <= 48: exact in bf16 as well
        assert np.array_equal(oracle.pool_keys_gated(k_I.astype(np.float32), g.astype(np.float32), rnd), expect)


def test_pool_keys_gated_fma_chain_and_single_rounding():
    # one token: gate 1 + 2^-12 times key 1 + 2^-12 = 1 + 2^-11 + 2^-24 exactly; the first fma
    # from 0 rounds it to fp32 (a tie, to even: 1 + 2^-11), then fma with the next token
    # 2^-24 * 1 lands on the tie again (1 + 2^-11 + 2^-24 -> 1 + 2^-11)
    a = np.float32(1 + 2.0 ** -12)
    k_I = np.array([[a], [1.0], [0.0], [0.0]], np.float32)
    g = np.array([a, 2.0 ** -24, 0.0, 0.0], np.float32)
    assert oracle.pool_keys_gated(k_I, g, False)[0, 0] == np.float32(1 + 2.0 ** -11)
    # fused, not multiply-then-add: token 0 leaves acc = -(3 + 2^-21); token 1's product
    # 3 * (1 + 2^-23) = 3 + 3*2^-23 is not exact in fp32.  One fma gives the exact
    # -(3 + 2^-21) + 3 + 3*2^-23 = -2^-23; rounding the product first (a tie, to even:
    # 3 + 2^-21) and then adding would give 0.
    k_I = np.array([[-(3 + 2.0 ** -21)], [1 + 2.0 ** -23], [0.0], [0.0]], np.float32)
    g = np.array([1.0, 3.0, 0.0, 0.0], np.float32)
    assert oracle.pool_keys_gated(k_I, g, False)[0, 0] == np.float32(-(2.0 ** -23))


# ------------------------------------------------------------------ indexer
def _rand_idx_inputs(rng, L, Hi, di, positive=False):
    if positive:
        q = rng.integers(1, 4, size=(L, Hi, di)).astype(np.float32)
        k = rng.integers(1, 4, size=(L, di)).astype(np.float32)
    else:
        q = rng.integers(-3, 4, size=(L, Hi, di)).astype(np.float32)
        k = rng.integers(-3, 4, size=(L, di)).astype(np.float32)
    w = rng.integers(1, 5, size=(L, Hi)).astype(np.float32)
    return q, k, w


def test_indexer_causal_mask_is_exactly_elig():
    rng = np.random.default_rng(2)
    L = 64
    q, k, w = _rand_idx_inputs(rng, L, 2, 8)
    s = oracle.indexer_scores(q, oracle.pool_keys(k, False), w)
    for t in range(L):
        e = (t + 1) // 4          # pool p is complete at token t iff 4p+3 <= t
        assert np.all(np.isfinite(s[t, :e])) and np.all(np.isnan(s[t, e:]))


def test_indexer_without_active_relu_collapses_heads_into_one_matmul():
    # All-positive q and k: ReLU never clips, so sum_h w_h (q_h . kp) = (sum_h w_h q_h) . kp,
    # a single matrix product computed by numpy in a different association.
    rng = np.random.default_rng(3)
    L, Hi, di = 128, 4, 16
    q, k, w = _rand_idx_inputs(rng, L, Hi, di, positive=True)
    kp = oracle.pool_keys(k, False)
    s = oracle.indexer_scores(q, kp, w)
    qeff = np.einsum("th,thi->ti", w.astype(np.float64), q.astype(np.float64))
    full = qeff @ kp.astype(np.float64).T
    for t in range(L):
        e = (t + 1) // 4
        assert np.array_equal(s[t, :e], full[t, :e])


def test_indexer_relu_clips_negative_heads():
    # head 0 = +u, head 1 = -u with positive pool keys: head 1 is clipped to 0.
    rng = np.random.default_rng(4)
    L, di = 32, 8
    u = rng.integers(1, 4, size=(L, di)).astype(np.float32)
    q = np.stack([u, -u], axis=1)
    k = rng.integers(1, 3, size=(L, di)).astype(np.float32)
    w = np.array([[2.0, 3.0]] * L, np.float32)
    kp = oracle.pool_keys(k, False)
    s = oracle.indexer_scores(q, kp, w)
    ref = 2.0 * (u.astype(np.float64) @ kp.astype(np.float64).T)
    for t in range(L):
        e = (t + 1) // 4
        assert np.array_equal(s[t, :e], ref[t, :e])
    # swapping the head weights scales by 3/2 -- catches a w/head index mix-up
    s2 = oracle.indexer_scores(q, kp, w[:, ::-1].copy())
    for t in range(L):
        e = (t + 1) // 4
        assert np.allclose(s2[t, :e], 1.5 * s[t, :e], rtol=0, atol=0)


def test_indexer_homogeneity_and_head_additivity():
    rng = np.random.default_rng(5)
    L, Hi, di = 48, 3, 8
    q, k, w = _rand_idx_inputs(rng, L, Hi, di)
    kp = oracle.pool_keys(k, False)
    s = oracle.indexer_scores(q, kp, w)
    assert np.array_equal(oracle.indexer_scores(2 * q, kp, w), 2 * s, equal_nan=True)
    assert np.array_equal(oracle.indexer_scores(q, kp, -w), -s, equal_nan=True)
    parts = 0
    for h in range(Hi):
        wh = np.zeros_like(w)
        wh[:, h] = w[:, h]
        parts = parts + oracle.indexer_scores(q, kp, wh)
    assert np.array_equal(parts, s, equal_nan=True)


def test_indexer_rows_are_independent_of_chunking():
    rng = np.random.default_rng(6)
    L = 96
    q, k, w = _rand_idx_inputs(rng, L, 2, 8)
    kp = oracle.pool_keys(k, False)
    full = oracle.indexer_scores(q, kp, w)
    for a, b in ((0, 32), (32, 64), (64, 96), (17, 59)):
        assert np.array_equal(oracle.indexer_scores(q, kp, w, np.arange(a, b)), full[a:b], equal_nan=True)


# -------------------------------------------------------------------- top-k
def _exchange_ok(sel, s, e):
    """Defining property of 'top-k, ties to the lower index' on a row."""
    sel = set(sel)
    for p in sel:
        for q in range(e):
            if q in sel:
                continue
            if not (s[p] > s[q] or (s[p] == s[q] and p < q)):
                return False
    return True


@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force_tiny(seed):
    rng = np.random.default_rng(100 + seed)
    L = 32
    P = L // 4
    for k in (1, 2, 3):
        # coarse integer scores -> many ties
        s = rng.integers(-2, 3, size=(L, P)).astype(np.float64)
        for t in range(L):
            s[t, (t + 1) // 4:] = np.nan
        idx = oracle.topk(s, L, k)
        for t in range(L):
            e = (t + 1) // 4
            m = min(k, e)
            sel = [p for p in idx[t] if p >= 0]
            assert len(sel) == m and list(idx[t][m:]) == [-1] * (k - m)
            assert sel == sorted(sel)
            # brute force: exactly one m-subset satisfies the exchange property, and it is ours
            good = [c for c in itertools.combinations(range(e), m) if _exchange_ok(c, s[t], e)]
            assert good == [tuple(sel)]


def test_topk_ties_signed_zero_and_negative_scores():
    L = 32
    P = L // 4
    s = np.full((L, P), np.nan)
    t = L - 1                           # e = 8
    s[t] = [-0.0, 0.0, -1.0, -0.0, 2.0, -3.0, 0.0, -1.0]
    idx = oracle.topk(s, L, 4, rows=None)[t]
    # 2.0 first, then the zeros (-0 == +0) by ascending index: 0, 1, 3
    assert list(idx) == [0, 1, 3, 4]
    s2 = np.full((L, P), np.nan)
    s2[t] = 5.0
    assert list(oracle.topk(s2, L, 3)[t]) == [0, 1, 2]


def test_topk_short_rows_pad_with_minus_one():
    L, k = 40, 4
    s = np.full((L, L // 4), np.nan)
    for t in range(L):
        s[t, :(t + 1) // 4] = 1.0
    idx = oracle.topk(s, L, k)
    assert list(idx[0]) == [-1] * 4 and list(idx[2]) == [-1] * 4
    assert list(idx[3]) == [0, -1, -1, -1]
    assert list(idx[11]) == [0, 1, 2, -1]


# --------------------------------------------------------------- key counts
def test_key_counts_and_the_2051_bound():
    with open(os.path.join(GOLDEN, "key_counts.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for t_s, k_s, n_s in rows:
        t, k, n = int(t_s), int(k_s), int(n_s)
        e = (t + 1) // 4
        idx_row = np.array(list(range(min(k, e))) + [-1] * (k - min(k, e)), np.int32)
        assert oracle.key_set(t, idx_row, k).size == n


def test_key_set_contents():
    k = 2
    assert list(oracle.key_set(0, np.array([-1, -1], np.int32), k)) == [0]
    assert list(oracle.key_set(2, np.array([-1, -1], np.int32), k)) == [0, 1, 2]
    assert list(oracle.key_set(3, np.array([0, -1], np.int32), k)) == [0, 1, 2, 3]     # own pool complete: competes
    assert list(oracle.key_set(3, np.array([-1, -1], np.int32), k)) == []
    assert list(oracle.key_set(9, np.array([0, 1], np.int32), k)) == [0, 1, 2, 3, 4, 5, 6, 7, 8, 9]
    with pytest.raises(ValueError):
        oracle.key_set(5, np.array([1, -1], np.int32), k)                               # pool 1 ends at token 7 > 5


# ---------------------------------------------------------------- attention
def _mask_from_idx(idx, L):
    k = idx.shape[1]
    m = np.zeros((L, L), bool)
    for t in range(L):
        m[t, oracle.key_set(t, idx[t], k)] = True
    return m


def _torch_masked_attention(Q, K, V, mask, scale):
    q = torch.from_numpy(Q.astype(np.float64)).transpose(0, 1)        # [Hq, L, d]
    kk = torch.from_numpy(K.astype(np.float64))
    vv = torch.from_numpy(V.astype(np.float64))
    s = scale * q @ kk.T                                              # [Hq, L, L]
    s = s.masked_fill(~torch.from_numpy(mask), float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    o = torch.softmax(s, dim=-1) @ vv
    return o.transpose(0, 1).numpy(), lse.T.numpy()


def test_attention_with_all_pools_equals_dense_causal_sdpa():
    rng = np.random.default_rng(7)
    L, Hq, d = 256, 4, 16
    Q = rng.standard_normal((L, Hq, d)).astype(np.float32)
    K = rng.standard_normal((L, d)).astype(np.float32)
    V = rng.standard_normal((L, d)).astype(np.float32)
    k = L // 4                                     # every eligible pool is selected
    idx = np.full((L, k), -1, np.int32)
    for t in range(L):
        e = (t + 1) // 4
        idx[t, :e] = np.arange(e)
    scale = 1 / math.sqrt(d)
    O, LSE = oracle.attn_fwd(Q, K, V, idx, scale)
    q = torch.from_numpy(Q.astype(np.float64)).transpose(0, 1)[None]
    kk = torch.from_numpy(K.astype(np.float64))[None, None].expand(1, Hq, L, d)
    vv = torch.from_numpy(V.astype(np.float64))[None, None].expand(1, Hq, L, d)
    ref = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, is_causal=True, scale=scale)
    assert np.abs(O - ref[0].transpose(0, 1).numpy()).max() < 1e-12


def test_attention_matches_torch_softmax_on_sparse_mask():
    rng = np.random.default_rng(8)
    L, Hq, d, k = 128, 3, 8, 5
    Q = rng.standard_normal((L, Hq, d)).astype(np.float32)
    K = rng.standard_normal((L, d)).astype(np.float32)
    V = rng.standard_normal((L, d)).astype(np.float32)
    q_I, k_I, w = _rand_idx_inputs(rng, L, 2, 8)
    kp = oracle.pool_keys(k_I, False)
    idx = oracle.topk(oracle.indexer_scores(q_I, kp, w), L, k)
    O, LSE = oracle.attn_fwd(Q, K, V, idx, 0.3)
    Or, LSEr = _torch_masked_attention(Q, K, V, _mask_from_idx(idx, L), 0.3)
    assert np.abs(O - Or).max() < 1e-12 and np.abs(LSE - LSEr).max() < 1e-12


def test_attention_special_cases():
    rng = np.random.default_rng(9)
    L, Hq, d, k = 64, 2, 8, 3
    Q = rng.standard_normal((L, Hq, d)).astype(np.float32)
    K = np.tile(rng.standard_normal((1, d)).astype(np.float32), (L, 1))    # all keys equal
    V = rng.standard_normal((L, d)).astype(np.float32)
    idx = np.full((L, k), -1, np.int32)
    for t in range(L):
        e = (t + 1) // 4
        idx[t, :min(k, e)] = np.arange(max(0, e - min(k, e)), e)
    O, LSE = oracle.attn_fwd(Q, K, V, idx, 0.5)
    for t in (0, 1, 3, 10, 63):
        keys = oracle.key_set(t, idx[t], k)
        assert np.abs(O[t] - V[keys].astype(np.float64).mean(0)).max() < 1e-12
        s = 0.5 * Q[t].astype(np.float64) @ K[0].astype(np.float64)
        assert np.abs(LSE[t] - (s + math.log(len(keys)))).max() < 1e-12
    # k=1 at t=3: only pool 0, i.e. the mean of V[0..3]
    idx1 = np.full((L, 1), -1, np.int32)
    idx1[3, 0] = 0
    O1, _ = oracle.attn_fwd(Q, K, V, idx1, 0.5, rows=[3])
    assert np.abs(O1[0] - V[0:4].astype(np.float64).mean(0)).max() < 1e-12


# ----------------------------------------------------------------- backward
def _small_case(seed, L=64, Hq=2, d=8, k=4):
    rng = np.random.default_rng(seed)
    Q = rng.standard_normal((L, Hq, d))
    K = rng.standard_normal((L, d))
    V = rng.standard_normal((L, d))
    dO = rng.standard_normal((L, Hq, d))
    q_I, k_I, w = _rand_idx_inputs(rng, L, 2, 8)
    idx = oracle.topk(oracle.indexer_scores(q_I, oracle.pool_keys(k_I, False), w), L, k)
    # inputs exact in fp32, which the oracle takes
    return [a.astype(np.float32) for a in (Q, K, V, dO)] + [idx]


def test_backward_matches_central_finite_differences():
    Q, K, V, dO, idx = _small_case(10)
    scale = 1 / math.sqrt(Q.shape[2])
    dQ, dK, dV = oracle.attn_bwd(Q, K, V, idx, dO, scale)
    go = dO.astype(np.float64)

    def loss(Qx, Kx, Vx):
        # the oracle takes fp32 arrays; perturb in fp64 through the torch formulation
        q = torch.from_numpy(Qx).transpose(0, 1)
        s = scale * q @ torch.from_numpy(Kx).T
        s = s.masked_fill(~torch.from_numpy(mask), float("-inf"))
        o = torch.softmax(s, -1) @ torch.from_numpy(Vx)
        return float((o.transpose(0, 1).numpy() * go).sum())

    mask = _mask_from_idx(idx, Q.shape[0])
    h = 1e-6
    rng = np.random.default_rng(11)
    Q64, K64, V64 = (a.astype(np.float64) for a in (Q, K, V))
    for name, X, G in (("Q", Q64, dQ), ("K", K64, dK), ("V", V64, dV)):
        for _ in range(12):
            pos = tuple(int(rng.integers(0, n)) for n in X.shape)
            Xp, Xm = X.copy(), X.copy()
            Xp[pos] += h
            Xm[pos] -= h
            args_p = {"Q": Q64, "K": K64, "V": V64}
            args_m = dict(args_p)
            args_p[name], args_m[name] = Xp, Xm
            fd = (loss(args_p["Q"], args_p["K"], args_p["V"]) - loss(args_m["Q"], args_m["K"], args_m["V"])) / (2 * h)
            assert abs(fd - G[pos]) <= 1e-6 * max(1.0, abs(G[pos])), (name, pos, fd, G[pos])


def test_backward_matches_torch_autograd_and_sharding():
    Q, K, V, dO, idx = _small_case(12, L=96, Hq=3, d=8, k=3)
    L = Q.shape[0]
    scale = 0.4
    mask = torch.from_numpy(_mask_from_idx(idx, L))
    q = torch.from_numpy(Q.astype(np.float64)).requires_grad_()
    kk = torch.from_numpy(K.astype(np.float64)).requires_grad_()
    vv = torch.from_numpy(V.astype(np.float64)).requires_grad_()
    s = scale * q.transpose(0, 1) @ kk.T
    o = torch.softmax(s.masked_fill(~mask, float("-inf")), -1) @ vv
    o.transpose(0, 1).backward(torch.from_numpy(dO.astype(np.float64)))
    dQ, dK, dV = oracle.attn_bwd(Q, K, V, idx, dO, scale)
    assert np.abs(dQ - q.grad.numpy()).max() < 1e-12
    assert np.abs(dK - kk.grad.numpy()).max() < 1e-12
    assert np.abs(dV - vv.grad.numpy()).max() < 1e-12
    dQ4, dK4, dV4 = oracle.attn_bwd(Q, K, V, idx, dO, scale, threads=4)
    assert np.abs(dQ4 - dQ).max() < 1e-12 and np.abs(dK4 - dK).max() < 1e-12 and np.abs(dV4 - dV).max() < 1e-12


def test_layer_forward_end_to_end_tiny_matches_torch():
    rng = np.random.default_rng(13)
    L, Hq, d, Hi, di, k = 64, 2, 8, 2, 8, 3
    Q = rng.standard_normal((L, Hq, d)).astype(np.float32)
    K = rng.standard_normal((L, d)).astype(np.float32)
    V = rng.standard_normal((L, d)).astype(np.float32)
    q_I, k_I, w = _rand_idx_inputs(rng, L, Hi, di)
    kp, idx, O, LSE = oracle.layer_fwd(Q, K, V, q_I, k_I, w, k, 0.35, False)
    # selection by brute force on integer scores computed with torch (a different formulation: einsum)
    kpt = torch.from_numpy(k_I.astype(np.float64)).view(L // 4, 4, di).sum(1)
    dots = torch.einsum("thi,pi->thp", torch.from_numpy(q_I.astype(np.float64)), kpt).clamp_min(0)
    sc = torch.einsum("th,thp->tp", torch.from_numpy(w.astype(np.float64)), dots).numpy()
    for t in range(L):
        e = (t + 1) // 4
        m = min(k, e)
        order = sorted(range(e), key=lambda p: (-sc[t, p], p))[:m]
        assert list(idx[t][:m]) == sorted(order)
    Or, _ = _torch_masked_attention(Q, K, V, _mask_from_idx(idx, L), 0.35)
    assert np.abs(O - Or).max() < 1e-12

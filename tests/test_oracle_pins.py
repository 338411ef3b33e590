"""Pins for the CPU oracle (no GPU).

Each test ties an oracle function to something other than itself: a library
routine that a special case reduces to (numpy matmul, torch's bf16 rounding,
torch SDPA and autograd in fp64), exhaustive enumeration on tiny inputs,
closed forms, invariants, or the golden values under tests/golden/.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def bf16_bits(x) -> np.ndarray:
    """fp32/fp64 array -> bf16 bit patterns via torch's own rounding."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b) -> np.ndarray:
    return oracle.bf16_to_f32(b).astype(np.float64)


def rand_bf16(shape, std=1.0, rng=RNG):
    return bf16_bits(rng.standard_normal(shape) * std)


# ---------------------------------------------------------------- bf16


def test_bf16_rounding_matches_torch():
    vals = np.concatenate([
        RNG.standard_normal(4000).astype(np.float32),
        (RNG.standard_normal(2000) * 1e-38).astype(np.float32),  # subnormal
        (RNG.standard_normal(2000) * 1e30).astype(np.float32),
        # exact halfway points between bf16 neighbours, odd and even
        (np.arange(1, 600, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, -3.3895314e38],
                 np.float32),
    ])
    ours = oracle.f32_to_bf16(vals)
    ref = bf16_bits(vals)
    np.testing.assert_array_equal(ours, ref)


# ---------------------------------------------------------------- pool


def test_pool_of_identical_keys_is_the_key():
    k = rand_bf16((1, 32))
    kk = np.repeat(k, 4, axis=0)
    np.testing.assert_array_equal(oracle.pool(kk), k)


def test_pool_groups_aligned_blocks_and_drops_tail():
    # token i carries value i: pool p must be the mean of 4p..4p+3 = 4p+1.5,
    # and the 2 trailing tokens of S=42 form no pool.
    S = 42
    k = bf16_bits(np.arange(S, dtype=np.float32)[:, None] * np.ones((1, 3)))
    kp = bits_to_f64(oracle.pool(k))
    assert kp.shape == (S // 4, 3)
    np.testing.assert_array_equal(kp[:, 0], 4 * np.arange(S // 4) + 1.5)


def test_pool_exact_mean_reduces_to_numpy():
    # multiples of 2^-6 below 2: every fp32 partial sum is exact, so the
    # pooled key is the exact mean rounded once to bf16.
    S, D = 64, 48
    m = RNG.integers(-120, 120, size=(S, D)).astype(np.float64) / 64.0
    k = bf16_bits(m)
    assert np.array_equal(bits_to_f64(k), m)
    ref = bf16_bits(m.reshape(S // 4, 4, D).mean(axis=1))
    np.testing.assert_array_equal(oracle.pool(k), ref)


def test_pool_rounding_rule_golden():
    # tests/golden/pool_rounding.txt: pairwise fp32 sum order is observable.
    rows = [l.split() for l in open(os.path.join(GOLDEN, "pool_rounding.txt"))
            if l.strip() and not l.startswith("#")]
    for r in rows:
        keys = np.array([float.fromhex(x) for x in r[:4]], np.float64)
        want = float.fromhex(r[4])
        k = bf16_bits(keys[:, None])
        assert np.array_equal(bits_to_f64(k)[:, 0], keys)
        got = bits_to_f64(oracle.pool(k))[0, 0]
        assert got == want, (r, got)


# --------------------------------------------------------- gated pool


def test_gated_pool_with_equal_gates_is_the_mean_pool():
    # a softmax of equal scores weighs every key 1/4: the mean pooling
    S, D = 64, 48
    m = RNG.integers(-120, 120, size=(S, D)).astype(np.float64) / 64.0
    k = bf16_bits(m)
    for g in (np.zeros(S), np.full(S, -7.25), np.repeat(RNG.standard_normal(S // 4), 4)):
        np.testing.assert_array_equal(oracle.pool_gated(k, g.astype(np.float32)),
                                      oracle.pool(k))


def test_gated_pool_with_one_dominant_gate_is_that_key():
    # exp(-80) relative weight: the other three keys vanish below bf16's
    # resolution, so the pool is the dominant token's key exactly
    S, D = 32, 16
    k = rand_bf16((S, D))
    win = RNG.integers(0, 4, size=S // 4)
    g = np.zeros(S, np.float32)
    g[4 * np.arange(S // 4) + win] = 80.0
    got = oracle.pool_gated(k, g)
    np.testing.assert_array_equal(got, k[4 * np.arange(S // 4) + win])


def test_gated_pool_softmax_weights_closed_form():
    # gates (0, ln 3, 0, 0) on one-hot keys: weights 1/6, 1/2, 1/6, 1/6
    k = bf16_bits(np.eye(4))
    g = np.array([0.0, math.log(3.0), 0.0, 0.0], np.float32)
    got = bits_to_f64(oracle.pool_gated(k, g))[0]
    want = bits_to_f64(bf16_bits(np.array([1 / 6, 1 / 2, 1 / 6, 1 / 6])))
    np.testing.assert_array_equal(got, want)


def test_gated_pool_invariances():
    # adding a constant to a pool's gates, or permuting its four tokens
    # (keys with their gates), leaves the pool unchanged
    S, D = 128, 32
    k = rand_bf16((S, D), std=0.3)
    g = RNG.standard_normal(S).astype(np.float32)
    base = oracle.pool_gated(k, g)
    shift = np.repeat(RNG.integers(-5, 5, size=S // 4).astype(np.float32), 4)
    np.testing.assert_array_equal(oracle.pool_gated(k, g + shift), base)
    perm = np.concatenate([4 * p + RNG.permutation(4) for p in range(S // 4)])
    diff = bits_to_f64(oracle.pool_gated(k[perm], g[perm])) - bits_to_f64(base)
    # the fp64 sum order changes; after bf16 rounding at most a rare ulp
    assert np.mean(diff == 0) > 0.99
    assert np.all(np.abs(diff) <= 2.0 ** -7 * np.abs(bits_to_f64(base)) + 1e-30)


# ------------------------------------------------------------- indexer


def _indexer_case(S, H, D, seed=0):
    rng = np.random.default_rng(seed)
    q = rand_bf16((S, H, D), 1 / math.sqrt(D), rng)
    k = rand_bf16((S, D), 1 / math.sqrt(D), rng)
    w = rng.random((S, H)).astype(np.float32) + 0.05
    return q, k, w


def test_indexer_single_head_unit_weight_is_relu_matmul():
    S, D = 64, 64
    q, k, _ = _indexer_case(S, 1, D, 1)
    w = np.ones((S, 1), np.float32)
    kp = oracle.pool(k)
    got = oracle.index_scores(q, kp, w)
    ref = np.maximum(bits_to_f64(q[:, 0, :]) @ bits_to_f64(kp).T, 0.0)
    nf = (np.arange(S) + 1) // 4
    for t in range(S):
        np.testing.assert_allclose(got[t, :nf[t]], ref[t, :nf[t]], rtol=1e-12,
                                   atol=1e-15)


def test_indexer_relu_is_per_head():
    # heads 0 and 1 carry q and -q with unit weights: ReLU(x) + ReLU(-x) =
    # |x|.  A ReLU applied after the head sum would give 0 instead.
    S, D = 48, 32
    q1, k, _ = _indexer_case(S, 1, D, 2)
    q = np.concatenate([q1, q1 ^ np.uint16(0x8000)], axis=1)
    w = np.ones((S, 2), np.float32)
    kp = oracle.pool(k)
    got = oracle.index_scores(q, kp, w)
    ref = np.abs(bits_to_f64(q1[:, 0, :]) @ bits_to_f64(kp).T)
    for t in range(S):
        nf = (t + 1) // 4
        np.testing.assert_allclose(got[t, :nf], ref[t, :nf], rtol=1e-12,
                                   atol=1e-15)


def test_indexer_linear_in_weights_and_head_permutation():
    S, H, D = 40, 4, 32
    q, k, w = _indexer_case(S, H, D, 3)
    kp = oracle.pool(k)
    w2 = (np.random.default_rng(9).random((S, H)) - 0.5).astype(np.float32)
    a = oracle.index_scores(q, kp, w)
    b = oracle.index_scores(q, kp, w2)
    c = oracle.index_scores(q, kp, (w.astype(np.float64) + w2).astype(np.float32))
    ok = np.isfinite(a)
    # w + w2 rounds to fp32; compare with a tolerance on that rounding.
    np.testing.assert_allclose(c[ok], (a + b)[ok], rtol=1e-6, atol=1e-7)
    perm = np.array([2, 0, 3, 1])
    d = oracle.index_scores(q[:, perm, :], kp, w[:, perm])
    np.testing.assert_allclose(d[ok], a[ok], rtol=1e-12, atol=1e-15)
    neg = oracle.index_scores(q, kp, -w)
    np.testing.assert_array_equal(neg[ok], -a[ok])
    assert (a[ok] >= 0).all()


def test_indexer_scores_only_complete_earlier_pools():
    S = 23
    q, k, w = _indexer_case(S, 2, 16, 4)
    got = oracle.index_scores(q, oracle.pool(k), w)
    for t in range(S):
        for p in range(S // 4):
            complete_and_earlier = all(4 * p + j <= t for j in range(4))
            assert np.isfinite(got[t, p]) == complete_and_earlier, (t, p)


def test_indexer_rows_are_independent_of_chunking():
    S = 64
    q, k, w = _indexer_case(S, 4, 32, 5)
    kp = oracle.pool(k)
    full = oracle.index_scores(q, kp, w)
    for C in (1, 7, 16, 64):
        parts = []
        for r0 in range(0, S, C):
            r = np.arange(r0, min(S, r0 + C))
            parts.append(oracle.index_scores(q[r], kp, w[r], r, S))
        np.testing.assert_array_equal(np.concatenate(parts), full)


# --------------------------------------------------------------- top-k


def _brute_topk(row: np.ndarray, n: int, K: int):
    """All K-subsets of the first n entries: maximal sum, then the
    lexicographically smallest sorted index tuple (integer scores: exact)."""
    take = min(K, n)
    best, best_set = None, None
    for comb in itertools.combinations(range(n), take):
        s = int(sum(row[list(comb)]))
        if best is None or s > best or (s == best and comb < best_set):
            best, best_set = s, comb
    out = list(best_set) + [-1] * (K - take)
    return np.array(out, np.int32)


@pytest.mark.parametrize("K", [1, 2, 3, 5, 8])
def test_topk_matches_exhaustive_enumeration(K):
    rng = np.random.default_rng(K)
    S = 64  # 16 pools
    rows = np.arange(S, dtype=np.int64)
    scores = rng.integers(-3, 4, size=(S, S // 4)).astype(np.float64)
    got = oracle.topk(scores, rows, K)
    for t in range(S):
        n = (t + 1) // 4
        np.testing.assert_array_equal(got[t], _brute_topk(scores[t], n, K))


def test_topk_matches_numpy_stable_sort_fp32():
    rng = np.random.default_rng(7)
    S, K = 2048, 64
    P = S // 4
    rows = np.arange(S, dtype=np.int64)
    scores = rng.standard_normal((S, P)).astype(np.float32)
    scores[:, ::7] = scores[:, :1]  # plenty of exact ties
    got = oracle.topk(scores, rows, K)
    for t in range(0, S, 13):
        n = (t + 1) // 4
        order = np.argsort(-scores[t, :n].astype(np.float64), kind="stable")
        ref = np.sort(order[:K])
        ref = np.concatenate([ref, -np.ones(K - ref.size, np.int64)])
        np.testing.assert_array_equal(got[t], ref)


def test_topk_crafted_rows():
    K = 4
    rows = np.array([39, 39, 39, 39, 39, 11], np.int64)  # n_full 10, 10.., 3
    big = np.float32(1e30)
    sc = np.zeros((6, 12), np.float32)
    sc[0, :] = 0.5                                   # all equal
    sc[1, :10] = np.arange(10, 0, -1)                # strictly decreasing
    sc[2, :10] = [0.0, -0.0, -1, 0.0, -0.0, 2, -0.0, -3, 0.0, -0.0]
    sc[3, :10] = -np.arange(10)                      # increasing penalty
    sc[3, 10:] = big                                 # masked tail: ignored
    sc[4, :10] = [1, 1, 1, 2, 2, 2, 2, 2, 1, 1]
    sc[5, :] = big                                   # row with 3 pools
    got = oracle.topk(sc, rows, K)
    np.testing.assert_array_equal(got[0], [0, 1, 2, 3])
    np.testing.assert_array_equal(got[1], [0, 1, 2, 3])
    np.testing.assert_array_equal(got[2], [0, 1, 3, 5])  # +-0 tie, lower idx
    np.testing.assert_array_equal(got[3], [0, 1, 2, 3])
    np.testing.assert_array_equal(got[4], [3, 4, 5, 6])
    np.testing.assert_array_equal(got[5], [0, 1, 2, -1])


def test_topk_invariants_random():
    rng = np.random.default_rng(11)
    S, K = 4096, 100
    rows = np.arange(0, S, 3, dtype=np.int64)
    sc = rng.standard_normal((rows.size, S // 4))
    got = oracle.topk(sc, rows, K)
    for i, t in enumerate(rows):
        n = (t + 1) // 4
        sel = got[i][got[i] >= 0]
        assert sel.size == min(K, n)
        assert (np.diff(sel) > 0).all()
        assert (sel < n).all()
        if sel.size and n > sel.size:
            rest = np.setdiff1d(np.arange(n), sel)
            assert sc[i, sel].min() >= sc[i, rest].max()
        assert (got[i][sel.size:] == -1).all()


# -------------------------------------------------------------- key set


def test_key_set_full_budget_2051_is_causal_prefix():
    K_p = 8
    for t in range(40):
        n = (t + 1) // 4
        idx = np.array(list(range(min(n, K_p))) + [-1] * (K_p - min(n, K_p)),
                       np.int32)
        ks = oracle.key_set(t, K_p, 3, idx)
        if n <= K_p:
            np.testing.assert_array_equal(ks, np.arange(t + 1))


def test_key_set_2048_is_pool_tokens_only():
    K_p = 4
    idx = np.array([0, 2, 5, -1], np.int32)
    np.testing.assert_array_equal(
        oracle.key_set(30, K_p, 0, idx),
        [0, 1, 2, 3, 8, 9, 10, 11, 20, 21, 22, 23])
    # the 3 locals 21..23 are already inside pool 5: counted once
    np.testing.assert_array_equal(oracle.key_set(23, K_p, 3, idx),
                                  [0, 1, 2, 3, 8, 9, 10, 11, 20, 21, 22, 23])
    np.testing.assert_array_equal(oracle.key_set(26, K_p, 3, idx),
                                  [0, 1, 2, 3, 8, 9, 10, 11, 20, 21, 22, 23,
                                   24, 25, 26])
    assert oracle.key_set(2, K_p, 0, np.full(K_p, -1, np.int32)).size == 0
    np.testing.assert_array_equal(
        oracle.key_set(1, K_p, 3, np.full(K_p, -1, np.int32)), [0, 1])


# ---------------------------------------------------------- attention


def _attn_case(S, H, d, seed):
    rng = np.random.default_rng(seed)
    q = bf16_bits(rng.standard_normal((S, H, d)) * 2.0 / math.sqrt(d))
    k = bf16_bits(rng.standard_normal((S, d)) / math.sqrt(d))
    v = bf16_bits(rng.standard_normal((S, d)))
    return q, k, v


def _full_budget_idx(S, K_p):
    idx = np.full((S, K_p), -1, np.int32)
    for t in range(S):
        n = (t + 1) // 4
        assert n <= K_p
        idx[t, :n] = np.arange(n)
    return idx


def _sdpa(q, k, v, mask, scale):
    """torch SDPA in fp64 with a boolean [S,S] mask -> (O [S,H,d_v], lse)."""
    Q = torch.from_numpy(bits_to_f64(q)).permute(1, 0, 2)       # [H,S,d]
    K = torch.from_numpy(bits_to_f64(k))[None].expand(Q.shape[0], -1, -1)
    V = torch.from_numpy(bits_to_f64(v))[None].expand(Q.shape[0], -1, -1)
    m = torch.from_numpy(mask.astype(bool))
    O = F.scaled_dot_product_attention(Q, K, V, attn_mask=m, scale=scale)
    s = (Q @ K.transpose(-1, -2)) * scale
    lse = torch.logsumexp(s.masked_fill(~m, -math.inf), dim=-1)
    return O.permute(1, 0, 2).numpy(), lse.T.numpy()


def test_attn_full_budget_with_locals_is_dense_causal():
    S, H, d, K_p = 40, 3, 16, 16
    q, k, v = _attn_case(S, H, d, 21)
    scale = 1 / math.sqrt(d)
    o, lse = oracle.attn_fwd(q, k, v, _full_budget_idx(S, K_p), K_p, 3, scale)
    causal = np.tril(np.ones((S, S), np.uint8))
    O, L = _sdpa(q, k, v, causal, scale)
    np.testing.assert_allclose(o, O, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, L, rtol=1e-12, atol=1e-12)


def test_attn_full_budget_without_locals_is_pool_granular_causal():
    S, H, d, K_p = 37, 2, 16, 16
    q, k, v = _attn_case(S, H, d, 22)
    scale = 0.3
    o, lse = oracle.attn_fwd(q, k, v, _full_budget_idx(S, K_p), K_p, 0, scale)
    t = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    mask = (j < 4 * ((t + 1) // 4)).astype(np.uint8)
    live = mask.any(axis=1)
    O, L = _sdpa(q, k, v, np.where(live[:, None], mask, 1), scale)
    np.testing.assert_allclose(o[live], O[live], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse[live], L[live], rtol=1e-12, atol=1e-12)
    assert (o[~live] == 0).all() and np.isneginf(lse[~live]).all()


@pytest.mark.parametrize("n_loc", [0, 3])
def test_attn_random_selection_matches_sdpa_and_dense(n_loc):
    S, H, d, K_p = 64, 2, 16, 5
    q, k, v = _attn_case(S, H, d, 23 + n_loc)
    rng = np.random.default_rng(5)
    idx = np.full((S, K_p), -1, np.int32)
    mask = np.zeros((S, S), np.uint8)
    for t in range(S):
        n = (t + 1) // 4
        sel = np.sort(rng.choice(n, size=min(n, K_p), replace=False))
        idx[t, :sel.size] = sel
        for p in sel:                       # mask from the definition
            mask[t, 4 * p:4 * p + 4] = 1
        for s in range(max(0, t - n_loc + 1), t + 1):
            mask[t, s] = 1
    scale = 1 / math.sqrt(d)
    o, lse = oracle.attn_fwd(q, k, v, idx, K_p, n_loc, scale)
    od, lsed = oracle.dense_masked_attn(q, k, v, mask, scale)
    live = mask.any(axis=1)
    O, L = _sdpa(q, k, v, np.where(live[:, None], mask, 1), scale)
    np.testing.assert_allclose(o[live], O[live], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse[live], L[live], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o, od, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(np.isneginf(lse), ~live[:, None].repeat(H, 1))


def test_attn_zero_query_gives_mean_of_values():
    S, H, d, K_p = 48, 2, 8, 3
    _, k, v = _attn_case(S, H, d, 30)
    q = np.zeros((S, H, d), np.uint16)
    rng = np.random.default_rng(3)
    idx = np.full((S, K_p), -1, np.int32)
    for t in range(S):
        n = (t + 1) // 4
        sel = np.sort(rng.choice(n, size=min(n, K_p), replace=False))
        idx[t, :sel.size] = sel
    o, lse = oracle.attn_fwd(q, k, v, idx, K_p, 3, 1.0)
    vv = bits_to_f64(v)
    for t in range(S):
        toks = sorted({4 * p + j for p in idx[t] if p >= 0 for j in range(4)}
                      | {s for s in (t - 2, t - 1, t) if s >= 0})
        np.testing.assert_allclose(o[t], np.broadcast_to(vv[toks].mean(0),
                                                         (H, d)), rtol=1e-12,
                                   atol=1e-14)
        np.testing.assert_allclose(lse[t], math.log(len(toks)), rtol=1e-13)


# ------------------------------------------------------------ backward


def _sdpa_grads(q, k, v, dO, mask, scale):
    Q = torch.from_numpy(bits_to_f64(q)).permute(1, 0, 2).requires_grad_()
    Kt = torch.from_numpy(bits_to_f64(k)).requires_grad_()
    Vt = torch.from_numpy(bits_to_f64(v)).requires_grad_()
    H = Q.shape[0]
    m = torch.from_numpy(mask.astype(bool))
    O = F.scaled_dot_product_attention(Q, Kt[None].expand(H, -1, -1),
                                       Vt[None].expand(H, -1, -1),
                                       attn_mask=m, scale=scale)
    G = torch.from_numpy(bits_to_f64(dO)).permute(1, 0, 2)
    (O * G).sum().backward()
    return (Q.grad.permute(1, 0, 2).numpy(), Kt.grad.numpy(), Vt.grad.numpy())


@pytest.mark.parametrize("n_loc", [0, 3])
def test_bwd_matches_torch_autograd(n_loc):
    S, H, d, K_p = 48, 3, 16, 4
    q, k, v = _attn_case(S, H, d, 40 + n_loc)
    rng = np.random.default_rng(8 + n_loc)
    dO = bf16_bits(rng.standard_normal((S, H, d)))
    idx = np.full((S, K_p), -1, np.int32)
    mask = np.zeros((S, S), np.uint8)
    for t in range(S):
        n = (t + 1) // 4
        sel = np.sort(rng.choice(n, size=min(n, K_p), replace=False))
        idx[t, :sel.size] = sel
        for p in sel:
            mask[t, 4 * p:4 * p + 4] = 1
        for s in range(max(0, t - n_loc + 1), t + 1):
            mask[t, s] = 1
    live = mask.any(axis=1)
    scale = 1 / math.sqrt(d)
    rows = np.arange(S)
    dq, dk, dv = oracle.attn_bwd(q, k, v, dO, idx, K_p, n_loc, scale, rows)
    # dead rows contribute nothing: give SDPA a harmless mask and zero dO
    dO_l = np.where(live[:, None, None], dO, np.uint16(0))
    rq, rk, rv = _sdpa_grads(q, k, v, dO_l, np.where(live[:, None], mask, 1),
                             scale)
    np.testing.assert_allclose(dq[live], rq[live], rtol=1e-9, atol=1e-12)
    assert (dq[~live] == 0).all()
    np.testing.assert_allclose(dk, rk, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(dv, rv, rtol=1e-9, atol=1e-12)


def test_bwd_with_one_tensor_as_keys_and_values_matches_autograd():
    # K = V = c (an MLA-style shared latent): autograd through SDPA with the
    # same leaf as K and V returns dK + dV for c; the oracle's dk + dv must
    # equal it (and its forward is the same as with v = k)
    S, H, d, K_p = 44, 4, 16, 4
    q, c, _ = _attn_case(S, H, d, 61)
    rng = np.random.default_rng(61)
    dO = bf16_bits(rng.standard_normal((S, H, d)))
    idx = np.full((S, K_p), -1, np.int32)
    mask = np.zeros((S, S), np.uint8)
    for t in range(S):
        n = (t + 1) // 4
        sel = np.sort(rng.choice(n, size=min(n, K_p), replace=False))
        idx[t, :sel.size] = sel
        for p in sel:
            mask[t, 4 * p:4 * p + 4] = 1
        for s_ in range(max(0, t - 2), t + 1):
            mask[t, s_] = 1
    scale = 1 / math.sqrt(d)
    rows = np.arange(S)
    dq, dk, dv = oracle.attn_bwd(q, c, c, dO, idx, K_p, 3, scale, rows)
    Q = torch.from_numpy(bits_to_f64(q)).permute(1, 0, 2).requires_grad_()
    Ct = torch.from_numpy(bits_to_f64(c)).requires_grad_()
    Ce = Ct[None].expand(H, -1, -1)
    O = F.scaled_dot_product_attention(Q, Ce, Ce, attn_mask=torch.from_numpy(
        mask.astype(bool)), scale=scale)
    (O * torch.from_numpy(bits_to_f64(dO)).permute(1, 0, 2)).sum().backward()
    np.testing.assert_allclose(dq, Q.grad.permute(1, 0, 2).numpy(), rtol=1e-9,
                               atol=1e-12)
    np.testing.assert_allclose(dk + dv, Ct.grad.numpy(), rtol=1e-9, atol=1e-12)


def test_bwd_row_subset_equals_zeroed_upstream_gradient():
    # the sampled-row form (dO zero outside the listed rows) used at large S
    S, H, d, K_p = 40, 2, 8, 3
    q, k, v = _attn_case(S, H, d, 50)
    rng = np.random.default_rng(50)
    dO = bf16_bits(rng.standard_normal((S, H, d)))
    idx = np.full((S, K_p), -1, np.int32)
    for t in range(S):
        n = (t + 1) // 4
        sel = np.sort(rng.choice(n, size=min(n, K_p), replace=False))
        idx[t, :sel.size] = sel
    rows = np.array([3, 17, 18, 39])
    dq_r, dk_r, dv_r = oracle.attn_bwd(q[rows], k, v, dO[rows], idx, K_p, 3,
                                       0.5, rows)
    dOz = np.zeros_like(dO)
    dOz[rows] = dO[rows]
    dq_f, dk_f, dv_f = oracle.attn_bwd(q, k, v, dOz, idx, K_p, 3, 0.5)
    np.testing.assert_array_equal(dq_r, dq_f[rows])
    np.testing.assert_allclose(dk_r, dk_f, rtol=0, atol=0)
    np.testing.assert_allclose(dv_r, dv_f, rtol=0, atol=0)
    # compact key addressing returns the same rows
    keys = np.array([0, 5, 9, 17, 30])
    _, dk_c, dv_c = oracle.attn_bwd(q[rows], k, v, dO[rows], idx, K_p, 3, 0.5,
                                    rows, keys)
    np.testing.assert_array_equal(dk_c, dk_f[keys])
    np.testing.assert_array_equal(dv_c, dv_f[keys])
    o_r, l_r = oracle.attn_fwd(q[rows], k, v, idx, K_p, 3, 0.5, rows)
    o_f, l_f = oracle.attn_fwd(q, k, v, idx, K_p, 3, 0.5)
    np.testing.assert_array_equal(o_r, o_f[rows])
    np.testing.assert_array_equal(l_r, l_f[rows])


def test_bwd_scatter_identity_and_finite_difference():
    # sum_t <dQ_t, q_t> == sum_j <dK_j, k_j>: both equal
    # scale * sum dS * (q . k); checks the scattered dK against row-local dQ.
    S, H, d, K_p = 32, 2, 8, 3
    rng = np.random.default_rng(60)
    # values on a 2^-10 grid below 1/4 so q +- 2^-10 stays exact in bf16
    q = bf16_bits(rng.integers(-200, 200, (S, H, d)) / 1024.0)
    k = bf16_bits(rng.integers(-200, 200, (S, d)) / 1024.0)
    v = bf16_bits(rng.standard_normal((S, d)))
    dO = bf16_bits(rng.standard_normal((S, H, d)))
    idx = np.full((S, K_p), -1, np.int32)
    for t in range(S):
        n = (t + 1) // 4
        sel = np.sort(rng.choice(n, size=min(n, K_p), replace=False))
        idx[t, :sel.size] = sel
    scale = 3.0
    dq, dk, dv = oracle.attn_bwd(q, k, v, dO, idx, K_p, 3, scale)
    lhs = np.sum(dq * bits_to_f64(q))
    rhs = np.sum(dk * bits_to_f64(k))
    np.testing.assert_allclose(lhs, rhs, rtol=1e-10)

    def loss(qb):
        o, _ = oracle.attn_fwd(qb, k, v, idx, K_p, 3, scale)
        return np.sum(o * bits_to_f64(dO))

    eps = 1.0 / 1024.0
    for (t, h, c) in [(5, 0, 1), (20, 1, 7), (31, 0, 3)]:
        qp = q.copy()
        qm = q.copy()
        qp[t, h, c] = bf16_bits([float(bits_to_f64(q[t, h, c])[0]) + eps])[0]
        qm[t, h, c] = bf16_bits([float(bits_to_f64(q[t, h, c])[0]) - eps])[0]
        fd = (loss(qp) - loss(qm)) / (2 * eps)
        np.testing.assert_allclose(fd, dq[t, h, c], rtol=2e-3, atol=1e-6)

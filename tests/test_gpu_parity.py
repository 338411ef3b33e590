"""GPU parity: the CUDA library (called through its C ABI) against the fp64
CPU oracle on the same seeded inputs."""
import math

import numpy as np
import pytest
import torch

import long_context_sparse_gb300 as dsa
import oracle
from long_context_sparse_gb300 import synth
from tests.helpers import (abs_bits, assert_close, bits, check_index_rows, f64,
                           oracle_attn_bwd, oracle_attn_fwd, tol)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _cfg(wl, **over):
    return dsa.config_for(wl, **over)


def _status_ok(ws):
    st = dsa.get_device_status(ws)
    assert st == 0, dsa.STATUS_NAMES.get(st, st)


# ------------------------------------------------------------------ pool


@pytest.mark.parametrize("S,D", [(4, 64), (7, 128), (1024, 64), (16387, 128)])
def test_pool_bit_exact(S, D):
    wl = synth.scaled(synth.WORKLOADS["glm_s16k"], S, D_I=D)
    _, k_idx, _ = synth.indexer_inputs(wl, 1, "cpu")
    got = dsa.pool_keys(_cfg(wl), k_idx.to(DEV))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(got), oracle.pool(bits(k_idx)))


@pytest.mark.parametrize("S,D", [(4, 64), (1024, 128), (16387, 128)])
def test_pool_gated_matches_oracle(S, D):
    """fp32 softmax weights on the GPU vs the fp64 definition: equal up to
    one bf16 ulp (different exp implementations), and bit-exactly the mean
    pool when the gates of a pool are equal."""
    wl = synth.scaled(synth.WORKLOADS["glm_s16k"], S, D_I=D)
    cfg = _cfg(wl)
    _, k_idx, _ = synth.indexer_inputs(wl, 1, "cpu")
    gate = synth.gate_inputs(wl, 1, "cpu")
    got = dsa.pool_keys_gated(cfg, k_idx.to(DEV), gate.to(DEV))
    torch.cuda.synchronize()
    g = oracle.bf16_to_f32(bits(got)).astype(np.float64)
    r = oracle.bf16_to_f32(oracle.pool_gated(bits(k_idx), gate.numpy())).astype(np.float64)
    # one bf16 ulp of the result, plus the fp32 weights' and sums' error,
    # which scales with sum_j w_j |k_j| (a cancelling sum can be tiny)
    mag = oracle.bf16_to_f32(oracle.pool_gated(abs_bits(bits(k_idx)),
                                                gate.numpy())).astype(np.float64)
    assert np.all(np.abs(g - r) <= 2.0 ** -7 * np.abs(r) + 2.0 ** -18 * mag + 1e-30)
    assert np.mean(g == r) > 0.99
    flat = torch.repeat_interleave(gate[::4].contiguous(), 4)[:S].contiguous()
    same = dsa.pool_keys_gated(cfg, k_idx.to(DEV), flat.to(DEV))
    mean = dsa.pool_keys(cfg, k_idx.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(same, mean)


# ----------------------------------------------------------------- top-k


def _craft_scores(rows, ld, seed):
    g = np.random.default_rng(seed)
    s = g.standard_normal((rows, ld)).astype(np.float32)
    s[:, ::5] = s[:, 1:2]                      # many exact ties
    s[0::3, ::2] = 0.0
    s[0::3, 1::4] = -0.0                       # +-0 ties
    s[1::7, :] = 1.5                           # whole row equal
    s[2::11, :] = np.abs(s[2::11, :])          # non-negative (like ReLU sums)
    return s


@pytest.mark.parametrize("row0,rows,ld,K", [
    (0, 300, 80, 8), (0, 2048, 512, 64), (16000, 384, 4096, 512),
    (131000, 64, 32768, 512), (400000, 4, 100000, 512), (37, 5, 16, 1),
    (2000, 17, 600, 2048)])
def test_topk_bit_exact_on_shared_scores(row0, rows, ld, K):
    wl = synth.scaled(synth.WORKLOADS["glm_s16k"], max(row0 + rows, 4 * ld),
                      K_p=K)
    cfg = _cfg(wl)
    s = _craft_scores(rows, ld, row0 + K)
    st = torch.from_numpy(s).to(DEV)
    ws = dsa.workspace(cfg, dsa.WS_STATUS, DEV)
    got = dsa.topk_from_scores(cfg, st, row0, ws=ws).cpu().numpy()
    _status_ok(ws)
    ref = oracle.topk(s, np.arange(row0, row0 + rows), K)
    np.testing.assert_array_equal(got, ref)


def _radix_edge_rows(ld, K, seed):
    """Rows whose keys around rank K sit in radix bins of every occupancy:
    keys spread over 40 octaves (mostly alone in their bin, so a bin is
    taken whole after one or two digits), a cluster of distinct keys
    2^-12 apart inside one first-digit bin (settled by a later digit), a
    run of exact ties across rank K (no bin is taken whole: the ties rule),
    and keys one ulp apart (resolved by the last digit)."""
    g = np.random.default_rng(seed)
    base = g.uniform(0.0, 1.0, ld).astype(np.float32)
    rows = []
    a = base.copy()
    pos = g.choice(ld, K + 64, replace=False)
    a[pos] = np.exp2(g.uniform(-20.0, 20.0, K + 64)).astype(np.float32) + np.float32(1.0)
    rows.append(a)
    b = base.copy()
    pos = g.choice(ld, K + 64, replace=False)
    b[pos] = np.float32(16.0) + np.arange(K + 64, dtype=np.float32) * np.float32(2.0 ** -12)
    rows.append(b)
    c = base.copy()
    pos = g.choice(ld, K + 40, replace=False)
    c[pos[:K - 20]] = np.float32(32.0) + g.uniform(0.0, 1.0, K - 20).astype(np.float32)
    c[pos[K - 20:]] = np.float32(20.0)                 # 60 equal keys across rank K
    rows.append(c)
    d = base.copy()
    pos = g.choice(ld, K + 16, replace=False)
    ulp = np.float32(np.nextafter(np.float32(24.0), np.float32(25.0)) - np.float32(24.0))
    d[pos] = np.float32(24.0) + np.arange(K + 16, dtype=np.float32) * ulp
    rows.append(d)
    return np.stack(rows).astype(np.float32)


@pytest.mark.parametrize("ld,K", [(8192, 512), (4000, 64), (32768, 512), (3000, 2048)])
def test_topk_bit_exact_where_the_radix_select_stops(ld, K):
    """The exact selection stops when every key of the chosen bin ranks
    among the K largest; rows built to stop after the first digit, after
    the second, or never (ties, last-bit differences) must still give the
    oracle's selection bit for bit, on the cut path (rows longer than the
    candidate buffer) and on the whole-row path."""
    row0 = 4 * ld + 100
    wl = synth.scaled(synth.WORKLOADS["glm_s16k"], row0 + 8, K_p=K)
    cfg = _cfg(wl)
    s = _radix_edge_rows(ld, K, ld + K)
    rows = np.arange(row0, row0 + s.shape[0])
    ws = dsa.workspace(cfg, dsa.WS_STATUS, DEV)
    got = dsa.topk_from_scores(cfg, torch.from_numpy(s).to(DEV), row0, ws=ws).cpu().numpy()
    _status_ok(ws)
    np.testing.assert_array_equal(got, oracle.topk(s, rows, K))


# --------------------------------------------------------------- indexer


@pytest.mark.parametrize("name,S,t0,rows", [
    ("tiny_fwd_s1k", 1024, 0, 1024), ("glm_s16k", 4099, 3000, 300),
    ("glm_s16k", 16384, 15000, 256), ("padded2051_s64k", 2600, 1, 700)])
def test_index_scores_match_oracle(name, S, t0, rows):
    wl = synth.scaled(synth.WORKLOADS[name], S)
    cfg = _cfg(wl)
    q_idx, k_idx, w = synth.indexer_inputs(wl, 3, "cpu")
    kp = oracle.pool(bits(k_idx))
    kp_dev = torch.from_numpy(kp.view(np.int16)).view(torch.bfloat16).to(DEV)
    ws = dsa.workspace(cfg, dsa.WS_STATUS, DEV)
    sc = dsa.index_scores(cfg, q_idx.to(DEV), kp_dev, w.to(DEV), t0, rows,
                          ws=ws).cpu().numpy()
    _status_ok(ws)
    r = np.arange(t0, t0 + rows)
    pick = r[:: max(1, rows // 64)]
    ref = oracle.index_scores(bits(q_idx)[pick], kp, w.numpy()[pick], pick, S)
    for i, t in enumerate(pick):
        n = (t + 1) // 4
        got = sc[t - t0, :n].astype(np.float64)
        # bf16 products are exact in fp32; fp32 sums over D_I and H_I
        tol = 1e-5 * np.abs(ref[i, :n]).max(initial=1e-3) + 1e-7
        np.testing.assert_allclose(got, ref[i, :n], rtol=2e-5, atol=tol)


def test_index_scores_independent_of_chunking_bit_exact():
    wl = synth.scaled(synth.WORKLOADS["glm_s16k"], 9000)
    cfg = _cfg(wl)
    q_idx, k_idx, w = (x.to(DEV) for x in synth.indexer_inputs(wl, 5, "cpu"))
    kp = dsa.pool_keys(cfg, k_idx)
    whole = dsa.index_scores(cfg, q_idx, kp, w, 8000, 1000)
    parts = [dsa.index_scores(cfg, q_idx, kp, w, t0, n)
             for t0, n in [(8000, 1), (8001, 255), (8256, 500), (8756, 244)]]
    torch.cuda.synchronize()
    rows = [whole[0:1], whole[1:256], whole[256:756], whole[756:1000]]
    for a, b, t0 in zip(parts, rows, [8000, 8001, 8256, 8756]):
        n = (t0 + a.shape[0]) // 4 - 1          # valid for every row of a
        assert torch.equal(a[:, :n], b[:, :n])


# ------------------------------------------------------ index + top-k


@pytest.mark.parametrize("name,S,nrows", [
    ("tiny_fwd_s1k", 1024, 0), ("glm_s16k", 2051, 0), ("glm_s16k", 16384, 40),
    ("padded2051_s64k", 9000, 40)])
def test_index_topk_matches_oracle(name, S, nrows):
    wl = synth.scaled(synth.WORKLOADS[name], S)
    cfg = _cfg(wl)
    q_idx, k_idx, w = synth.indexer_inputs(wl, 7, "cpu")
    ws = dsa.workspace(cfg, dsa.WS_INDEX, DEV)
    got = dsa.index_scores_topk(cfg, q_idx.to(DEV), k_idx.to(DEV), w.to(DEV),
                                ws=ws).cpu().numpy()
    _status_ok(ws)
    rows = (np.arange(S) if nrows == 0 else
            synth.sample_rows(wl, nrows, 11).numpy())
    ref, sc = oracle.index_topk(bits(q_idx), bits(k_idx), w.numpy(), wl.K_p,
                                rows)
    eq, ex = check_index_rows(got[rows], ref, sc, rows, wl.K_p)
    assert eq + ex == rows.size and eq >= 0.9 * rows.size


def test_index_topk_chunked_equals_unchunked_bit_exact():
    wl = synth.scaled(synth.WORKLOADS["glm_s16k"], 6000)
    q_idx, k_idx, w = (x.to(DEV) for x in synth.indexer_inputs(wl, 9, "cpu"))
    outs = []
    for C in (1, 37, 256, 4096):
        cfg = _cfg(wl, chunk_q=C)
        outs.append(dsa.index_scores_topk(cfg, q_idx, k_idx, w))
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


@pytest.mark.parametrize("ranges", [
    [(0, 6000)], [(1000, 3333), (3333, 3334), (5, 5), (4000, 6000)],
    [(0, 1), (17, 2100), (5999, 6000)]])
def test_index_topk_range_equals_whole_sequence_rows(ranges):
    """Each range's rows equal the whole-sequence call's rows (bit-exact:
    a row's scores do not depend on which rows share its chunk) and the
    oracle's selection of those rows (tie band)."""
    wl = synth.scaled(synth.WORKLOADS["glm_s16k"], 6000)
    cfg = _cfg(wl, chunk_q=256)
    q_idx, k_idx, w = synth.indexer_inputs(wl, 9, "cpu")
    qd, kd, wd = q_idx.to(DEV), k_idx.to(DEV), w.to(DEV)
    whole = dsa.index_scores_topk(cfg, qd, kd, wd)
    ws = dsa.workspace(cfg, dsa.WS_INDEX, DEV)
    for t0, t1 in ranges:
        got = dsa.index_scores_topk_range(cfg, qd[t0:t1].contiguous(), kd,
                                          wd[t0:t1].contiguous(), t0, t1, ws=ws)
        _status_ok(ws)
        assert got.shape == (t1 - t0, wl.K_p)
        assert torch.equal(got, whole[t0:t1])
        if t1 > t0:
            rows = np.unique(np.linspace(t0, t1 - 1, 24).astype(np.int64))
            ref, sc = oracle.index_topk(bits(q_idx), bits(k_idx), w.numpy(),
                                        wl.K_p, rows)
            eq, ex = check_index_rows(got.cpu().numpy()[rows - t0], ref, sc,
                                      rows, wl.K_p)
            assert eq + ex == rows.size


@pytest.mark.parametrize("name,S,t0,t1", [("glm_s16k", 6000, 0, 6000),
                                          ("padded2051_s64k", 9000, 3000, 7777)])
def test_index_topk_gated_matches_oracle(name, S, t0, t1):
    wl = synth.scaled(synth.WORKLOADS[name], S)
    cfg = _cfg(wl)
    q_idx, k_idx, w = synth.indexer_inputs(wl, 3, "cpu")
    gate = synth.gate_inputs(wl, 3, "cpu")
    ws = dsa.workspace(cfg, dsa.WS_INDEX, DEV)
    got = dsa.index_scores_topk_range(cfg, q_idx[t0:t1].contiguous().to(DEV),
                                      k_idx.to(DEV), w[t0:t1].contiguous().to(DEV),
                                      t0, t1, k_gate=gate.to(DEV), ws=ws)
    _status_ok(ws)
    got = got.cpu().numpy()
    rows = np.unique(np.concatenate([
        np.linspace(t0, t1 - 1, 48).astype(np.int64), [t0, t1 - 1]]))
    ref, sc = oracle.index_topk(bits(q_idx), bits(k_idx), w.numpy(), wl.K_p,
                                rows, gate=gate.numpy())
    eq, ex = check_index_rows(got[rows - t0], ref, sc, rows, wl.K_p)
    assert eq + ex == rows.size and eq >= 0.9 * rows.size


@pytest.mark.parametrize("S,over,t0,t1", [
    (6000, {}, 0, 6000),                          # 32 x 128, K_p = 512
    (4103, dict(H_I=64), 5, 4103),               # 4 queries per tile, ragged ends
    (3000, dict(D_I=64, K_p=100), 0, 3000),
    (2500, dict(K_p=16), 1, 2),                   # one row
    (9000, dict(K_p=512), 7000, 9000),           # long rows: several compactions
    (9000, dict(K_p=768), 6000, 9000),           # the largest supported K_p
    (20, dict(K_p=8), 0, 20),                     # empty and full-budget rows
])
def test_index_topk_streaming_equals_chunked_bit_exact(S, over, t0, t1):
    """The fused selection sees the same fp32 scores as the chunked path:
    its rows must be bit-identical, and within the tie band of the oracle."""
    wl = synth.scaled(synth.WORKLOADS["glm_s16k"], S, **over)
    cfg = _cfg(wl)
    q_idx, k_idx, w = synth.indexer_inputs(wl, 13, "cpu")
    qd, kd = q_idx[t0:t1].contiguous().to(DEV), k_idx.to(DEV)
    wd = w[t0:t1].contiguous().to(DEV)
    ws = dsa.workspace(cfg, dsa.WS_STREAM, DEV)
    got = dsa.index_topk_streaming(cfg, qd, kd, wd, t0, t1, ws=ws)
    _status_ok(ws)
    ref_gpu = dsa.index_scores_topk_range(cfg, qd, kd, wd, t0, t1)
    torch.cuda.synchronize()
    assert torch.equal(got, ref_gpu)
    rows = np.unique(np.linspace(t0, t1 - 1, 16).astype(np.int64))
    ref, sc = oracle.index_topk(bits(q_idx), bits(k_idx), w.numpy(), wl.K_p, rows)
    eq, ex = check_index_rows(got.cpu().numpy()[rows - t0], ref, sc, rows, wl.K_p)
    assert eq + ex == rows.size


def test_index_topk_streaming_gated_and_unsupported():
    wl = synth.scaled(synth.WORKLOADS["glm_s16k"], 5000)
    cfg = _cfg(wl)
    q_idx, k_idx, w = (x.to(DEV) for x in synth.indexer_inputs(wl, 17, "cpu"))
    gate = synth.gate_inputs(wl, 17, "cpu").to(DEV)
    got = dsa.index_topk_streaming(cfg, q_idx, k_idx, w, k_gate=gate)
    ref = dsa.index_scores_topk_range(cfg, q_idx, k_idx, w, 0, wl.S, k_gate=gate)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    small = synth.scaled(synth.WORKLOADS["tiny_fwd_s1k"], 512)   # H_I = 4
    with pytest.raises(dsa.DsaError) as e:
        qs, ks, ws_ = (x.to(DEV) for x in synth.indexer_inputs(small, 1, "cpu"))
        dsa.index_topk_streaming(_cfg(small), qs, ks, ws_)
    assert e.value.code == 2
    big = synth.scaled(synth.WORKLOADS["glm_s16k"], 4096, K_p=769)  # above the list cap
    with pytest.raises(dsa.DsaError) as e:
        qb, kb, wb = (x.to(DEV) for x in synth.indexer_inputs(big, 1, "cpu"))
        dsa.index_topk_streaming(_cfg(big), qb, kb, wb)
    assert e.value.code == 2


def test_index_topk_full_budget_selects_every_pool():
    wl = synth.scaled(synth.WORKLOADS["tiny_fwd_s1k"], 256, K_p=64)
    cfg = _cfg(wl)
    q_idx, k_idx, w = (x.to(DEV) for x in synth.indexer_inputs(wl, 2, "cpu"))
    got = dsa.index_scores_topk(cfg, q_idx, k_idx, w).cpu().numpy()
    for t in range(256):
        n = (t + 1) // 4
        np.testing.assert_array_equal(got[t, :n], np.arange(n))
        assert (got[t, n:] == -1).all()


# ------------------------------------------------------------ attention


def _attn_case(name, S, seed, scale="pages", **over):
    wl = synth.scaled(synth.WORKLOADS[name], S, **over)
    q, k, v, dO = synth.attention_inputs_scaled(wl, seed, scale, "cpu")
    idx = synth.random_selection(wl, seed, "cpu")
    return wl, q, k, v, dO, idx


# Input scales (synth.ATTN_INPUT_SCALES): "pages" is the workloads' own; at
# "unit" and "peaked" O, dQ, dK and dV are of order one, so every check below
# fails for a kernel that leaves one of them at zero, gets its sign or scale
# wrong, or drops a term (delta, the online-softmax rescale of later tiles).
@pytest.mark.parametrize("name,S,over,scale", [
    ("tiny_fwd_s1k", 1024, {}, "pages"),
    ("tiny_fwd_s1k", 1024, {}, "peaked"),
    ("tiny_fwd_s1k", 77, dict(K_p=5, n_loc=3), "pages"),
    ("tiny_fwd_s1k", 77, dict(K_p=5, n_loc=3), "unit"),
    ("glm_s16k", 3000, {}, "pages"),
    ("glm_s16k", 3000, {}, "peaked"),       # 16 key tiles, sampled rows
    ("glm_s16k", 640, {}, "unit"),          # 64 heads, d = 512, every row
    ("glm_s16k", 640, {}, "peaked"),
    ("glm_s16k", 300, dict(H=80), "pages"),  # two head blocks
    ("glm_s16k", 300, dict(H=80), "unit"),
    ("padded2051_s64k", 2300, {}, "pages"),  # 16 heads, 2051 keys
    ("padded2051_s64k", 2300, {}, "unit"),
    ("padded2051_s64k", 520, {}, "peaked"),
    ("glm_s16k", 13, dict(n_loc=3), "pages"),  # tiny, empty rows
    ("glm_s16k", 13, dict(n_loc=3), "unit"),
])
def test_attn_fwd_bwd_match_oracle(name, S, over, scale):
    wl, q, k, v, dO, idx = _attn_case(name, S, 21, scale, **over)
    cfg = _cfg(wl)
    qd, kd, vd, dOd, idd = (x.to(DEV) for x in (q, k, v, dO, idx))
    wsf = dsa.workspace(cfg, dsa.WS_FWD, DEV)
    o, lse = dsa.sparse_attn_fwd(cfg, qd, kd, vd, idd, ws=wsf)
    _status_ok(wsf)
    rows = np.arange(S) if S <= 700 else synth.sample_rows(wl, 48, 3).numpy()
    qb, kb, vb, dOb, idx_h = bits(q), bits(k), bits(v), bits(dO), idx.numpy()
    ro, rl = oracle_attn_fwd(qb[rows], kb, vb, idx_h, wl.K_p, wl.n_loc, cfg.scale,
                             rows)
    go, gl = f64(o)[rows], f64(lse)[rows]
    fin = np.isfinite(rl)
    assert (go[~fin.any(1)] == 0).all()        # empty key set: O = 0
    om, _ = oracle_attn_fwd(qb[rows], kb, abs_bits(vb), idx_h, wl.K_p, wl.n_loc,
                            cfg.scale, rows)
    assert_close(go, ro, "o", mag=om, **tol(scale))   # om = sum_j P_j |v_j|
    assert_close(gl, rl, "lse")                # -inf rows must match exactly
    if not wl.backward and S > 200:
        return
    wsb = dsa.workspace(cfg, dsa.WS_BWD, DEV)
    dq, dk, dv = dsa.sparse_attn_bwd(cfg, qd, kd, vd, o, lse, dOd, idd, ws=wsb)
    _status_ok(wsb)
    if S <= 700:
        allr = np.arange(S)
        rdq, rdk, rdv = oracle_attn_bwd(qb, kb, vb, dOb, idx_h, wl.K_p, wl.n_loc,
                                        cfg.scale, allr)
        # sum P |dO| bounds the bf16-operand error of dV = P^T dO
        _, _, mdv = oracle_attn_bwd(qb, kb, vb, abs_bits(dOb), idx_h, wl.K_p,
                                    wl.n_loc, cfg.scale, allr)
        assert_close(f64(dq), rdq, "dq", **tol(scale))
        assert_close(f64(dk), rdk, "dk", **tol(scale))
        assert_close(f64(dv), rdv, "dv", mag=mdv, **tol(scale))
    else:
        rdq, _, _ = oracle_attn_bwd(qb[rows], kb, vb, dOb[rows], idx_h, wl.K_p,
                                    wl.n_loc, cfg.scale, rows, np.zeros(1, np.int64))
        assert_close(f64(dq)[rows], rdq, "dq", **tol(scale))


def _check_dk_half(dkv, rdk, rdv, mdv, name, scale):
    """K = V: dkv = dK + dV.  Where dV dominates, a wrong or missing dK half
    hides inside dkv's tolerance; compare dkv - dV_oracle with dK_oracle on
    its own scale.  The bf16 rounding of dkv (2^-9 |dK + dV|) is the floor of
    this comparison, so it is made only at the unit and peaked input scales,
    where |dK| is of the order of |dV|."""
    assert_close(dkv - rdv, rdk, name, mag=np.abs(rdk) + np.abs(mdv), **tol(scale))


@pytest.mark.parametrize("name,S,over,scale", [
    ("glm_s16k", 640, {}, "pages"),                 # 64 heads, d = 512
    ("glm_s16k", 640, {}, "unit"),
    ("padded2051_s64k", 520, {}, "pages"),          # 16 heads, 2051 keys
    ("padded2051_s64k", 520, {}, "peaked"),
    ("tiny_fwd_s1k", 300, dict(K_p=16), "pages"),   # 8 heads, d = 128
    ("tiny_fwd_s1k", 300, dict(K_p=16), "unit"),
    ("glm_s16k", 4096, {}, "pages"),                # sampled rows
    ("glm_s16k", 4096, {}, "unit"),
])
def test_attn_kv_aliased_matches_oracle(name, S, over, scale):
    """K = V = one tensor: forward as with v = k, backward dkv = dK + dV."""
    wl, q, k, _, dO, idx = _attn_case(name, S, 23, scale, **over)
    cfg = _cfg(wl)
    qd, kd, dOd, idd = (x.to(DEV) for x in (q, k, dO, idx))
    wsf = dsa.workspace(cfg, dsa.WS_FWD, DEV)
    o, lse = dsa.sparse_attn_fwd_kv(cfg, qd, kd, idd, ws=wsf)
    _status_ok(wsf)
    o2, lse2 = dsa.sparse_attn_fwd(cfg, qd, kd, kd, idd)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    wsb = dsa.workspace(cfg, dsa.WS_BWD, DEV)
    qb, kb, dOb, idx_h = bits(q), bits(k), bits(dO), idx.numpy()
    if S <= 700:
        dq, dkv = dsa.sparse_attn_bwd_kv(cfg, qd, kd, o, lse, dOd, idd, ws=wsb)
        _status_ok(wsb)
        allr = np.arange(S)
        rdq, rdk, rdv = oracle_attn_bwd(qb, kb, kb, dOb, idx_h, wl.K_p, wl.n_loc,
                                        cfg.scale, allr)
        _, _, mdv = oracle_attn_bwd(qb, kb, kb, abs_bits(dOb), idx_h, wl.K_p,
                                    wl.n_loc, cfg.scale, allr)
        assert_close(f64(dq), rdq, "dq", **tol(scale))
        assert_close(f64(dkv), rdk + rdv, "dkv", mag=np.abs(rdk) + np.abs(mdv),
                     **tol(scale))
        if scale != "pages":
            _check_dk_half(f64(dkv), rdk, rdv, mdv, "dkv - dV", scale)
        return
    rows = synth.sample_rows(wl, 24, 5).numpy()
    rt = torch.from_numpy(rows).to(DEV)
    dOz = torch.zeros_like(dOd)
    dOz[rt] = dOd[rt]
    dq, dkv = dsa.sparse_attn_bwd_kv(cfg, qd, kd, o, lse, dOz, idd, ws=wsb)
    _status_ok(wsb)
    keys = np.array(sorted({int(s_) for t in rows for s_ in
                            oracle.key_set(int(t), wl.K_p, wl.n_loc, idx_h[t])}),
                    np.int64)
    rdq, rdk, rdv = oracle_attn_bwd(qb[rows], kb, kb, dOb[rows], idx_h, wl.K_p,
                                    wl.n_loc, cfg.scale, rows, keys)
    assert_close(f64(dq[rt]), rdq, "dq", **tol(scale))
    kt = torch.from_numpy(keys).to(DEV)
    _, _, mdv = oracle_attn_bwd(qb[rows], kb, kb, abs_bits(dOb[rows]), idx_h, wl.K_p,
                                wl.n_loc, cfg.scale, rows, keys)
    assert_close(f64(dkv[kt]), rdk + rdv, "dkv", mag=np.abs(rdk) + np.abs(mdv),
                 **tol(scale))
    if scale != "pages":
        _check_dk_half(f64(dkv[kt]), rdk, rdv, mdv, "dkv - dV", scale)
    untouched = torch.ones(wl.S, dtype=torch.bool, device=DEV)
    untouched[kt] = False
    assert not dkv[untouched].any()


def _masked_dkdv_check(wl, cfg, q, k, v, dO, idx, o, lse, rows, scale="pages"):
    """dK/dV are not row-local: rerun the GPU backward with dO zeroed outside
    the sampled rows and compare with the oracle's contributions of those
    rows only, on every token they touch."""
    dOz = torch.zeros_like(dO)
    rt = torch.from_numpy(rows).to(dO.device)
    dOz[rt] = dO[rt]
    dq, dk, dv = dsa.sparse_attn_bwd(cfg, q, k, v, o, lse, dOz, idx)
    idx_h = idx.cpu().numpy()
    keys = sorted({int(s) for t in rows
                   for s in oracle.key_set(int(t), wl.K_p, wl.n_loc, idx_h[t])})
    keys = np.array(keys, np.int64)
    rdq, rdk, rdv = oracle.attn_bwd(bits(q[rt]), bits(k), bits(v),
                                    bits(dO[rt]), idx_h, wl.K_p, wl.n_loc,
                                    cfg.scale, rows, keys)
    _, _, mdv = oracle.attn_bwd(bits(q[rt]), bits(k), bits(v),
                                abs_bits(bits(dO[rt])), idx_h, wl.K_p, wl.n_loc,
                                cfg.scale, rows, keys)
    assert_close(f64(dq[rt]), rdq, "dq", **tol(scale))
    kt = torch.from_numpy(keys).to(dO.device)
    assert_close(f64(dk[kt]), rdk, "dk", **tol(scale))
    assert_close(f64(dv[kt]), rdv, "dv", mag=mdv, **tol(scale))
    # tokens nobody in `rows` attends get exactly zero
    untouched = torch.ones(wl.S, dtype=torch.bool, device=dO.device)
    untouched[kt] = False
    assert not dk[untouched].any() and not dv[untouched].any()


@pytest.mark.parametrize("name,S,scale", [
    ("glm_s16k", 16384, "pages"),
    ("glm_s16k", 16384, "unit"),
    ("padded2051_s64k", 16500, "pages"),
    ("padded2051_s64k", 16500, "peaked"),
    ("glm_s16k", 32768, "pages"),             # several waves of queries per CTA
])
def test_attn_large_sampled_rows(name, S, scale):
    wl, q, k, v, dO, idx = _attn_case(name, S, 33, scale)
    cfg = _cfg(wl)
    qd, kd, vd, dOd, idd = (x.to(DEV) for x in (q, k, v, dO, idx))
    o, lse = dsa.sparse_attn_fwd(cfg, qd, kd, vd, idd)
    rows = synth.sample_rows(wl, 12, 5).numpy()
    ro, rl = oracle.attn_fwd(bits(q)[rows], bits(k), bits(v), idx.numpy(),
                             wl.K_p, wl.n_loc, cfg.scale, rows)
    om, _ = oracle.attn_fwd(bits(q)[rows], bits(k), abs_bits(bits(v)), idx.numpy(),
                            wl.K_p, wl.n_loc, cfg.scale, rows)
    assert_close(f64(o)[rows], ro, "o", mag=om, **tol(scale))
    assert_close(f64(lse)[rows], rl, "lse")
    _masked_dkdv_check(wl, cfg, qd, kd, vd, dOd, idd, o, lse, rows[-6:], scale)


def test_bad_index_is_latched_not_read():
    wl, q, k, v, dO, idx = _attn_case("tiny_fwd_s1k", 256, 4)
    cfg = _cfg(wl)
    bad = idx.clone()
    bad[100, 0] = 1000          # pool beyond n_full(100) = 25
    ws = dsa.workspace(cfg, dsa.WS_FWD, DEV)
    dsa.sparse_attn_fwd(cfg, q.to(DEV), k.to(DEV), v.to(DEV), bad.to(DEV),
                        ws=ws)
    assert dsa.get_device_status(ws) == 7
    assert dsa.get_device_status(ws) == 0      # read clears


def test_unsupported_shapes_raise_before_launch():
    wl = synth.scaled(synth.WORKLOADS["glm_s16k"], 64)
    with pytest.raises(dsa.DsaError) as e:
        dsa.workspace(_cfg(wl, d_qk=576, d_v=512), dsa.WS_FWD, DEV)
    assert e.value.code == 2


# ------------------------------------------- query ranges and whole steps


def _close_bf16(got, ref):
    """Equal up to one bf16 rounding: fp32 sums accumulated in another
    order can straddle a rounding boundary."""
    g, r = f64(got), f64(ref)
    scale = np.abs(r).max() if r.size else 0.0
    assert np.all(np.abs(g - r) <= 2.0 ** -7 * np.abs(r) + 2.0 ** -20 * scale)
    assert np.mean(g == r) > 0.9


@pytest.mark.parametrize("name,S,over,cuts", [
    ("glm_s16k", 3000, {}, [0, 1000, 1004, 1004, 2999, 3000]),
    ("tiny_fwd_s1k", 77, dict(K_p=5, n_loc=3), [0, 12, 77]),  # 16-byte rows
    ("glm_s16k", 300, dict(H=80), [0, 150, 300]),     # two head blocks
    ("padded2051_s64k", 1100, {}, [0, 512, 1100]),    # 16 heads, 2051 keys
])
def test_attn_ranges_equal_whole_call(name, S, over, cuts):
    """Forward rows and dq rows of range calls are bit-identical to the
    whole-sequence call's; the fp32 dK/dV contributions of ranges that
    partition the queries add up to the whole call's dK/dV."""
    wl, q, k, v, dO, idx = _attn_case(name, S, 31, **over)
    cfg = _cfg(wl)
    qd, kd, vd, dOd, idd = (x.to(DEV) for x in (q, k, v, dO, idx))
    o, lse = dsa.sparse_attn_fwd(cfg, qd, kd, vd, idd)
    dq, dk, dv = dsa.sparse_attn_bwd(cfg, qd, kd, vd, o, lse, dOd, idd)
    dk_acc = torch.zeros((S, cfg.d_qk), dtype=torch.float32, device=DEV)
    dv_acc = torch.zeros_like(dk_acc)
    wsf = dsa.workspace(cfg, dsa.WS_FWD, DEV)
    wsr = dsa.workspace(cfg, dsa.WS_BWD_ROWS, DEV)
    for a, b in zip(cuts[:-1], cuts[1:]):
        o_r, lse_r = dsa.sparse_attn_fwd_range(cfg, qd[a:b], kd, vd, idd[a:b], a, b,
                                               ws=wsf)
        dq_r = dsa.sparse_attn_bwd_range(cfg, qd[a:b], kd, vd, o_r, lse_r, dOd[a:b],
                                         idd[a:b], a, b, dk_acc, dv_acc, ws=wsr)
        torch.cuda.synchronize()
        assert torch.equal(o_r, o[a:b]) and torch.equal(lse_r, lse[a:b]), (a, b)
        assert torch.equal(dq_r, dq[a:b]), (a, b)
    _status_ok(wsf)
    _status_ok(wsr)
    _close_bf16(dsa.accum_to_bf16(dk_acc), dk)
    _close_bf16(dsa.accum_to_bf16(dv_acc), dv)
    # K = V: one accumulator receives dK + dV
    o2, lse2 = dsa.sparse_attn_fwd_kv(cfg, qd, kd, idd)
    _, dkv = dsa.sparse_attn_bwd_kv(cfg, qd, kd, o2, lse2, dOd, idd)
    acc = torch.zeros_like(dk_acc)
    for a, b in zip(cuts[:-1], cuts[1:]):
        dsa.sparse_attn_bwd_range(cfg, qd[a:b], kd, kd, o2[a:b], lse2[a:b], dOd[a:b],
                                  idd[a:b], a, b, acc, None, ws=wsr)
    _close_bf16(dsa.accum_to_bf16(acc), dkv)


def test_attn_bwd_range_rejects_one_accumulator_for_separate_kv():
    wl, q, k, v, dO, idx = _attn_case("tiny_fwd_s1k", 64, 3)
    cfg = _cfg(wl)
    qd, kd, vd, dOd, idd = (x.to(DEV) for x in (q, k, v, dO, idx))
    o, lse = dsa.sparse_attn_fwd(cfg, qd, kd, vd, idd)
    acc = torch.zeros((64, cfg.d_qk), dtype=torch.float32, device=DEV)
    with pytest.raises(dsa.DsaError) as e:
        dsa.sparse_attn_bwd_range(cfg, qd, kd, vd, o, lse, dOd, idd, 0, 64, acc, None)
    assert e.value.code == 1


def _step_tensors(wl, seed, gated=False, kv=False, backward=True):
    q_idx, k_idx, w = synth.indexer_inputs(wl, seed, "cpu")
    q, k, v, dO = synth.attention_inputs(wl, seed, "cpu")
    x = {"q_idx": q_idx, "k_idx": k_idx, "w": w, "q": q, "k": k}
    if not kv:
        x["v"] = v
    if gated:
        x["k_gate"] = synth.gate_inputs(wl, seed, "cpu")
    if backward:
        x["dO"] = dO
    return x


def _step_outputs(cfg, shapes, like, device):
    out = {}
    for name in ("topk_idx", "o", "lse", "dq", "dk", "dv"):
        if name in shapes:
            shape, dtype = shapes[name]
            out[name] = torch.empty(shape, dtype=dtype, device=device,
                                    pin_memory=device == "cpu")
    return out


@pytest.mark.parametrize("S,gated,kv,backward", [
    (3000, False, False, True),
    (2500, True, False, True),
    (2000, False, True, True),
    (1800, False, False, False),
])
def test_step_equals_separate_calls(S, gated, kv, backward):
    wl = synth.scaled(synth.WORKLOADS["glm_s16k"], S)
    cfg = _cfg(wl)
    x = {n: t.to(DEV) for n, t in _step_tensors(wl, 41, gated, kv, backward).items()}
    shapes = dsa.step_shapes(cfg, kv, backward, gated)
    dev = dict(x, **_step_outputs(cfg, shapes, x, DEV))
    ws = dsa.workspace(cfg, dsa.WS_STEP, DEV)
    dsa.step(cfg, dev, ws=ws)
    _status_ok(ws)
    if gated:
        idx = dsa.index_scores_topk_range(cfg, x["q_idx"], x["k_idx"], x["w"], 0, S,
                                          k_gate=x["k_gate"])
    else:
        idx = dsa.index_scores_topk(cfg, x["q_idx"], x["k_idx"], x["w"])
    v = x["k"] if kv else x["v"]
    o, lse = dsa.sparse_attn_fwd(cfg, x["q"], x["k"], v, idx)
    torch.cuda.synchronize()
    assert torch.equal(dev["topk_idx"], idx)
    assert torch.equal(dev["o"], o) and torch.equal(dev["lse"], lse)
    if not backward:
        return
    if kv:
        dq, dkv = dsa.sparse_attn_bwd_kv(cfg, x["q"], x["k"], o, lse, x["dO"], idx)
        _close_bf16(dev["dk"], dkv)
    else:
        dq, dk, dv = dsa.sparse_attn_bwd(cfg, x["q"], x["k"], v, o, lse, x["dO"], idx)
        _close_bf16(dev["dk"], dk)
        _close_bf16(dev["dv"], dv)
    assert torch.equal(dev["dq"], dq)


def test_host_buffer_is_page_locked_and_serves_the_host_step():
    """dsa.host_buffer: a registered (page-locked) host tensor of the asked
    shape; the host step over such buffers equals the one over cudaHostAlloc
    buffers."""
    wl = synth.scaled(synth.WORKLOADS["glm_s16k"], 2500)
    cfg = _cfg(wl)
    shapes = dsa.step_shapes(cfg, False, True, False)
    inp = _step_tensors(wl, 47)
    res = []
    for alloc in ("pin", "huge"):
        if alloc == "pin":
            host = {n: t.pin_memory() for n, t in inp.items()}
            host.update(_step_outputs(cfg, shapes, host, "cpu"))
        else:
            host = {}
            for n, t in inp.items():
                host[n] = dsa.host_buffer(t.shape, t.dtype)
                host[n].copy_(t)
            for n in ("topk_idx", "o", "lse", "dq", "dk", "dv"):
                shape, dtype = shapes[n]
                host[n] = dsa.host_buffer(shape, dtype)
            assert host["q"].is_pinned() and host["dq"].is_pinned()
            assert host["q"].shape == inp["q"].shape and host["w"].dtype == torch.float32
        dev = {n: torch.empty(shape, dtype=dtype, device=DEV)
               for n, (shape, dtype) in shapes.items()}
        dsa.step_host(cfg, host, dev, 3)
        torch.cuda.synchronize()
        res.append({n: host[n].clone() for n in ("topk_idx", "o", "lse", "dq", "dk", "dv")})
    for n in ("topk_idx", "o", "lse", "dq"):
        assert torch.equal(res[0][n], res[1][n]), n
    for n in ("dk", "dv"):      # fp32 additions in another order
        _close_bf16(res[0][n], res[1][n])


@pytest.mark.parametrize("S,n_chunks,gated,kv,backward", [
    (3000, 1, False, False, True),
    (3000, 3, False, False, True),
    (16384, 8, False, False, True),           # the 16k configuration, 8 ranges
    (2049, 64, True, False, True),            # more ranges than CTAs per range
    (2000, 5, False, True, True),
    (1800, 4, False, False, False),
])
def test_step_host_equals_device_step(S, n_chunks, gated, kv, backward):
    """Inputs from pinned host memory, outputs back to it, copies overlapped
    with the kernels on side streams: the same results as dsa_step."""
    wl = synth.scaled(synth.WORKLOADS["glm_s16k"], S)
    cfg = _cfg(wl)
    shapes = dsa.step_shapes(cfg, kv, backward, gated)
    inp = _step_tensors(wl, 43, gated, kv, backward)
    host = {n: t.pin_memory() for n, t in inp.items()}
    host.update(_step_outputs(cfg, shapes, host, "cpu"))
    dev = {n: torch.empty(shape, dtype=dtype, device=DEV)
           for n, (shape, dtype) in shapes.items()}
    ws = dsa.workspace(cfg, dsa.WS_STEP, DEV)
    dsa.step_host(cfg, host, dev, n_chunks, ws=ws)
    torch.cuda.synchronize()
    _status_ok(ws)
    ref = {n: t.to(DEV) for n, t in inp.items()}
    ref.update(_step_outputs(cfg, shapes, ref, DEV))
    dsa.step(cfg, ref, ws=ws)
    torch.cuda.synchronize()
    _status_ok(ws)
    for name in ("topk_idx", "o", "lse") + (("dq",) if backward else ()):
        assert torch.equal(host[name], ref[name].cpu()), name
    if backward:
        _close_bf16(host["dk"], ref["dk"].cpu())
        if not kv:
            _close_bf16(host["dv"], ref["dv"].cpu())


def test_bounded_wait_times_out_and_the_context_survives():
    """A wait that nothing satisfies ends after its limit with
    DSA_ERR_DEVICE_TIMEOUT in the status word; the next calls run normally."""
    wl = synth.scaled(synth.WORKLOADS["tiny_fwd_s1k"], 512)
    cfg = _cfg(wl)
    ws = dsa.workspace(cfg, dsa.WS_STATUS, DEV)
    dsa.check_wait_timeout(ws, 50)
    assert dsa.get_device_status(ws) == 6          # DSA_ERR_DEVICE_TIMEOUT
    assert dsa.get_device_status(ws) == 0          # read and cleared
    _, k_idx, _ = synth.indexer_inputs(wl, 1, "cpu")
    got = dsa.pool_keys(cfg, k_idx.to(DEV))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(got), oracle.pool(bits(k_idx)))


def test_topk_on_vertical_slash_rows_at_1m_tokens():
    """The 1M-token stress configuration: indexer scores of 262k-pool rows
    skewed toward a vertical-slash pattern (+3 sigma on the 256 most recent
    pools and on 16 seeded global columns, sigma the spread of the unbiased
    scores on sampled rows, measured by the oracle), then top-k.  The band
    crowds one warp's stretch of the row, so the kernel's second,
    exact-placement sweep runs.  Checked bit-exactly against the oracle's
    top-k of the same biased fp32 scores, and against the oracle's own fp64
    scores with the same bias within the tie band."""
    wl = synth.WORKLOADS["stress_fwd_s1m"]
    cfg = _cfg(wl)
    S, P, n_rows = wl.S, wl.P, 48
    blocks = [S - n_rows, S // 2]
    q_rows, k_idx, w_rows = synth.indexer_row_inputs(wl, 29, n_rows * len(blocks), "cpu")
    kpool_h = oracle.pool(bits(k_idx))
    # the spread of the unbiased scores, from the oracle on sampled rows
    probe = np.array([blocks[0] + 5, blocks[0] + n_rows - 1, blocks[1] + 3], np.int64)
    probe_i = np.array([5, n_rows - 1, n_rows + 3], np.int64)
    sc_probe = oracle.index_scores(bits(q_rows)[probe_i], kpool_h,
                                   w_rows.numpy()[probe_i], probe, S)
    sigma = float(np.std(sc_probe[np.isfinite(sc_probe)]))
    bias = float(np.float32(3.0 * sigma))
    cols = synth.vertical_slash_columns(wl, 29)
    q_full = torch.zeros((S, wl.H_I, wl.D_I), dtype=torch.bfloat16, device=DEV)
    w_full = torch.zeros((S, wl.H_I), dtype=torch.float32, device=DEV)
    kp = dsa.pool_keys(cfg, k_idx.to(DEV))
    ws = dsa.workspace(cfg, dsa.WS_STATUS, DEV)
    ld = (P + 127) // 128 * 128
    for b, t0 in enumerate(blocks):
        rows = np.arange(t0, t0 + n_rows, dtype=np.int64)
        q_full[t0:t0 + n_rows] = q_rows[b * n_rows:(b + 1) * n_rows].to(DEV)
        w_full[t0:t0 + n_rows] = w_rows[b * n_rows:(b + 1) * n_rows].to(DEV)
        sc = dsa.index_scores(cfg, q_full, kp, w_full, t0, n_rows, ld=ld, ws=ws)
        synth.vertical_slash_bias(sc, rows, bias, cols)
        got = dsa.topk_from_scores(cfg, sc, t0, ws=ws)
        _status_ok(ws)
        # bit-exact on the shared (GPU-computed, biased) fp32 scores
        ref_shared = oracle.topk(sc.cpu().numpy(), rows, wl.K_p)
        np.testing.assert_array_equal(got.cpu().numpy(), ref_shared)
        # against the oracle's fp64 scores with the same bias, on sampled rows
        pick = np.array([0, n_rows // 2, n_rows - 1], np.int64)
        sel = b * n_rows + pick
        sc64 = oracle.index_scores(bits(q_rows)[sel], kpool_h, w_rows.numpy()[sel],
                                   rows[pick], S)
        synth.vertical_slash_bias(sc64, rows[pick], bias, cols)
        ref = oracle.topk(sc64, rows[pick], wl.K_p)
        eq, ex = check_index_rows(got.cpu().numpy()[pick], ref, sc64, rows[pick], wl.K_p)
        assert eq + ex == pick.size
        # the skew took effect: about half the +3 sigma band is selected (an
        # unbiased band of 256 pools would hold about 0.5 of 512 out of 262k)
        band_hits = (got.cpu().numpy()[pick] >= (rows[pick, None] + 1) // 4 - 256).sum(1)
        assert band_hits.min() >= 16 and band_hits.mean() >= 48, band_hits
        q_full[t0:t0 + n_rows] = 0
        w_full[t0:t0 + n_rows] = 0


def test_forward_at_1m_tokens_sampled_rows():
    """The 1M-token forward configuration end to end on the GPU: chunked
    indexer + top-k under the 2 GiB scratch cap (256 MiB chunks of 262k-pool
    rows), then the sparse attention forward; sampled late and middle rows
    checked against the oracle (selection within the tie band, O and LSE
    within the attention tolerance on the GPU's selection)."""
    wl = synth.WORKLOADS["stress_fwd_s1m"]
    cfg = _cfg(wl)
    S = wl.S
    torch.cuda.empty_cache()
    try:
        q_idx = synth.normal_bf16_blocks((S, wl.H_I, wl.D_I), 1 / math.sqrt(wl.D_I), 61,
                                         DEV, 65536)
        k_idx = synth.normal_bf16_blocks((S, wl.D_I), 1 / math.sqrt(wl.D_I), 62, DEV, S)
        w = torch.softmax(torch.randn((S, wl.H_I), generator=synth._gen(63, DEV),
                                      device=DEV), dim=-1).contiguous()
        idx = dsa.index_scores_topk(cfg, q_idx, k_idx, w)
        q = synth.normal_bf16_blocks((S, wl.H, wl.d_qk), 1 / math.sqrt(wl.d_qk), 64, DEV,
                                     8192)
        k = synth.normal_bf16_blocks((S, wl.d_qk), 1 / math.sqrt(wl.d_qk), 65, DEV, S)
        v = synth.normal_bf16_blocks((S, wl.d_v), 1 / math.sqrt(wl.d_v), 66, DEV, S)
        wsf = dsa.workspace(cfg, dsa.WS_FWD, DEV)
        o, lse = dsa.sparse_attn_fwd(cfg, q, k, v, idx, ws=wsf)
        _status_ok(wsf)
        rows = np.array([S // 2 + 7, S - 257, S - 1], np.int64)
        rt = torch.from_numpy(rows).to(DEV)
        idx_h = idx.cpu().numpy()
        kp = oracle.pool(bits(k_idx))
        sc = oracle.index_scores(bits(q_idx[rt]), kp, w[rt].cpu().numpy(), rows, S)
        ref = oracle.topk(sc, rows, wl.K_p)
        eq, ex = check_index_rows(idx_h[rows], ref, sc, rows, wl.K_p)
        assert eq + ex == rows.size
        ro, rl = oracle.attn_fwd(bits(q[rt]), bits(k), bits(v), idx_h, wl.K_p, wl.n_loc,
                                 cfg.scale, rows)
        om, _ = oracle.attn_fwd(bits(q[rt]), bits(k), abs_bits(bits(v)), idx_h, wl.K_p,
                                wl.n_loc, cfg.scale, rows)
        assert_close(f64(o[rt]), ro, "o", mag=om)
        assert_close(f64(lse[rt]), rl, "lse")
    finally:
        q_idx = k_idx = w = idx = q = k = v = o = lse = None
        torch.cuda.empty_cache()


@pytest.mark.parametrize("name,n_index_rows,n_attn_rows", [
    ("glm_chunked_s128k", 4096, 16),   # the bench configuration, full size
    ("padded2051_s64k", 1024, 16),     # 2,051 keys, 16 heads, full size
])
def test_full_size_configuration_sampled_rows(name, n_index_rows, n_attn_rows):
    """A configuration at its full sequence length, in the launch
    configuration the bench times (chunked indexer + top-k, forward,
    backward): the selection of n_index_rows sampled queries (seeded rows
    plus the edge rows) against the unchunked fp64 oracle within the tie
    band, and O, LSE, dq, dK, dV of sampled rows against the oracle."""
    import concurrent.futures
    import os
    wl = synth.WORKLOADS[name]
    cfg = _cfg(wl)
    S = wl.S
    torch.cuda.empty_cache()
    try:
        q_idx = synth.normal_bf16_blocks((S, wl.H_I, wl.D_I), 1 / math.sqrt(wl.D_I), 71,
                                         DEV, 16384)
        k_idx = synth.normal_bf16_blocks((S, wl.D_I), 1 / math.sqrt(wl.D_I), 72, DEV, S)
        w = torch.softmax(torch.randn((S, wl.H_I), generator=synth._gen(73, DEV),
                                      device=DEV), dim=-1).contiguous()
        q = synth.normal_bf16_blocks((S, wl.H, wl.d_qk), 1 / math.sqrt(wl.d_qk), 74, DEV,
                                     8192)
        k = synth.normal_bf16_blocks((S, wl.d_qk), 1 / math.sqrt(wl.d_qk), 75, DEV, S)
        v = synth.normal_bf16_blocks((S, wl.d_v), 1 / math.sqrt(wl.d_v), 76, DEV, S)
        dO = synth.normal_bf16_blocks((S, wl.H, wl.d_v), 1.0, 77, DEV, 8192)
        wsi = dsa.workspace(cfg, dsa.WS_INDEX, DEV)
        idx = dsa.index_scores_topk(cfg, q_idx, k_idx, w, ws=wsi)
        o, lse = dsa.sparse_attn_fwd(cfg, q, k, v, idx)
        _status_ok(wsi)
        # ---- the selection, sampled rows, oracle calls spread over the cores
        rows = synth.sample_rows(wl, n_index_rows, 9).numpy()
        rt = torch.from_numpy(rows).to(DEV)
        q_rows, w_rows = bits(q_idx[rt]), w[rt].cpu().numpy()
        kp = oracle.pool(bits(k_idx))
        got = idx[rt].cpu().numpy()
        parts = np.array_split(np.arange(rows.size), max(1, min(32, os.cpu_count() or 1)))

        def check(part):
            sc = oracle.index_scores(q_rows[part], kp, w_rows[part], rows[part], S)
            ref = oracle.topk(sc, rows[part], wl.K_p)
            return check_index_rows(got[part], ref, sc, rows[part], wl.K_p)
        with concurrent.futures.ThreadPoolExecutor(len(parts)) as ex:
            res = list(ex.map(check, parts))
        eq = sum(r[0] for r in res)
        exempt = sum(r[1] for r in res)
        assert eq + exempt == rows.size and eq >= 0.9 * rows.size
        # ---- attention on sampled rows (the GPU selection on both sides)
        arows = synth.sample_rows(wl, n_attn_rows, 10).numpy()
        at = torch.from_numpy(arows).to(DEV)
        idx_h = idx.cpu().numpy()
        ro, rl = oracle.attn_fwd(bits(q[at]), bits(k), bits(v), idx_h, wl.K_p, wl.n_loc,
                                 cfg.scale, arows)
        om, _ = oracle.attn_fwd(bits(q[at]), bits(k), abs_bits(bits(v)), idx_h, wl.K_p,
                                wl.n_loc, cfg.scale, arows)
        assert_close(f64(o[at]), ro, "o", mag=om)
        assert_close(f64(lse[at]), rl, "lse")
        dq, _, _ = dsa.sparse_attn_bwd(cfg, q, k, v, o, lse, dO, idx)
        rdq, _, _ = oracle.attn_bwd(bits(q[at]), bits(k), bits(v), bits(dO[at]), idx_h,
                                    wl.K_p, wl.n_loc, cfg.scale, arows,
                                    np.zeros(1, np.int64))
        assert_close(f64(dq[at]), rdq, "dq")
        dq = None
        _masked_dkdv_check(wl, cfg, q, k, v, dO, idx, o, lse, arows[-6:])
        # ---- the same selection with attention inputs of order one, where
        # O, dq, dK and dV cannot pass as zeros
        q = k = v = dO = o = lse = None
        torch.cuda.empty_cache()
        sq, sk, sv, sg = synth.attention_std(wl, "unit")
        q = synth.normal_bf16_blocks((S, wl.H, wl.d_qk), sq, 84, DEV, 8192)
        k = synth.normal_bf16_blocks((S, wl.d_qk), sk, 85, DEV, S)
        v = synth.normal_bf16_blocks((S, wl.d_v), sv, 86, DEV, S)
        dO = synth.normal_bf16_blocks((S, wl.H, wl.d_v), sg, 87, DEV, 8192)
        o, lse = dsa.sparse_attn_fwd(cfg, q, k, v, idx)
        ro, rl = oracle.attn_fwd(bits(q[at]), bits(k), bits(v), idx_h, wl.K_p, wl.n_loc,
                                 cfg.scale, arows)
        om, _ = oracle.attn_fwd(bits(q[at]), bits(k), abs_bits(bits(v)), idx_h, wl.K_p,
                                wl.n_loc, cfg.scale, arows)
        assert_close(f64(o[at]), ro, "o (unit inputs)", mag=om, **tol("unit"))
        assert_close(f64(lse[at]), rl, "lse (unit inputs)")
        _masked_dkdv_check(wl, cfg, q, k, v, dO, idx, o, lse, arows[-6:], "unit")
    finally:
        q_idx = k_idx = w = q = k = v = dO = idx = o = lse = None
        torch.cuda.empty_cache()

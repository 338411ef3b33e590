"""Shared test helpers: tensor <-> bit-pattern conversion, the output
comparison rule, the index-set comparison rule with its relative tie band,
and the oracle's attention calls spread over host threads."""
from __future__ import annotations

import concurrent.futures
import os

import numpy as np
import torch

import oracle

# Acceptance tolerances for bf16 I/O with fp32 accumulation.
ATOL_OUT = 2e-2          # O, LSE, dQ, dK, dV: max-abs
# Outputs are stored in bf16, whose rounding alone moves x by up to
# 2^-9 |x|; one bf16 ulp (2^-8 |x|) also covers fp32 summation order and the
# bf16-rounded P / dS operands of the tensor-core products.  For the
# workloads' magnitudes (|O|, |dQ|, |dK|, |dV| <~ 1) the bound is the 2e-2.
RTOL_BF16 = 2.0 ** -8
# Scale-aware bound on a whole tensor: max|got - ref| <= REL_MAX * max|ref|.
# At the pages' input scale O, dQ and dK sit far below ATOL_OUT, so the
# absolute bound alone would accept a kernel that wrote zeros; this one
# cannot (zeros give an error of max|ref|).  The bf16 roundings above make
# errors of a few 2^-9 of the typical magnitude; 2e-2 is about ten times that.
REL_MAX = 2e-2
# At the unit and peaked input scales (synth.ATTN_INPUT_SCALES) the outputs
# are of order one and the absolute 2e-2 is not the acceptance bound: a dK
# element sums thousands of (query, head) terms whose magnitudes far exceed
# the (cancelling) result, and two bf16 roundings inside the method move it
# by a few 2^-9 of those terms -- delta is formed from the bf16 O the
# backward receives, and dS enters the tensor-core products in bf16 (a CPU
# emulation at S=640, 64 heads, d=512 puts each near 0.03 on early keys whose
# |dK| is 0.01..10).  There the checks are relative to the whole tensor: the
# REL_MAX bound on the largest error, and the relative Frobenius error
# ||got - ref|| <= REL_FROB ||ref|| (bf16 roundings give about 2^-9).
REL_FROB = 1e-2
TIE_BAND = 1e-3          # relative gap below which index sets may differ


def tol(scale: str) -> dict:
    """assert_close keyword arguments for attention outputs at an input scale."""
    return {} if scale == "pages" else {"atol": None, "frob": REL_FROB}

# (test, tensor, max err, max |ref|) of every comparison in this process;
# written out by conftest when DSA_PARITY_REPORT names a file
PARITY_LOG: list = []


def assert_close(got, ref, name="", mag=None, atol=ATOL_OUT, rtol=RTOL_BF16,
                 rel=REL_MAX, frob=None):
    """|got - ref| <= atol + rtol * mag elementwise (atol=None skips it),
    infinities equal, max|got - ref| <= rel * max|ref| over the finite
    entries (rel=None skips it) and, when frob is given,
    ||got - ref||_F <= frob * ||ref||_F.

    mag is the magnitude the result is built from: |ref| by default, or,
    where the oracle can give it, the sum of the absolute values of the
    summed terms (e.g. sum_j P_j |v_j| for O, sum P |dO| for dV).  A
    tensor-core product rounds its bf16 operands (P, dS) by up to 2^-9 each,
    so its error scales with that sum, not with the (possibly cancelling)
    result."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    m = np.abs(ref) if mag is None else np.maximum(np.abs(ref), np.abs(mag))
    inf = np.isinf(ref)
    assert np.array_equal(got[inf], ref[inf]), f"{name}: infinities differ"
    g, r, m = got[~inf], ref[~inf], m[~inf]
    assert np.isfinite(g).all(), f"{name}: non-finite values"
    if g.size:
        excess = (np.abs(g - r) - rtol * m).max()
        err = np.abs(g - r).max()
        top = np.abs(r).max()
        PARITY_LOG.append((os.environ.get("PYTEST_CURRENT_TEST", ""), name,
                           float(err), float(top)))
        if atol is not None:
            assert excess <= atol, f"{name}: max err {err:.3g} (excess {excess:.3g})"
        if rel is not None:
            assert err <= rel * top, (f"{name}: max err {err:.3g} above "
                                      f"{rel} x max|ref| = {rel * top:.3g}")
        if frob is not None:
            fe, fr = float(np.linalg.norm(g - r)), float(np.linalg.norm(r))
            assert fe <= frob * fr, (f"{name}: relative Frobenius error "
                                     f"{fe / fr if fr else fe:.3g} above {frob}")


def _parts(n: int, parts: int | None):
    k = max(1, min(n, parts or min(32, os.cpu_count() or 1)))
    return [p for p in np.array_split(np.arange(n), k) if p.size]


def oracle_attn_fwd(q_rows, k, v, idx, K_p, n_loc, scale, rows, parts=None):
    """oracle.attn_fwd on `rows` (q_rows holds those rows, in order), the
    rows spread over host threads (ctypes releases the GIL; rows are
    independent, so the results are the single call's)."""
    rows = np.asarray(rows, np.int64)
    blocks = _parts(rows.size, parts)
    with concurrent.futures.ThreadPoolExecutor(len(blocks)) as ex:
        res = list(ex.map(lambda b: oracle.attn_fwd(q_rows[b], k, v, idx, K_p, n_loc,
                                                    scale, rows[b]), blocks))
    return (np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res]))


def oracle_attn_bwd(q_rows, k, v, dO_rows, idx, K_p, n_loc, scale, rows,
                    keys=None, parts=None):
    """oracle.attn_bwd on `rows`, spread over host threads: dq rows are
    independent; the dk/dv contributions of the row blocks are summed (fp64,
    another order than one call's, so equal to fp64 rounding)."""
    rows = np.asarray(rows, np.int64)
    blocks = _parts(rows.size, parts)
    with concurrent.futures.ThreadPoolExecutor(len(blocks)) as ex:
        res = list(ex.map(lambda b: oracle.attn_bwd(q_rows[b], k, v, dO_rows[b], idx,
                                                    K_p, n_loc, scale, rows[b], keys),
                          blocks))
    dq = np.concatenate([r[0] for r in res])
    return dq, sum(r[1] for r in res), sum(r[2] for r in res)


def abs_bits(b: np.ndarray) -> np.ndarray:
    """|x| of bf16 bit patterns (clear the sign bit; exact)."""
    return np.asarray(b, np.uint16) & np.uint16(0x7FFF)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(
        np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_index_rows(gpu: np.ndarray, ora: np.ndarray, scores: np.ndarray,
                     rows: np.ndarray, K: int, band: float = TIE_BAND):
    """Compare GPU and oracle top-K rows.  A row may differ only when the
    oracle's K-th and (K+1)-th best fp64 scores are within `band` relative
    (both zero counts as within); then every index in one set but not the
    other must score within the band of the K-th best.
    Returns (n_rows_equal, n_rows_exempt_and_valid)."""
    eq = ex = 0
    for i, t in enumerate(rows):
        n = (int(t) + 1) // 4
        g, o = gpu[i], ora[i]
        if np.array_equal(g, o):
            eq += 1
            continue
        assert n > K, f"row {t}: {n} pools <= K={K} but sets differ"
        s = scores[i, :n]
        order = np.sort(s)[::-1]
        sk, sk1 = order[K - 1], order[K]
        gap_ok = abs(sk - sk1) <= band * max(abs(sk), abs(sk1))
        assert gap_ok, (f"row {t}: index sets differ without a tie "
                        f"(s_k={sk!r}, s_k+1={sk1!r})")
        gs, os_ = set(g[g >= 0].tolist()), set(o[o >= 0].tolist())
        assert len(gs) == len(os_) == min(K, n)
        for p in gs ^ os_:
            assert abs(s[p] - sk) <= band * max(abs(s[p]), abs(sk)) + 1e-300, \
                f"row {t}: pool {p} (score {s[p]!r}) outside the tie band"
        ex += 1
    return eq, ex

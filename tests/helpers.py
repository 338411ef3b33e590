"""Shared test helpers: tensor <-> bit-pattern conversion and the index-set
comparison rule with its relative tie band."""
from __future__ import annotations

import numpy as np
import torch

# Acceptance tolerances for bf16 I/O with fp32 accumulation.
ATOL_OUT = 2e-2          # O, LSE, dQ, dK, dV: max-abs
# Outputs are stored in bf16, whose rounding alone moves x by up to
# 2^-9 |x|; one bf16 ulp (2^-8 |x|) also covers fp32 summation order and the
# bf16-rounded P / dS operands of the tensor-core products.  For the
# workloads' magnitudes (|O|, |dQ|, |dK|, |dV| <~ 1) the bound is the 2e-2.
RTOL_BF16 = 2.0 ** -8
TIE_BAND = 1e-3          # relative gap below which index sets may differ


def assert_close(got, ref, name="", mag=None, atol=ATOL_OUT, rtol=RTOL_BF16):
    """|got - ref| <= atol + rtol * mag elementwise, infinities equal.

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
        assert excess <= atol, f"{name}: max err {err:.3g} (excess {excess:.3g})"


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

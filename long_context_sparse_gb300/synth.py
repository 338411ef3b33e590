"""Seeded synthetic inputs for the DSA hot path.

This module only draws random tensors of the shapes and distributions of the
workloads; it holds none of the method's arithmetic, so both the CUDA library
and the CPU oracle can be fed from it.

Workloads follow the sizes of the DSA layer described in "Scaling Training to
1M Token Context on GLM-5.3-Flash" (sections "DeepSeek Sparse Attention (DSA)
Optimizations", "Making Sparse Attention Actually Sparse" and "Splitting the
DSA Indexer"): pools of 4 tokens, 512 selected pools (2048 keys) or 512 pools
plus 3 local tokens (2051 keys), NoPE q/k, one K and one V shared by all
heads, and a chunked indexer.  That page measures on random tokens with
random-init weights, so random inputs are its own workload type.

Distributions: bf16 tensors ~ N(0,1)/sqrt(dim); indexer head weights
w = softmax over heads of N(0,1) (fp32); upstream gradient dO ~ N(0,1) bf16.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    S: int            # sequence length (batch 1)
    H_I: int          # indexer heads
    D_I: int          # indexer dim
    K_p: int          # selected pools per query
    n_loc: int        # 0 -> 4*K_p keys, 3 -> 4*K_p + 3 keys
    H: int            # attention query heads (one shared K/V)
    d_qk: int
    d_v: int
    chunk_q: int      # queries scored per indexer chunk
    scratch_cap: int  # bytes allowed for one score chunk
    backward: bool    # fwd+bwd (True) or forward only
    description: str

    @property
    def P(self) -> int:
        return self.S // 4

    @property
    def keys_per_query(self) -> int:
        return 4 * self.K_p + self.n_loc


GiB = 1 << 30

WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_fwd_s1k", 1024, 4, 64, 64, 0, 8, 128, 128, 256, 2 * GiB,
                 False, "S=1024, indexer 4x64, top-64 pools (256 keys), "
                 "8 heads, d=128, forward only"),
        Workload("glm_s16k", 16384, 32, 128, 512, 0, 64, 512, 512, 256,
                 2 * GiB, True, "S=16384, indexer 32x128, top-512 pools "
                 "(2048 keys), 64 heads, d_qk=d_v=512, fwd+bwd"),
        Workload("glm_chunked_s128k", 131072, 32, 128, 512, 0, 64, 512, 512,
                 256, 2 * GiB, True, "S=131072, indexer 32x128 scored 256 "
                 "queries per chunk under a 2 GiB cap, top-512 pools (2048 "
                 "keys), 64 heads, d_qk=d_v=512, fwd+bwd"),
        Workload("padded2051_s64k", 65536, 16, 128, 512, 3, 16, 512, 512, 256,
                 2 * GiB, True, "S=65536, indexer 16x128, top-512 pools + 3 "
                 "local tokens (2051 keys), 16 heads, d=512, fwd+bwd"),
        Workload("stress_fwd_s1m", 1048576, 32, 128, 512, 0, 64, 512, 512, 256,
                 2 * GiB, False, "S=1048576, indexer 32x128, top-512 pools, "
                 "64 heads, d=512, forward only"),
    ]
}


def scaled(wl: Workload, S: int, **over) -> Workload:
    """The same shapes at another sequence length (parity-test sizes)."""
    return dataclasses.replace(wl, S=S, name=f"{wl.name}@S{S}", **over)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal_bf16(shape, std: float, g, device) -> torch.Tensor:
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return (x * std).to(torch.bfloat16)


def indexer_inputs(wl: Workload, seed: int, device="cpu"):
    """q_idx [S,H_I,D_I] bf16, k_idx [S,D_I] bf16, w [S,H_I] fp32."""
    g = _gen(seed, device)
    std = 1.0 / math.sqrt(wl.D_I)
    q_idx = _normal_bf16((wl.S, wl.H_I, wl.D_I), std, g, device)
    k_idx = _normal_bf16((wl.S, wl.D_I), std, g, device)
    w = torch.softmax(torch.randn((wl.S, wl.H_I), generator=g, device=device),
                      dim=-1).contiguous()
    return q_idx, k_idx, w


def normal_bf16_blocks(shape, std: float, seed: int, device,
                       block_rows: int) -> torch.Tensor:
    """bf16 N(0,1)*std of `shape`, drawn block_rows leading rows at a time
    from one seeded generator (no fp32 temporary of the whole tensor)."""
    g = _gen(seed, device)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    for r0 in range(0, shape[0], block_rows):
        r1 = min(shape[0], r0 + block_rows)
        out[r0:r1] = _normal_bf16((r1 - r0,) + tuple(shape[1:]), std, g, device)
    return out


def indexer_row_inputs(wl: Workload, seed: int, n_rows: int, device="cpu"):
    """Indexer inputs for a block of n_rows queries only (long sequences):
    q_idx [n_rows,H_I,D_I] bf16, k_idx [S,D_I] bf16 (every key), w [n_rows,H_I]
    fp32, with the distributions of indexer_inputs."""
    g = _gen(seed + 7, device)
    std = 1.0 / math.sqrt(wl.D_I)
    k_idx = _normal_bf16((wl.S, wl.D_I), std, g, device)
    q_idx = _normal_bf16((n_rows, wl.H_I, wl.D_I), std, g, device)
    w = torch.softmax(torch.randn((n_rows, wl.H_I), generator=g, device=device),
                      dim=-1).contiguous()
    return q_idx, k_idx, w


def vertical_slash_columns(wl: Workload, seed: int, n_cols: int = 16) -> np.ndarray:
    """The seeded global pool columns of the vertical-slash score skew."""
    rng = np.random.default_rng(seed + 31337)
    return np.sort(rng.choice(max(1, wl.P), size=min(n_cols, wl.P), replace=False))


def vertical_slash_bias(scores, rows, bias: float, cols, band: int = 256):
    """Add `bias` in place to the skewed entries of score rows (numpy or
    torch, row i <-> query rows[i]): the local band of the `band` most recent
    complete pools, p in [n_full(t) - band, n_full(t)), and the global
    columns `cols` with p < n_full(t) (each entry once).  This shapes the
    synthetic scores of the 1M-token stress configuration after the
    vertical-slash pattern; it is input shaping, not part of the method."""
    for i, t in enumerate(rows):
        nf = (int(t) + 1) // 4
        lo = max(0, nf - band)
        scores[i, lo:nf] += bias
        c = [int(x) for x in cols if int(x) < lo]
        if c:
            scores[i, c] += bias
    return scores


def gate_inputs(wl: Workload, seed: int, device="cpu"):
    """Per-token pool gate scores [S] fp32 ~ N(0,1) (gated pooling)."""
    g = _gen(seed + 4242, device)
    return torch.randn(wl.S, generator=g, device=device, dtype=torch.float32)


def attention_inputs(wl: Workload, seed: int, device="cpu"):
    """q [S,H,d_qk], k [S,d_qk], v [S,d_v], dO [S,H,d_v], all bf16."""
    g = _gen(seed + 7919, device)
    q = _normal_bf16((wl.S, wl.H, wl.d_qk), 1.0 / math.sqrt(wl.d_qk), g,
                     device)
    k = _normal_bf16((wl.S, wl.d_qk), 1.0 / math.sqrt(wl.d_qk), g, device)
    v = _normal_bf16((wl.S, wl.d_v), 1.0 / math.sqrt(wl.d_v), g, device)
    dO = _normal_bf16((wl.S, wl.H, wl.d_v), 1.0, g, device)
    return q, k, v, dO


# Input scales of the attention parity cases.  "pages": the workloads' own
# N(0,1)/sqrt(dim), under which O, dQ and dK are far below one (a check with
# an absolute bound cannot tell them from zero).  "unit": q, k, v, dO ~ N(0,1)
# per element, so the logits have unit spread after the 1/sqrt(d) scale and
# O, dQ, dK, dV are of order one.  "peaked": as "unit" with q eight times
# larger, so each softmax row is dominated by a few keys and later key tiles
# often raise the running maximum far above the first tile's.
ATTN_INPUT_SCALES = ("pages", "unit", "peaked")
_Q_GAIN = {"unit": 1.0, "peaked": 8.0}


def attention_inputs_scaled(wl: Workload, seed: int, scale: str = "pages",
                            device="cpu"):
    """attention_inputs at one of ATTN_INPUT_SCALES (same shapes, dtypes)."""
    if scale == "pages":
        return attention_inputs(wl, seed, device)
    gain = _Q_GAIN[scale]
    g = _gen(seed + 6007, device)
    q = _normal_bf16((wl.S, wl.H, wl.d_qk), gain, g, device)
    k = _normal_bf16((wl.S, wl.d_qk), 1.0, g, device)
    v = _normal_bf16((wl.S, wl.d_v), 1.0, g, device)
    dO = _normal_bf16((wl.S, wl.H, wl.d_v), 1.0, g, device)
    return q, k, v, dO


def attention_std(wl: Workload, scale: str = "pages"):
    """Standard deviations (q, k, v, dO) of attention_inputs_scaled, for
    drawing the same distributions in row blocks on the device."""
    if scale == "pages":
        return (1.0 / math.sqrt(wl.d_qk), 1.0 / math.sqrt(wl.d_qk),
                1.0 / math.sqrt(wl.d_v), 1.0)
    return (_Q_GAIN[scale], 1.0, 1.0, 1.0)


def random_selection(wl: Workload, seed: int, device="cpu",
                     rows_per_draw: int = 1024) -> torch.Tensor:
    """A valid pool selection [S, K_p] int32 drawn uniformly at random:
    row t holds min(K_p, n_full(t)) distinct pools < n_full(t) in ascending
    order, then -1.  This is what random indexer inputs produce (every subset
    equally likely); it lets attention be checked on the same index array on
    both sides without running the indexer."""
    g = _gen(seed + 104729, device)
    S, P, K = wl.S, wl.P, wl.K_p
    out = torch.full((S, K), -1, dtype=torch.int32, device=device)
    if P == 0:
        return out
    for r0 in range(0, S, rows_per_draw):
        r1 = min(S, r0 + rows_per_draw)
        t = torch.arange(r0, r1, device=device)
        nf = (t + 1) // 4
        u = torch.rand((r1 - r0, P), generator=g, device=device)
        col = torch.arange(P, device=device)
        u = torch.where(col[None, :] < nf[:, None], u, torch.full_like(u, -1.0))
        kk = min(K, P)
        top = torch.topk(u, kk, dim=1).indices
        valid = torch.gather(u, 1, top) >= 0
        top = torch.where(valid, top, torch.full_like(top, P + 1))
        top = torch.sort(top, dim=1).values
        top = torch.where(top > P, torch.full_like(top, -1), top)
        out[r0:r1, :kk] = top.to(torch.int32)
    return out


def sample_rows(wl: Workload, n: int, seed: int) -> torch.Tensor:
    """Seeded uniform rows plus the edge rows of the selection: t <= 8, the
    chunk boundaries c*C-1 and c*C around the sampled region, the row where
    n_full(t) reaches K_p, and S-1.  Sorted, unique, int64 (CPU)."""
    g = _gen(seed + 15485863, "cpu")
    S, C = wl.S, wl.chunk_q
    edge = list(range(min(S, 9)))
    for c in (1, 2, S // C // 2, S // C - 1):
        for t in (c * C - 1, c * C):
            if 0 <= t < S:
                edge.append(t)
    for t in (4 * wl.K_p - 2, 4 * wl.K_p - 1, 4 * wl.K_p, S - 1):
        if 0 <= t < S:
            edge.append(t)
    rnd = torch.randint(0, S, (max(0, n - len(edge)),), generator=g).tolist()
    return torch.tensor(sorted(set(edge + rnd)), dtype=torch.int64)

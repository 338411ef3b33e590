"""CPU oracle for the DSA hot path -- TEST INFRASTRUCTURE ONLY.

Plain, slow, single-threaded C in fp64 (``dsa_oracle.c``), wrapped here with
ctypes and numpy.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package; the library
path never does.  It shares no code with the CUDA library.

Every function cites the passage it follows (see the C file's header):
  [SkyRL]     "Scaling Training to 1M Token Context on GLM-5.3-Flash"
  [MTraining] "MTraining: Efficient Distributed Training for Ultra-Long
              Contexts via Dynamic Sparse Attention"

All bf16 arrays cross this boundary as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_dbl = ctypes.c_double
_p = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (ISO C11, no FP contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_bf16_to_f32.restype = ctypes.c_float
            lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
            lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.oracle_n_full.restype = _i64
            lib.oracle_n_full.argtypes = [_i64]
            lib.oracle_pool.restype = None
            lib.oracle_pool.argtypes = [_i64, _i32, _p, _p]
            lib.oracle_pool_gated.restype = None
            lib.oracle_pool_gated.argtypes = [_i64, _i32, _p, _p, _p]
            lib.oracle_index_scores.restype = None
            lib.oracle_index_scores.argtypes = [_i64, _i32, _i32, _p, _p, _p,
                                                _i64, _p, _p]
            lib.oracle_topk_f64.restype = ctypes.c_int
            lib.oracle_topk_f64.argtypes = [_i64, _i64, _p, _p, _i32, _p]
            lib.oracle_topk_f32.restype = ctypes.c_int
            lib.oracle_topk_f32.argtypes = [_i64, _i64, _p, _p, _i32, _p]
            lib.oracle_key_set.restype = _i64
            lib.oracle_key_set.argtypes = [_i64, _i32, _i32, _p, _p]
            lib.oracle_attn_fwd.restype = ctypes.c_int
            lib.oracle_attn_fwd.argtypes = [_i64, _i32, _i32, _i32, _i32, _i32,
                                            _dbl, _p, _p, _p, _p, _i64, _p,
                                            _p, _p]
            lib.oracle_attn_bwd.restype = ctypes.c_int
            lib.oracle_attn_bwd.argtypes = [_i64, _i32, _i32, _i32, _i32, _i32,
                                            _dbl, _p, _p, _p, _p, _p, _i64,
                                            _p, _p, _i64, _p, _p, _p]
            lib.oracle_dense_masked_attn.restype = None
            lib.oracle_dense_masked_attn.argtypes = [_i64, _i32, _i32, _i32,
                                                     _dbl, _p, _p, _p, _p, _p,
                                                     _p]
            _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# ------------------------------------------------------------------ bf16


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    b = _c(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x) -> np.ndarray:
    """fp32 -> bf16 bit patterns, nearest-even (scalar loop in C)."""
    lib = _load()
    a = _c(x, np.float32).ravel()
    out = np.empty(a.shape, np.uint16)
    for i, v in enumerate(a):
        out[i] = lib.oracle_f32_to_bf16(float(v))
    return out.reshape(np.shape(x))


def n_full(t: int) -> int:
    """Complete pools at or before query t ([SkyRL] "DeepSeek Sparse
    Attention (DSA) Optimizations": only earlier pools are scored)."""
    return int(_load().oracle_n_full(int(t)))


# -------------------------------------------------------------- a1 pool


def pool(k_idx: np.ndarray) -> np.ndarray:
    """k_pool [S//4, D_I] bf16 bits from k_idx [S, D_I] bf16 bits (mean of 4
    consecutive keys, fp32 pairwise sum, bf16 nearest-even)."""
    k = _c(k_idx, np.uint16)
    S, D = k.shape
    out = np.empty((S // 4, D), np.uint16)
    _load().oracle_pool(S, D, _ptr(k), _ptr(out))
    return out


def pool_gated(k_idx: np.ndarray, gate: np.ndarray) -> np.ndarray:
    """Gated pool keys [S//4, D_I] bf16 bits: softmax over each pool's 4 gate
    scores (fp32 [S]) weighting its keys, fp64, rounded via fp32 to bf16."""
    k = _c(k_idx, np.uint16)
    g = _c(gate, np.float32)
    S, D = k.shape
    assert g.shape == (S,)
    out = np.empty((S // 4, D), np.uint16)
    _load().oracle_pool_gated(S, D, _ptr(k), _ptr(g), _ptr(out))
    return out


# ----------------------------------------------------------- a2 indexer


def index_scores(q_idx: np.ndarray, k_pool: np.ndarray, w: np.ndarray,
                 rows=None, S: int = None) -> np.ndarray:
    """I[t,p] in fp64 for the given query rows; -inf where p >= n_full(t).
    k_pool [S//4, D_I] bf16 bits.  Without `rows`: q_idx [S,H_I,D_I] bf16
    bits and w [S,H_I] f32 cover every query.  With `rows`: q_idx and w hold
    those rows only, in that order (then S defaults to 4 * len(k_pool))."""
    q = _c(q_idx, np.uint16)
    kp = _c(k_pool, np.uint16)
    ww = _c(w, np.float32)
    n, H, D = q.shape
    if rows is None:
        S = n
        r = np.arange(S, dtype=np.int64)
    else:
        r = _c(rows, np.int64)
        S = 4 * kp.shape[0] if S is None else S
    P = S // 4
    assert kp.shape == (P, D) and ww.shape == (r.size, H) and n == r.size
    out = np.empty((r.size, P), np.float64)
    _load().oracle_index_scores(S, H, D, _ptr(q), _ptr(kp), _ptr(ww), r.size,
                                _ptr(r), _ptr(out))
    return out


# ------------------------------------------------------------- a4 top-k


def topk(scores: np.ndarray, rows, K_p: int) -> np.ndarray:
    """Top-K_p pools of each score row (ties -> lower pool index), ascending,
    padded with -1.  Row i belongs to query rows[i]; its first n_full(rows[i])
    entries are the candidates.  fp32 input is compared as fp32 values (the
    bit-exact check), fp64 input as fp64."""
    r = _c(rows, np.int64)
    lib = _load()
    out = np.empty((r.size, K_p), np.int32)
    if scores.dtype == np.float32:
        s = _c(scores, np.float32)
        rc = lib.oracle_topk_f32(r.size, s.shape[1], _ptr(s), _ptr(r), K_p,
                                 _ptr(out))
    else:
        s = _c(scores, np.float64)
        rc = lib.oracle_topk_f64(r.size, s.shape[1], _ptr(s), _ptr(r), K_p,
                                 _ptr(out))
    if rc != 0:
        raise MemoryError("oracle top-k: allocation failed")
    return out


def index_topk(q_idx, k_idx, w, K_p: int, rows=None, gate=None):
    """Pool (mean, or gated when `gate` [S] is given) + fp64 indexer + top-k
    for the given rows.  Returns (topk [nrows, K_p] int32, scores [nrows, P]
    fp64)."""
    S = k_idx.shape[0]
    kp = pool(k_idx) if gate is None else pool_gated(k_idx, gate)
    if rows is None:
        r = np.arange(S, dtype=np.int64)
        sc = index_scores(q_idx, kp, w)
    else:
        r = _c(rows, np.int64)
        sc = index_scores(np.asarray(q_idx)[r], kp, np.asarray(w)[r], r, S)
    return topk(sc, r, K_p), sc


# ----------------------------------------------------------- a5 key set


def key_set(t: int, K_p: int, n_loc: int, idx_row: np.ndarray) -> np.ndarray:
    """Tokens attended by query t (ascending, each once)."""
    ir = _c(idx_row, np.int32)
    assert ir.size == K_p
    keys = np.empty(4 * K_p + n_loc + 1, np.int64)
    n = _load().oracle_key_set(int(t), K_p, n_loc, _ptr(ir), _ptr(keys))
    return keys[:n].copy()


# ------------------------------------------------------ a6 attention fwd


def attn_fwd(q, k, v, topk_idx, K_p: int, n_loc: int, scale: float,
             rows=None):
    """fp64 sparse attention forward on the listed rows.
    k [S,d_qk], v [S,d_v] bf16 bits; topk_idx [S,K_p] int32.  Without
    `rows`, q is [S,H,d_qk]; with `rows`, q holds those rows only, in order.
    Returns (o [nrows,H,d_v], lse [nrows,H])."""
    qq, kk, vv = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    ii = _c(topk_idx, np.int32)
    n, H, dqk = qq.shape
    S, dv = vv.shape
    assert kk.shape == (S, dqk) and ii.shape == (S, K_p)
    r = np.arange(S, dtype=np.int64) if rows is None else _c(rows, np.int64)
    assert n == r.size
    o = np.empty((r.size, H, dv), np.float64)
    lse = np.empty((r.size, H), np.float64)
    rc = _load().oracle_attn_fwd(S, H, dqk, dv, K_p, n_loc, float(scale),
                                 _ptr(qq), _ptr(kk), _ptr(vv), _ptr(ii),
                                 r.size, _ptr(r), _ptr(o), _ptr(lse))
    if rc != 0:
        raise MemoryError("oracle attn_fwd: allocation failed")
    return o, lse


# ------------------------------------------------------ a8 attention bwd


def attn_bwd(q, k, v, dO_rows, topk_idx, K_p: int, n_loc: int, scale: float,
             rows=None, keys=None):
    """fp64 analytic backward with upstream gradient dO_rows [nrows,H,d_v]
    (bf16 bits) on the listed rows and zero elsewhere.  q is [S,H,d_qk]
    without `rows`, else the listed rows only, in order.
    Returns (dq [nrows,H,d_qk], dk, dv): dk/dv are [S, d] or, when `keys`
    (token ids) is given, [len(keys), d] holding only those tokens' rows."""
    qq, kk, vv = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    gg = _c(dO_rows, np.uint16)
    ii = _c(topk_idx, np.int32)
    n, H, dqk = qq.shape
    S, dv = vv.shape
    r = np.arange(S, dtype=np.int64) if rows is None else _c(rows, np.int64)
    assert gg.shape == (r.size, H, dv) and n == r.size
    if keys is None:
        slot, n_slots = None, S
    else:
        keys = _c(keys, np.int64)
        slot = np.full(S, -1, np.int64)
        slot[keys] = np.arange(keys.size)
        n_slots = keys.size
    dq = np.empty((r.size, H, dqk), np.float64)
    dk = np.empty((n_slots, dqk), np.float64)
    dvv = np.empty((n_slots, dv), np.float64)
    rc = _load().oracle_attn_bwd(S, H, dqk, dv, K_p, n_loc, float(scale),
                                 _ptr(qq), _ptr(kk), _ptr(vv), _ptr(gg),
                                 _ptr(ii), r.size, _ptr(r),
                                 None if slot is None else _ptr(slot),
                                 n_slots, _ptr(dq), _ptr(dk), _ptr(dvv))
    if rc != 0:
        raise MemoryError("oracle attn_bwd: allocation failed")
    return dq, dk, dvv


def dense_masked_attn(q, k, v, mask: np.ndarray, scale: float):
    """Textbook dense attention under an explicit [S,S] 0/1 mask."""
    qq, kk, vv = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    S, H, dqk = qq.shape
    dv = vv.shape[1]
    m = _c(mask, np.uint8)
    assert m.shape == (S, S)
    o = np.empty((S, H, dv), np.float64)
    lse = np.empty((S, H), np.float64)
    _load().oracle_dense_masked_attn(S, H, dqk, dv, float(scale), _ptr(qq),
                                     _ptr(kk), _ptr(vv), _ptr(m), _ptr(o),
                                     _ptr(lse))
    return o, lse


def key_mask(S: int, topk_idx: np.ndarray, K_p: int, n_loc: int) -> np.ndarray:
    """[S,S] 0/1 mask of the key sets K(t), built from key_set."""
    m = np.zeros((S, S), np.uint8)
    for t in range(S):
        m[t, key_set(t, K_p, n_loc, topk_idx[t])] = 1
    return m

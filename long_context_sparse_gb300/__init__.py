"""GB300-native DeepSeek-Sparse-Attention hot path.

Thin ctypes binding over the C ABI in ``include/dsa.h`` (library
``libdsa_gb300.so`` in this directory, built by ``build.py``).  This module
only marshals arguments: torch supplies device memory and the current CUDA
stream, every step of the computation runs in the library's CUDA kernels.
There is no CPU or dense fallback: if the library is missing or the device
cannot run it, calls raise.

Function names follow the C entry points without the ``dsa_`` prefix.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import threading

import torch

from .synth import Workload

__all__ = [
    "Config", "DsaError", "config_for", "workspace_size", "workspace",
    "pool_keys", "index_scores", "topk_from_scores", "index_scores_topk",
    "index_scores_topk_static", "static_device_status", "host_buffer",
    "sparse_attn_fwd", "sparse_attn_bwd", "get_device_status",
    "status_string", "library_path", "WS_INDEX", "WS_FWD", "WS_BWD",
    "WS_STATUS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
# DSA_GB300_CHECKS=1 loads the debug build (built by build(checks=True)):
# every kernel bounds-checks its shared-memory, TMEM and global offsets and
# latches DSA_ERR_DEVICE_CHECK instead of making the access
_LIB_PATH = os.path.join(
    _HERE, "libdsa_gb300_checks.so" if os.environ.get("DSA_GB300_CHECKS") == "1"
    else "libdsa_gb300.so")
_lock = threading.Lock()
_lib = None

WS_INDEX, WS_FWD, WS_BWD, WS_STATUS, WS_STREAM, WS_BWD_ROWS, WS_STEP = range(7)

STATUS_NAMES = {
    0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED_SHAPE",
    3: "DSA_ERR_WORKSPACE_TOO_SMALL", 4: "DSA_ERR_MISALIGNED",
    5: "DSA_ERR_CUDA", 6: "DSA_ERR_DEVICE_TIMEOUT",
    7: "DSA_ERR_DEVICE_BAD_INDEX", 8: "DSA_ERR_SCRATCH_CAP", 9: "DSA_ERR_DEVICE_CHECK",
}

# every symbol include/dsa.h declares
EXPORTS = [
    "dsa_workspace_size", "dsa_workspace_init", "dsa_pool_keys",
    "dsa_index_scores", "dsa_topk_from_scores", "dsa_index_scores_topk",
    "dsa_sparse_attn_fwd", "dsa_sparse_attn_bwd", "dsa_get_device_status",
    "dsa_status_string", "dsa_abi_version", "dsa_last_cuda_error",
    "dsa_index_scores_topk_static", "dsa_index_scores_topk_range",
    "dsa_pool_keys_gated", "dsa_sparse_attn_fwd_kv", "dsa_sparse_attn_bwd_kv",
    "dsa_index_topk_streaming", "dsa_sparse_attn_fwd_range",
    "dsa_sparse_attn_bwd_range", "dsa_accum_to_bf16", "dsa_step",
    "dsa_step_host", "dsa_check_wait_timeout", "dsa_static_device_status",
]


class DsaError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str = ""):
        self.code = int(code)
        msg = f"{where}: {STATUS_NAMES.get(self.code, self.code)}"
        super().__init__(msg + (f" ({detail})" if detail else ""))


class _CConfig(ctypes.Structure):
    _fields_ = [
        ("seq_len", ctypes.c_int64), ("pool_size", ctypes.c_int32),
        ("topk_pools", ctypes.c_int32), ("n_local", ctypes.c_int32),
        ("idx_heads", ctypes.c_int32), ("idx_dim", ctypes.c_int32),
        ("attn_heads", ctypes.c_int32), ("d_qk", ctypes.c_int32),
        ("d_v", ctypes.c_int32), ("chunk_q", ctypes.c_int32),
        ("sm_scale", ctypes.c_float), ("scratch_cap", ctypes.c_uint64),
    ]


assert ctypes.sizeof(_CConfig) == 56

# dsa_step_tensors_t: the step's tensors, in declaration order
STEP_FIELDS = ("q_idx", "k_idx", "w", "k_gate", "q", "k", "v", "dO",
               "topk_idx", "o", "lse", "dq", "dk", "dv")


class _CStepTensors(ctypes.Structure):
    _fields_ = [(f, ctypes.c_void_p) for f in STEP_FIELDS]


@dataclasses.dataclass(frozen=True)
class Config:
    """Mirror of dsa_config_t."""
    seq_len: int
    topk_pools: int = 512
    n_local: int = 0
    idx_heads: int = 32
    idx_dim: int = 128
    attn_heads: int = 64
    d_qk: int = 512
    d_v: int = 512
    chunk_q: int = 256
    sm_scale: float = 0.0
    scratch_cap: int = 2 << 30
    pool_size: int = 4

    @property
    def scale(self) -> float:
        return self.sm_scale if self.sm_scale > 0 else 1.0 / math.sqrt(self.d_qk)

    def c(self) -> _CConfig:
        return _CConfig(self.seq_len, self.pool_size, self.topk_pools,
                        self.n_local, self.idx_heads, self.idx_dim,
                        self.attn_heads, self.d_qk, self.d_v, self.chunk_q,
                        float(self.sm_scale), self.scratch_cap)


def config_for(wl: Workload, **over) -> Config:
    cfg = Config(seq_len=wl.S, topk_pools=wl.K_p, n_local=wl.n_loc,
                 idx_heads=wl.H_I, idx_dim=wl.D_I, attn_heads=wl.H,
                 d_qk=wl.d_qk, d_v=wl.d_v, chunk_q=wl.chunk_q,
                 scratch_cap=wl.scratch_cap)
    return dataclasses.replace(cfg, **over) if over else cfg


def library_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise ImportError(
                f"CUDA library {_LIB_PATH} is missing; build it with "
                "`python -m long_context_sparse_gb300.build` (add --checks "
                "for the debug build; there is no CPU fallback)")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I32, I64, SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                           ctypes.c_size_t)
        CP = ctypes.POINTER(_CConfig)
        sig = {
            "dsa_workspace_size": [CP, I32, ctypes.POINTER(SZ)],
            "dsa_workspace_init": [P, SZ, P],
            "dsa_pool_keys": [CP, P, P, P],
            "dsa_index_scores": [CP, P, P, P, I64, I64, P, I64, P, SZ, P],
            "dsa_topk_from_scores": [CP, P, I64, I64, I64, P, P, SZ, P],
            "dsa_index_scores_topk": [CP, P, P, P, P, P, SZ, P],
            "dsa_sparse_attn_fwd": [CP, P, P, P, P, P, P, P, SZ, P],
            "dsa_sparse_attn_bwd": [CP, P, P, P, P, P, P, P, P, P, P, P, SZ,
                                    P],
            "dsa_get_device_status": [P, P, ctypes.POINTER(ctypes.c_uint32)],
            "dsa_index_scores_topk_static": [CP, P, P, P, P, P],
            "dsa_static_device_status": [P, ctypes.POINTER(ctypes.c_uint32)],
            "dsa_index_scores_topk_range": [CP, P, P, P, P, I64, I64, P, P, SZ, P],
            "dsa_pool_keys_gated": [CP, P, P, P, P],
            "dsa_sparse_attn_fwd_kv": [CP, P, P, P, P, P, P, SZ, P],
            "dsa_index_topk_streaming": [CP, P, P, P, P, I64, I64, P, P, SZ, P],
            "dsa_sparse_attn_bwd_kv": [CP, P, P, P, P, P, P, P, P, P, SZ, P],
            "dsa_sparse_attn_fwd_range": [CP, P, P, P, P, I64, I64, P, P, P,
                                          SZ, P],
            "dsa_sparse_attn_bwd_range": [CP, P, P, P, P, P, P, P, I64, I64,
                                          P, P, P, P, SZ, P],
            "dsa_accum_to_bf16": [P, P, I64, P],
            "dsa_check_wait_timeout": [P, SZ, ctypes.c_uint32, P],
            "dsa_step": [CP, ctypes.POINTER(_CStepTensors), P, SZ, P],
            "dsa_step_host": [CP, ctypes.POINTER(_CStepTensors),
                              ctypes.POINTER(_CStepTensors), I32, P, SZ, P, P,
                              P],
        }
        for name, args in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        lib.dsa_status_string.argtypes = [ctypes.c_int]
        lib.dsa_status_string.restype = ctypes.c_char_p
        lib.dsa_abi_version.argtypes = []
        lib.dsa_abi_version.restype = ctypes.c_int32
        lib.dsa_last_cuda_error.argtypes = []
        lib.dsa_last_cuda_error.restype = ctypes.c_char_p
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return _load().dsa_status_string(int(code)).decode()


def _check(rc: int, where: str):
    if rc != 0:
        detail = _load().dsa_last_cuda_error().decode() if rc == 5 else ""
        raise DsaError(rc, where, detail)


def _stream(dev: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected "
                         f"{tuple(shape)}")


def workspace_size(cfg: Config, which: int) -> int:
    n = ctypes.c_size_t(0)
    cc = cfg.c()
    _check(_load().dsa_workspace_size(ctypes.byref(cc), which,
                                      ctypes.byref(n)), "dsa_workspace_size")
    return n.value


def workspace(cfg: Config, which: int, device="cuda") -> torch.Tensor:
    """A zero-initialised workspace for the call `which` (uint8 tensor)."""
    dev = torch.device(device)
    nbytes = workspace_size(cfg, which)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    _check(_load().dsa_workspace_init(_ptr(ws), nbytes, _stream(dev)),
           "dsa_workspace_init")
    return ws


def _ws(cfg, which, ws, dev):
    if ws is None:
        return workspace(cfg, which, dev)
    _need(ws, "ws", torch.uint8, device=dev)
    return ws


def pool_keys(cfg: Config, k_idx: torch.Tensor, k_pool=None) -> torch.Tensor:
    S, D = cfg.seq_len, cfg.idx_dim
    _need(k_idx, "k_idx", torch.bfloat16, (S, D))
    dev = k_idx.device
    if k_pool is None:
        k_pool = torch.empty((S // 4, D), dtype=torch.bfloat16, device=dev)
    _need(k_pool, "k_pool", torch.bfloat16, (S // 4, D), dev)
    cc = cfg.c()
    _check(_load().dsa_pool_keys(ctypes.byref(cc), _ptr(k_idx), _ptr(k_pool),
                                 _stream(dev)), "dsa_pool_keys")
    return k_pool


def index_scores(cfg: Config, q_idx, k_pool, w, t0: int, rows: int,
                 scores=None, ld: int = None, ws=None) -> torch.Tensor:
    """Indexer scores of queries t0..t0+rows-1: [rows, ld] fp32; entry (r,p)
    is valid for p < n_full(t0 + r)."""
    S = cfg.seq_len
    _need(q_idx, "q_idx", torch.bfloat16, (S, cfg.idx_heads, cfg.idx_dim))
    dev = q_idx.device
    _need(k_pool, "k_pool", torch.bfloat16, (S // 4, cfg.idx_dim), dev)
    _need(w, "w", torch.float32, (S, cfg.idx_heads), dev)
    if ld is None:
        ld = max(4, (S // 4 + 127) // 128 * 128)
    if scores is None:
        scores = torch.empty((rows, ld), dtype=torch.float32, device=dev)
    _need(scores, "scores", torch.float32, (rows, ld), dev)
    ws = _ws(cfg, WS_STATUS, ws, dev)
    cc = cfg.c()
    _check(_load().dsa_index_scores(ctypes.byref(cc), _ptr(q_idx), _ptr(k_pool),
                                    _ptr(w), t0, rows, _ptr(scores), ld,
                                    _ptr(ws), ws.numel(), _stream(dev)),
           "dsa_index_scores")
    return scores


def topk_from_scores(cfg: Config, scores: torch.Tensor, row0: int,
                     out=None, ws=None) -> torch.Tensor:
    """Top-K_p selection of fp32 score rows (row r <-> query row0 + r)."""
    if scores.dim() != 2:
        raise ValueError("scores must be [rows, ld]")
    rows, ld = scores.shape
    _need(scores, "scores", torch.float32)
    dev = scores.device
    if out is None:
        out = torch.empty((rows, cfg.topk_pools), dtype=torch.int32, device=dev)
    _need(out, "topk_idx", torch.int32, (rows, cfg.topk_pools), dev)
    ws = _ws(cfg, WS_STATUS, ws, dev)
    cc = cfg.c()
    _check(_load().dsa_topk_from_scores(ctypes.byref(cc), _ptr(scores), ld,
                                        row0, rows, _ptr(out), _ptr(ws),
                                        ws.numel(), _stream(dev)),
           "dsa_topk_from_scores")
    return out


def index_scores_topk(cfg: Config, q_idx, k_idx, w, out=None,
                      ws=None) -> torch.Tensor:
    """Pool, score (chunked) and select: topk_idx [S, K_p] int32."""
    S = cfg.seq_len
    _need(q_idx, "q_idx", torch.bfloat16, (S, cfg.idx_heads, cfg.idx_dim))
    dev = q_idx.device
    _need(k_idx, "k_idx", torch.bfloat16, (S, cfg.idx_dim), dev)
    _need(w, "w", torch.float32, (S, cfg.idx_heads), dev)
    if out is None:
        out = torch.empty((S, cfg.topk_pools), dtype=torch.int32, device=dev)
    _need(out, "topk_idx", torch.int32, (S, cfg.topk_pools), dev)
    ws = _ws(cfg, WS_INDEX, ws, dev)
    cc = cfg.c()
    _check(_load().dsa_index_scores_topk(ctypes.byref(cc), _ptr(q_idx),
                                         _ptr(k_idx), _ptr(w), _ptr(out),
                                         _ptr(ws), ws.numel(), _stream(dev)),
           "dsa_index_scores_topk")
    return out


def index_scores_topk_range(cfg: Config, q_idx, k_idx, w, t_begin: int,
                            t_end: int, k_gate=None, out=None,
                            ws=None) -> torch.Tensor:
    """Pool (mean, or gated by k_gate [S] fp32), score and select for
    queries t_begin .. t_end-1 only (one rank's share of a query-sharded
    indexer): q_idx [n, H_I, D_I] and w [n, H_I] hold the range's rows,
    k_idx [S, D_I] every key; returns topk_idx [n, K_p] int32,
    n = t_end - t_begin."""
    S = cfg.seq_len
    n = t_end - t_begin
    _need(q_idx, "q_idx", torch.bfloat16, (n, cfg.idx_heads, cfg.idx_dim))
    dev = q_idx.device
    _need(k_idx, "k_idx", torch.bfloat16, (S, cfg.idx_dim), dev)
    _need(w, "w", torch.float32, (n, cfg.idx_heads), dev)
    if k_gate is not None:
        _need(k_gate, "k_gate", torch.float32, (S,), dev)
    if out is None:
        out = torch.empty((n, cfg.topk_pools), dtype=torch.int32, device=dev)
    _need(out, "topk_idx", torch.int32, (n, cfg.topk_pools), dev)
    ws = _ws(cfg, WS_INDEX, ws, dev)
    cc = cfg.c()
    _check(_load().dsa_index_scores_topk_range(
        ctypes.byref(cc), _ptr(q_idx), _ptr(k_idx),
        _ptr(k_gate) if k_gate is not None else None, _ptr(w), t_begin, t_end,
        _ptr(out), _ptr(ws), ws.numel(), _stream(dev)),
        "dsa_index_scores_topk_range")
    return out


def index_topk_streaming(cfg: Config, q_idx, k_idx, w, t_begin: int = 0,
                         t_end: int = None, k_gate=None, out=None,
                         ws=None) -> torch.Tensor:
    """As index_scores_topk_range, with the selection fused into the
    indexer (no score stored; workspace: the pooled keys only)."""
    S = cfg.seq_len
    t_end = S if t_end is None else t_end
    n = t_end - t_begin
    _need(q_idx, "q_idx", torch.bfloat16, (n, cfg.idx_heads, cfg.idx_dim))
    dev = q_idx.device
    _need(k_idx, "k_idx", torch.bfloat16, (S, cfg.idx_dim), dev)
    _need(w, "w", torch.float32, (n, cfg.idx_heads), dev)
    if k_gate is not None:
        _need(k_gate, "k_gate", torch.float32, (S,), dev)
    if out is None:
        out = torch.empty((n, cfg.topk_pools), dtype=torch.int32, device=dev)
    _need(out, "topk_idx", torch.int32, (n, cfg.topk_pools), dev)
    ws = _ws(cfg, WS_STREAM, ws, dev)
    cc = cfg.c()
    _check(_load().dsa_index_topk_streaming(
        ctypes.byref(cc), _ptr(q_idx), _ptr(k_idx),
        _ptr(k_gate) if k_gate is not None else None, _ptr(w), t_begin, t_end,
        _ptr(out), _ptr(ws), ws.numel(), _stream(dev)),
        "dsa_index_topk_streaming")
    return out


def pool_keys_gated(cfg: Config, k_idx: torch.Tensor, k_gate: torch.Tensor,
                    k_pool=None) -> torch.Tensor:
    """Gated pool keys [S//4, D_I] bf16: softmax of each pool's 4 gate
    scores (k_gate [S] fp32) weights its keys."""
    S = cfg.seq_len
    _need(k_idx, "k_idx", torch.bfloat16, (S, cfg.idx_dim))
    dev = k_idx.device
    _need(k_gate, "k_gate", torch.float32, (S,), dev)
    if k_pool is None:
        k_pool = torch.empty((S // 4, cfg.idx_dim), dtype=torch.bfloat16, device=dev)
    _need(k_pool, "k_pool", torch.bfloat16, (S // 4, cfg.idx_dim), dev)
    cc = cfg.c()
    _check(_load().dsa_pool_keys_gated(ctypes.byref(cc), _ptr(k_idx), _ptr(k_gate),
                                       _ptr(k_pool), _stream(dev)),
           "dsa_pool_keys_gated")
    return k_pool


def query_shard(S: int, world: int, rank: int, align: int = 4):
    """Query rows [t_begin, t_end) of `rank` when S queries are split over
    `world` ranks in contiguous blocks of whole `align`-row groups (pool
    boundaries by default), the earlier ranks taking the remainder."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    groups = (S + align - 1) // align
    base, extra = divmod(groups, world)
    g0 = rank * base + min(rank, extra)
    g1 = g0 + base + (1 if rank < extra else 0)
    return min(S, g0 * align), min(S, g1 * align)


def index_scores_topk_static(cfg: Config, q_idx, k_idx, w,
                             out=None) -> torch.Tensor:
    """As index_scores_topk, with the library's own fixed scratch instead of
    a workspace (for callers that cannot allocate device memory; calls must
    not overlap on the GPU)."""
    S = cfg.seq_len
    _need(q_idx, "q_idx", torch.bfloat16, (S, cfg.idx_heads, cfg.idx_dim))
    dev = q_idx.device
    _need(k_idx, "k_idx", torch.bfloat16, (S, cfg.idx_dim), dev)
    _need(w, "w", torch.float32, (S, cfg.idx_heads), dev)
    if out is None:
        out = torch.empty((S, cfg.topk_pools), dtype=torch.int32, device=dev)
    _need(out, "topk_idx", torch.int32, (S, cfg.topk_pools), dev)
    cc = cfg.c()
    _check(_load().dsa_index_scores_topk_static(ctypes.byref(cc), _ptr(q_idx),
                                                _ptr(k_idx), _ptr(w),
                                                _ptr(out), _stream(dev)),
           "dsa_index_scores_topk_static")
    return out


def sparse_attn_fwd(cfg: Config, q, k, v, topk_idx, o=None, lse=None,
                    ws=None):
    """Sparse attention forward: (o [S,H,d_v] bf16, lse [S,H] fp32)."""
    S, H = cfg.seq_len, cfg.attn_heads
    _need(q, "q", torch.bfloat16, (S, H, cfg.d_qk))
    dev = q.device
    _need(k, "k", torch.bfloat16, (S, cfg.d_qk), dev)
    _need(v, "v", torch.bfloat16, (S, cfg.d_v), dev)
    _need(topk_idx, "topk_idx", torch.int32, (S, cfg.topk_pools), dev)
    if o is None:
        o = torch.empty((S, H, cfg.d_v), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((S, H), dtype=torch.float32, device=dev)
    _need(o, "o", torch.bfloat16, (S, H, cfg.d_v), dev)
    _need(lse, "lse", torch.float32, (S, H), dev)
    ws = _ws(cfg, WS_FWD, ws, dev)
    cc = cfg.c()
    _check(_load().dsa_sparse_attn_fwd(ctypes.byref(cc), _ptr(q), _ptr(k),
                                       _ptr(v), _ptr(topk_idx), _ptr(o),
                                       _ptr(lse), _ptr(ws), ws.numel(),
                                       _stream(dev)), "dsa_sparse_attn_fwd")
    return o, lse


def sparse_attn_bwd(cfg: Config, q, k, v, o, lse, dO, topk_idx, dq=None,
                    dk=None, dv=None, ws=None):
    """Sparse attention backward: (dq [S,H,d_qk], dk [S,d_qk], dv [S,d_v])."""
    S, H = cfg.seq_len, cfg.attn_heads
    _need(q, "q", torch.bfloat16, (S, H, cfg.d_qk))
    dev = q.device
    _need(k, "k", torch.bfloat16, (S, cfg.d_qk), dev)
    _need(v, "v", torch.bfloat16, (S, cfg.d_v), dev)
    _need(o, "o", torch.bfloat16, (S, H, cfg.d_v), dev)
    _need(lse, "lse", torch.float32, (S, H), dev)
    _need(dO, "dO", torch.bfloat16, (S, H, cfg.d_v), dev)
    _need(topk_idx, "topk_idx", torch.int32, (S, cfg.topk_pools), dev)
    if dq is None:
        dq = torch.empty_like(q)
    if dk is None:
        dk = torch.empty_like(k)
    if dv is None:
        dv = torch.empty_like(v)
    _need(dq, "dq", torch.bfloat16, (S, H, cfg.d_qk), dev)
    _need(dk, "dk", torch.bfloat16, (S, cfg.d_qk), dev)
    _need(dv, "dv", torch.bfloat16, (S, cfg.d_v), dev)
    ws = _ws(cfg, WS_BWD, ws, dev)
    cc = cfg.c()
    _check(_load().dsa_sparse_attn_bwd(ctypes.byref(cc), _ptr(q), _ptr(k),
                                       _ptr(v), _ptr(o), _ptr(lse), _ptr(dO),
                                       _ptr(topk_idx), _ptr(dq), _ptr(dk),
                                       _ptr(dv), _ptr(ws), ws.numel(),
                                       _stream(dev)), "dsa_sparse_attn_bwd")
    return dq, dk, dv


def sparse_attn_fwd_kv(cfg: Config, q, kv, topk_idx, o=None, lse=None, ws=None):
    """Sparse attention forward with K = V = kv [S, d]: (o, lse)."""
    S, H = cfg.seq_len, cfg.attn_heads
    _need(q, "q", torch.bfloat16, (S, H, cfg.d_qk))
    dev = q.device
    _need(kv, "kv", torch.bfloat16, (S, cfg.d_qk), dev)
    _need(topk_idx, "topk_idx", torch.int32, (S, cfg.topk_pools), dev)
    if o is None:
        o = torch.empty((S, H, cfg.d_v), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((S, H), dtype=torch.float32, device=dev)
    _need(o, "o", torch.bfloat16, (S, H, cfg.d_v), dev)
    _need(lse, "lse", torch.float32, (S, H), dev)
    ws = _ws(cfg, WS_FWD, ws, dev)
    cc = cfg.c()
    _check(_load().dsa_sparse_attn_fwd_kv(ctypes.byref(cc), _ptr(q), _ptr(kv),
                                          _ptr(topk_idx), _ptr(o), _ptr(lse),
                                          _ptr(ws), ws.numel(), _stream(dev)),
           "dsa_sparse_attn_fwd_kv")
    return o, lse


def sparse_attn_bwd_kv(cfg: Config, q, kv, o, lse, dO, topk_idx, dq=None,
                       dkv=None, ws=None):
    """Sparse attention backward with K = V = kv: (dq, dkv = dK + dV)."""
    S, H = cfg.seq_len, cfg.attn_heads
    _need(q, "q", torch.bfloat16, (S, H, cfg.d_qk))
    dev = q.device
    _need(kv, "kv", torch.bfloat16, (S, cfg.d_qk), dev)
    _need(o, "o", torch.bfloat16, (S, H, cfg.d_v), dev)
    _need(lse, "lse", torch.float32, (S, H), dev)
    _need(dO, "dO", torch.bfloat16, (S, H, cfg.d_v), dev)
    _need(topk_idx, "topk_idx", torch.int32, (S, cfg.topk_pools), dev)
    if dq is None:
        dq = torch.empty_like(q)
    if dkv is None:
        dkv = torch.empty_like(kv)
    _need(dq, "dq", torch.bfloat16, (S, H, cfg.d_qk), dev)
    _need(dkv, "dkv", torch.bfloat16, (S, cfg.d_qk), dev)
    ws = _ws(cfg, WS_BWD, ws, dev)
    cc = cfg.c()
    _check(_load().dsa_sparse_attn_bwd_kv(ctypes.byref(cc), _ptr(q), _ptr(kv),
                                          _ptr(o), _ptr(lse), _ptr(dO),
                                          _ptr(topk_idx), _ptr(dq), _ptr(dkv),
                                          _ptr(ws), ws.numel(), _stream(dev)),
           "dsa_sparse_attn_bwd_kv")
    return dq, dkv


def sparse_attn_fwd_range(cfg: Config, q, k, v, topk_idx, t_begin: int,
                          t_end: int, o=None, lse=None, ws=None):
    """Sparse attention forward for queries t_begin .. t_end-1 only: q
    [n,H,d_qk] and topk_idx [n,K_p] hold the range's rows, k and v every
    key; returns (o [n,H,d_v], lse [n,H]), rows bit-identical to the
    whole-sequence call's."""
    S, H, n = cfg.seq_len, cfg.attn_heads, t_end - t_begin
    _need(q, "q", torch.bfloat16, (n, H, cfg.d_qk))
    dev = q.device
    _need(k, "k", torch.bfloat16, (S, cfg.d_qk), dev)
    _need(v, "v", torch.bfloat16, (S, cfg.d_v), dev)
    _need(topk_idx, "topk_idx", torch.int32, (n, cfg.topk_pools), dev)
    if o is None:
        o = torch.empty((n, H, cfg.d_v), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((n, H), dtype=torch.float32, device=dev)
    _need(o, "o", torch.bfloat16, (n, H, cfg.d_v), dev)
    _need(lse, "lse", torch.float32, (n, H), dev)
    ws = _ws(cfg, WS_FWD, ws, dev)
    cc = cfg.c()
    _check(_load().dsa_sparse_attn_fwd_range(
        ctypes.byref(cc), _ptr(q), _ptr(k), _ptr(v), _ptr(topk_idx), t_begin,
        t_end, _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), _stream(dev)),
        "dsa_sparse_attn_fwd_range")
    return o, lse


def sparse_attn_bwd_range(cfg: Config, q, k, v, o, lse, dO, topk_idx,
                          t_begin: int, t_end: int, dk_acc, dv_acc=None,
                          dq=None, ws=None):
    """Sparse attention backward for queries t_begin .. t_end-1 only
    (row-indexed q, o, lse, dO, topk_idx, dq as in sparse_attn_fwd_range):
    returns dq [n,H,d_qk] and ADDS the range's dK/dV contributions into the
    fp32 accumulators dk_acc, dv_acc [S, d] (dv_acc None with v is k:
    dk_acc receives dK + dV)."""
    S, H, n = cfg.seq_len, cfg.attn_heads, t_end - t_begin
    _need(q, "q", torch.bfloat16, (n, H, cfg.d_qk))
    dev = q.device
    _need(k, "k", torch.bfloat16, (S, cfg.d_qk), dev)
    _need(v, "v", torch.bfloat16, (S, cfg.d_v), dev)
    _need(o, "o", torch.bfloat16, (n, H, cfg.d_v), dev)
    _need(lse, "lse", torch.float32, (n, H), dev)
    _need(dO, "dO", torch.bfloat16, (n, H, cfg.d_v), dev)
    _need(topk_idx, "topk_idx", torch.int32, (n, cfg.topk_pools), dev)
    _need(dk_acc, "dk_acc", torch.float32, (S, cfg.d_qk), dev)
    if dv_acc is not None:
        _need(dv_acc, "dv_acc", torch.float32, (S, cfg.d_v), dev)
    if dq is None:
        dq = torch.empty_like(q)
    _need(dq, "dq", torch.bfloat16, (n, H, cfg.d_qk), dev)
    ws = _ws(cfg, WS_BWD_ROWS, ws, dev)
    cc = cfg.c()
    _check(_load().dsa_sparse_attn_bwd_range(
        ctypes.byref(cc), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
        _ptr(dO), _ptr(topk_idx), t_begin, t_end, _ptr(dq), _ptr(dk_acc),
        _ptr(dv_acc) if dv_acc is not None else None, _ptr(ws), ws.numel(),
        _stream(dev)), "dsa_sparse_attn_bwd_range")
    return dq


def accum_to_bf16(acc: torch.Tensor, out=None) -> torch.Tensor:
    """bf16 (round to nearest even) copy of an fp32 accumulator."""
    _need(acc, "acc", torch.float32)
    if out is None:
        out = torch.empty(acc.shape, dtype=torch.bfloat16, device=acc.device)
    _need(out, "out", torch.bfloat16, tuple(acc.shape), acc.device)
    _check(_load().dsa_accum_to_bf16(_ptr(acc), _ptr(out), acc.numel(),
                                     _stream(acc.device)), "dsa_accum_to_bf16")
    return out


def step_shapes(cfg: Config, kv: bool = False, backward: bool = True,
                gated: bool = False) -> dict:
    """Name -> (shape, dtype) of the tensors of one whole step."""
    S, H, HI, DI = cfg.seq_len, cfg.attn_heads, cfg.idx_heads, cfg.idx_dim
    bf, f32 = torch.bfloat16, torch.float32
    shapes = {"q_idx": ((S, HI, DI), bf), "k_idx": ((S, DI), bf),
              "w": ((S, HI), f32), "q": ((S, H, cfg.d_qk), bf),
              "k": ((S, cfg.d_qk), bf), "topk_idx": ((S, cfg.topk_pools),
                                                      torch.int32),
              "o": ((S, H, cfg.d_v), bf), "lse": ((S, H), f32)}
    if gated:
        shapes["k_gate"] = ((S,), f32)
    if not kv:
        shapes["v"] = ((S, cfg.d_v), bf)
    if backward:
        shapes.update({"dO": ((S, H, cfg.d_v), bf), "dq": ((S, H, cfg.d_qk), bf),
                       "dk": ((S, cfg.d_qk), bf)})
        if not kv:
            shapes["dv"] = ((S, cfg.d_v), bf)
    return shapes


def _step_struct(cfg: Config, t: dict, device: bool) -> _CStepTensors:
    kv = "v" not in t or t["v"] is t["k"]
    shapes = step_shapes(cfg, kv, t.get("dO") is not None,
                         t.get("k_gate") is not None)
    for name, (shape, dtype) in shapes.items():
        x = t.get(name)
        if x is None:
            raise ValueError(f"step tensor {name} is missing")
        if device:
            _need(x, name, dtype, shape, t["q"].device)
        elif x.device.type != "cpu" or x.dtype != dtype or \
                tuple(x.shape) != shape or not x.is_contiguous():
            raise ValueError(f"host {name} must be a contiguous CPU {dtype} "
                             f"tensor of shape {shape}")
    vals = {f: (t[f].data_ptr() if t.get(f) is not None else None)
            for f in STEP_FIELDS}
    if kv:
        vals["v"] = vals["k"]
    return _CStepTensors(*[vals[f] for f in STEP_FIELDS])


def step(cfg: Config, dev: dict, ws=None) -> dict:
    """One whole step (indexer + top-k, forward, and the backward when dev
    has "dO") on device tensors named as in step_shapes(); outputs are
    written into dev's output tensors.  K = V when dev has no "v"."""
    d = dev["q"].device
    ws = _ws(cfg, WS_STEP, ws, d)
    st = _step_struct(cfg, dev, True)
    cc = cfg.c()
    _check(_load().dsa_step(ctypes.byref(cc), ctypes.byref(st), _ptr(ws),
                            ws.numel(), _stream(d)), "dsa_step")
    return dev


def step_host(cfg: Config, host: dict, dev: dict, n_chunks: int = 8, ws=None,
              copy_streams=None) -> dict:
    """step() with inputs read from and outputs written to host tensors
    (pinned for the copies to overlap the kernels), staged through the
    device tensors `dev`; copies run on two side streams, kernels on the
    current stream, which is ordered after the last copy back."""
    d = dev["q"].device
    ws = _ws(cfg, WS_STEP, ws, d)
    if copy_streams is None:
        copy_streams = (torch.cuda.Stream(d), torch.cuda.Stream(d))
    hs, ds = copy_streams
    sh = _step_struct(cfg, host, False)
    sd = _step_struct(cfg, dev, True)
    cc = cfg.c()
    _check(_load().dsa_step_host(
        ctypes.byref(cc), ctypes.byref(sh), ctypes.byref(sd), n_chunks,
        _ptr(ws), ws.numel(), _stream(d), ctypes.c_void_p(hs.cuda_stream),
        ctypes.c_void_p(ds.cuda_stream)), "dsa_step_host")
    return host


_HUGE = 2 << 20  # transparent huge page size requested for host buffers


def host_buffer(shape, dtype) -> torch.Tensor:
    """A page-locked host tensor for step_host's copies, backed by 2 MiB
    transparent huge pages (anonymous mmap + madvise(MADV_HUGEPAGE), then
    cudaHostRegister), unregistered and unmapped when the tensor is freed.

    On a Grace host the GPU's copies translate every host page; huge pages
    need 32 times fewer translations than the default 64 KiB pages.  After
    another process had touched and freed a large amount of memory (e.g. a
    test run just before), copies from some cudaHostAlloc buffers were
    measured at 15-25 GB/s instead of about 200 GB/s while huge-page
    buffers kept full rate; at other times a huge-page buffer was slow too.
    A slow buffer stays slow: time it once and allocate another if needed."""
    import weakref
    numel = 1
    for x in shape:
        numel *= int(x)
    nbytes = numel * torch.empty((), dtype=dtype).element_size()
    if nbytes == 0:
        return torch.empty(shape, dtype=dtype, pin_memory=True)
    libc = ctypes.CDLL("libc.so.6", use_errno=True)
    libc.mmap.restype = ctypes.c_void_p
    libc.mmap.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                          ctypes.c_int, ctypes.c_long]
    libc.munmap.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    libc.madvise.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
    span = (nbytes + _HUGE - 1) // _HUGE * _HUGE + _HUGE
    raw = libc.mmap(None, span, 0x1 | 0x2, 0x02 | 0x20, -1, 0)  # RW, private anonymous
    if raw in (None, ctypes.c_void_p(-1).value):
        raise MemoryError(f"host_buffer: mmap of {span} bytes failed")
    base = (raw + _HUGE - 1) // _HUGE * _HUGE
    libc.madvise(ctypes.c_void_p(base), span - (base - raw), 14)  # MADV_HUGEPAGE (a hint)
    cudart = torch.cuda.cudart()
    rc = cudart.cudaHostRegister(base, nbytes, 0)
    if int(rc) != 0:
        libc.munmap(ctypes.c_void_p(raw), span)
        raise DsaError(5, "host_buffer", f"cudaHostRegister returned {rc}")
    arr = (ctypes.c_uint8 * nbytes).from_address(base)

    def release(raw=raw, span=span, base=base, libc=libc, cudart=cudart):
        cudart.cudaHostUnregister(base)
        libc.munmap(ctypes.c_void_p(raw), span)
    # the buffer object lives as long as any tensor on its memory
    weakref.finalize(arr, release)
    return torch.frombuffer(arr, dtype=torch.uint8).view(dtype).view(shape)


def check_wait_timeout(ws: torch.Tensor, timeout_ms: int = 50) -> None:
    """Run the library's bounded-wait check: a kernel waits on an mbarrier
    nothing arrives on for timeout_ms and latches DSA_ERR_DEVICE_TIMEOUT in
    the status word of `ws` (read it with get_device_status)."""
    _need(ws, "ws", torch.uint8)
    _check(_load().dsa_check_wait_timeout(_ptr(ws), ws.numel(), int(timeout_ms),
                                          _stream(ws.device)),
           "dsa_check_wait_timeout")


def static_device_status(device=None) -> int:
    """Synchronise the current stream of `device`, read and clear the status
    word that index_scores_topk_static's kernels latch."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None \
        else torch.device(device)
    v = ctypes.c_uint32(0)
    _check(_load().dsa_static_device_status(_stream(dev), ctypes.byref(v)),
           "dsa_static_device_status")
    return v.value


def get_device_status(ws: torch.Tensor) -> int:
    """Synchronise the current stream, read and clear the status word."""
    v = ctypes.c_uint32(0)
    _check(_load().dsa_get_device_status(_ptr(ws), _stream(ws.device),
                                         ctypes.byref(v)),
           "dsa_get_device_status")
    return v.value

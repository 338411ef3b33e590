"""Benchmark of the DSA hot path on GB300: one step = indexer + top-k
(chunked), sparse attention forward, and backward (delta, dQ/dK/dV) over one
synthetic sequence, at S = 131072 by default.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Prints one JSON line (rank 0).  With N > 1 (torchrun) every rank runs an
independent replica on its own GPU (weak scaling, no collective on the data
path); the value is all ranks' tokens over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import long_context_sparse_gb300 as dsa  # noqa: E402
from long_context_sparse_gb300 import synth  # noqa: E402

METRIC = "DSA fwd+bwd tokens/s at S=128k on 1 GB300; % of tensor/HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                  "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------ work model


def n_full(t):
    return (t + 1) // 4


def keys_of_row(wl, t):
    """|K(t)| for a full selection (random inputs select min(K_p, n_full))."""
    sel = min(wl.K_p, n_full(t))
    if wl.n_loc == 0:
        return 4 * sel
    # locals not already covered: with a full budget all 4*n_full tokens are
    # pooled and the locals add t+1 - 4*n_full(t); otherwise up to 3 (taken
    # as 3, the rare overlap with a selected pool ignored here)
    if sel == n_full(t):
        return t + 1
    return 4 * sel + min(3, t + 1)


def work_model(wl, kv=False):
    """Algorithmic work of one step (valid causal pairs / selected keys).
    kv: K and V are one tensor, so a key brings one row and one reduced
    gradient row."""
    S = wl.S
    t = np.arange(S, dtype=np.int64)
    nf = (t + 1) // 4
    idx_flops = float(nf.sum()) * wl.H_I * 2 * wl.D_I
    sel = np.minimum(nf, wl.K_p)
    if wl.n_loc == 0:
        keys = 4 * sel
    else:
        keys = np.where(sel == nf, t + 1, 4 * sel + np.minimum(3, t + 1))
    nk = float(keys.sum())
    row_bytes = (wl.d_qk if kv else wl.d_qk + wl.d_v) * 2
    return {
        "indexer_flops": idx_flops,
        "topk_bytes": float(np.where(nf > wl.K_p, nf, 0).sum()) * 4 + S * wl.K_p * 4,
        "fwd_flops": nk * wl.H * 2 * (wl.d_qk + wl.d_v),
        "fwd_gather_bytes": nk * row_bytes,
        "bwd_flops": nk * wl.H * 2 * (3 * wl.d_qk + 2 * wl.d_v),
        "bwd_gather_bytes": nk * row_bytes,
        "bwd_scatter_bytes": nk * (wl.d_qk if kv else wl.d_qk + wl.d_v) * 4,
        "keys": nk,
    }


def launches_per_step(wl, streaming=False, kv=False):
    """Kernel launches of one step, mirroring the library's host loop."""
    C = min(wl.chunk_q, wl.S)
    n = 1 if wl.S >= 4 else 0                   # pool
    if streaming:
        n += 1                                  # fused indexer + selection
    for t0 in range(0, wl.S if not streaming else 0, C):
        rows = min(C, wl.S - t0)
        if n_full(t0 + rows - 1) > wl.K_p:
            n += 1                              # indexer chunk
        n += 1                                  # top-k chunk
    n += 1                                      # attention forward
    if wl.backward:                             # delta, zero, main, finalize
        n += 4 if kv else 6                     # (one accumulator when K = V)
    return n


# ---------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = max(mx, float(f[1]))
            except ValueError:
                continue
            for nm, val in zip(names, f[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ CPU oracle


_W = {}


def _oracle_init(wl_dict, paths, scale):
    sys.path.insert(0, ROOT)
    import oracle
    wl = synth.Workload(**wl_dict)
    d = {k: np.load(v, mmap_mode="r") for k, v in paths.items()}
    kp = (oracle.pool_gated(np.asarray(d["k_idx"]), np.asarray(d["k_gate"]))
          if "k_gate" in d else oracle.pool(np.asarray(d["k_idx"])))
    _W.update(oracle=oracle, wl=wl, d=d, scale=scale, kp=kp,
              idx=np.empty((wl.S, wl.K_p), np.int32))


def _oracle_row(i):
    """The oracle, as it stands, on one query row of the workload:
    index + top-k, forward and (fwd+bwd workloads) backward.  Runs in a
    spawned worker process."""
    o, wl, d, scale = _W["oracle"], _W["wl"], _W["d"], _W["scale"]
    t = int(d["rows"][i])
    r = np.array([t], np.int64)
    sc = o.index_scores(np.asarray(d["q_idx"][i:i + 1]), _W["kp"],
                        np.asarray(d["w"][i:i + 1]), r, wl.S)
    _W["idx"][t] = o.topk(sc, r, wl.K_p)[0]
    q = np.asarray(d["q"][i:i + 1])
    o.attn_fwd(q, d["k"], d["v"], _W["idx"], wl.K_p, wl.n_loc, scale, r)
    if wl.backward:
        keys = o.key_set(t, wl.K_p, wl.n_loc, _W["idx"][t])
        o.attn_bwd(q, d["k"], d["v"], np.asarray(d["dO"][i:i + 1]), _W["idx"],
                   wl.K_p, wl.n_loc, scale, r, keys)
    return 1


def _np(t):
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def oracle_rows_data(wl, inputs, n_rows=256, seed=99, kv=False):
    """Host copies of what the oracle needs for `n_rows` late rows (last
    S/8, the steady-state cost) of the workload: the rows' queries, weights
    and upstream gradients, and the full K/V and indexer keys."""
    rng = np.random.default_rng(seed)
    lo = max(0, wl.S - max(1, wl.S // 8))
    rows = np.sort(rng.integers(lo, wl.S, n_rows)).astype(np.int64)
    rt = torch.from_numpy(rows).to(inputs["q"].device)
    out = {"rows": rows, "k_idx": _np(inputs["k_idx"]), "k": _np(inputs["k"]),
           "v": _np(inputs["v"])}
    if "k_gate" in inputs:
        out["k_gate"] = _np(inputs["k_gate"])
    if kv:
        out["v"] = out["k"]
    for k in ("q_idx", "w", "q") + (("dO",) if wl.backward else ()):
        out[k] = _np(inputs[k][rt])
    return out


def run_oracle_sample(wl, data, seconds: float, cores: int):
    """Run the oracle on rows of `data` with `cores` spawned workers until
    about `seconds` have passed; returns (tokens_per_s, rows, cores, wall)."""
    import dataclasses
    import tempfile
    tmp = tempfile.mkdtemp(prefix="dsa_oracle_")
    paths = {}
    for k, a in data.items():
        paths[k] = os.path.join(tmp, k + ".npy")
        np.save(paths[k], a)
    scale = 1.0 / math.sqrt(wl.d_qk)
    wl_dict = {f.name: getattr(wl, f.name) for f in dataclasses.fields(wl)}
    n = len(data["rows"])
    ctx = mp.get_context("spawn")
    done, nxt = 0, 0
    with ctx.Pool(cores, initializer=_oracle_init,
                  initargs=(wl_dict, paths, scale)) as pool:
        pool.map(_oracle_row, [0] * cores)       # warm the workers (untimed)
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            batch = [(nxt + j) % n for j in range(cores)]
            nxt += cores
            done += sum(pool.map(_oracle_row, batch))
        wall = time.perf_counter() - t0
    for p in paths.values():
        os.remove(p)
    os.rmdir(tmp)
    return done / wall, done, cores, wall


# ----------------------------------------------------------------- main


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# each attention kernel at full size, from an ncu capture of the bench
# command on glm_chunked_s128k.  An entry holds only while the kernel's
# sources hash to the value the capture was taken with; after any change the
# traffic is reported as null until it is captured again.
MEASURED_TRAFFIC = {
    "attn_bwd_tc": {"workload": "glm_chunked_s128k", "S": 131072,
                    "bytes": 343.04e9 + 228.90e9,
                    "sources": ("attn_bwd_tc.cu", "attn_common.cuh",
                                "dsa_common.cuh"),
                    "sha256_16": "cd3300051e284773"},
    "attn_fwd_tc": {"workload": "glm_chunked_s128k", "S": 131072,
                    "bytes": 117.12e9 + 9.58e9,
                    "sources": ("attn_fwd_tc.cu", "attn_common.cuh",
                                "dsa_common.cuh"),
                    "sha256_16": "daa8f08e9c9d686c"},
}


def measured_traffic(kernel, wl, variant=""):
    """Captured DRAM bytes per launch, or None if stale, another size or
    another variant of the kernel (the captures are of the default one)."""
    e = MEASURED_TRAFFIC.get(kernel)
    if e is None or variant or e["workload"] != wl.name or e["S"] != wl.S:
        return None
    return e["bytes"] if sources_hash(e["sources"]) == e["sha256_16"] else None


def sources_hash(sources):
    """First 16 hex digits of the sha256 of the kernel sources, in order."""
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, "long_context_sparse_gb300", "csrc", f),
                  "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def make_inputs(wl, seed, device, gated=False, attention=True):
    """The workload's inputs on `device`.  Up to S = 131072 they come from
    synth.indexer_inputs / attention_inputs; beyond, the same distributions
    are drawn in row blocks (no fp32 temporary of a whole tensor)."""
    if wl.S <= 131072:
        q_idx, k_idx, w = synth.indexer_inputs(wl, seed, device)
        x = {"q_idx": q_idx, "k_idx": k_idx, "w": w}
        if attention:
            q, k, v, dO = synth.attention_inputs(wl, seed, device)
            x.update(q=q, k=k, v=v, dO=dO)
    else:
        S, blk = wl.S, 8192
        x = {"q_idx": synth.normal_bf16_blocks((S, wl.H_I, wl.D_I), 1 / math.sqrt(wl.D_I),
                                               seed, device, 65536),
             "k_idx": synth.normal_bf16_blocks((S, wl.D_I), 1 / math.sqrt(wl.D_I),
                                               seed + 1, device, S),
             "w": torch.softmax(torch.randn((S, wl.H_I), generator=synth._gen(seed + 2, device),
                                            device=device), dim=-1).contiguous()}
        if attention:
            sq, sk, sv, sg = synth.attention_std(wl)
            x["q"] = synth.normal_bf16_blocks((S, wl.H, wl.d_qk), sq, seed + 3, device, blk)
            x["k"] = synth.normal_bf16_blocks((S, wl.d_qk), sk, seed + 4, device, S)
            x["v"] = synth.normal_bf16_blocks((S, wl.d_v), sv, seed + 5, device, S)
            if wl.backward:
                x["dO"] = synth.normal_bf16_blocks((S, wl.H, wl.d_v), sg, seed + 6, device, blk)
    if attention and not wl.backward:
        x.pop("dO", None)
    if gated:
        x["k_gate"] = synth.gate_inputs(wl, seed, device)
    return x


def reference_rows_data(wl, seed, n_rows=256, gated=False, kv=False):
    """Seeded synthetic data for the oracle-only arm, generated on the host
    for the sampled rows only (same shapes and distributions)."""
    import math as _m
    g = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    lo = max(0, wl.S - max(1, wl.S // 8))
    rows = np.sort(rng.integers(lo, wl.S, n_rows)).astype(np.int64)

    def nb(shape, std):
        return _np((torch.randn(shape, generator=g) * std).to(torch.bfloat16))

    out = {"rows": rows,
            "k_idx": nb((wl.S, wl.D_I), 1 / _m.sqrt(wl.D_I)),
            "k": nb((wl.S, wl.d_qk), 1 / _m.sqrt(wl.d_qk)),
            "v": nb((wl.S, wl.d_v), 1 / _m.sqrt(wl.d_v)),
            "q_idx": nb((n_rows, wl.H_I, wl.D_I), 1 / _m.sqrt(wl.D_I)),
            "w": torch.softmax(torch.randn((n_rows, wl.H_I), generator=g),
                               -1).numpy(),
            "q": nb((n_rows, wl.H, wl.d_qk), 1 / _m.sqrt(wl.d_qk)),
            "dO": nb((n_rows, wl.H, wl.d_v), 1.0)}
    if gated:
        out["k_gate"] = torch.randn(wl.S, generator=g).numpy()
    if kv:
        out["v"] = out["k"]
    return out


class Step:
    """Device buffers and workspaces for one replica of the hot path."""

    def __init__(self, wl, dev, inputs, kv=False, streaming=False):
        self.wl, self.dev, self.kv, self.streaming = wl, dev, kv, streaming
        self.cfg = dsa.config_for(wl)
        self.x = inputs
        S, H = wl.S, wl.H
        self.idx = torch.empty((S, wl.K_p), dtype=torch.int32, device=dev)
        self.o = torch.empty((S, H, wl.d_v), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((S, H), dtype=torch.float32, device=dev)
        self.ws_i = dsa.workspace(self.cfg, dsa.WS_INDEX, dev)
        self.ws_f = dsa.workspace(self.cfg, dsa.WS_FWD, dev)
        if wl.backward:
            self.dq = torch.empty((S, H, wl.d_qk), dtype=torch.bfloat16, device=dev)
            self.dk = torch.empty((S, wl.d_qk), dtype=torch.bfloat16, device=dev)
            self.dv = torch.empty((S, wl.d_v), dtype=torch.bfloat16, device=dev)
            self.ws_b = dsa.workspace(self.cfg, dsa.WS_BWD, dev)
        if streaming:
            self.ws_i = dsa.workspace(self.cfg, dsa.WS_STREAM, dev)

    def run(self, ev=None):
        x, c = self.x, self.cfg
        if ev is not None:
            ev[0].record()
        if self.streaming:  # selection fused into the indexer, no scores stored
            dsa.index_topk_streaming(c, x["q_idx"], x["k_idx"], x["w"], 0,
                                     self.wl.S, k_gate=x.get("k_gate"),
                                     out=self.idx, ws=self.ws_i)
        elif "k_gate" in x:  # gated pools: the range entry over every query
            dsa.index_scores_topk_range(c, x["q_idx"], x["k_idx"], x["w"], 0,
                                        self.wl.S, k_gate=x["k_gate"],
                                        out=self.idx, ws=self.ws_i)
        else:
            dsa.index_scores_topk(c, x["q_idx"], x["k_idx"], x["w"], out=self.idx,
                                  ws=self.ws_i)
        if ev is not None:
            ev[1].record()
        if self.kv:  # one tensor as keys and values
            dsa.sparse_attn_fwd_kv(c, x["q"], x["k"], self.idx, o=self.o,
                                   lse=self.lse, ws=self.ws_f)
        else:
            dsa.sparse_attn_fwd(c, x["q"], x["k"], x["v"], self.idx, o=self.o,
                                lse=self.lse, ws=self.ws_f)
        if ev is not None:
            ev[2].record()
        if self.wl.backward and self.kv:
            dsa.sparse_attn_bwd_kv(c, x["q"], x["k"], self.o, self.lse, x["dO"],
                                   self.idx, dq=self.dq, dkv=self.dk, ws=self.ws_b)
        elif self.wl.backward:
            dsa.sparse_attn_bwd(c, x["q"], x["k"], x["v"], self.o, self.lse,
                                x["dO"], self.idx, dq=self.dq, dk=self.dk,
                                dv=self.dv, ws=self.ws_b)
        if ev is not None:
            ev[3].record()

    def outputs(self):
        out = [self.idx, self.o, self.lse]
        if self.wl.backward:
            out += [self.dq, self.dk] + ([] if self.kv else [self.dv])
        return out

    def status(self):
        ws = (self.ws_i, self.ws_f) + ((self.ws_b,) if self.wl.backward else ())
        return [dsa.get_device_status(w) for w in ws]


def index_only(args, wl, dev, seed, base_cfg, rank, dist_on):
    """Time dsa_index_scores_topk alone (pool + chunked indexer + top-k):
    inputs of the indexer only, so the whole sequence's selection fits in a
    small device footprint (about 1.4 GB at S = 131072)."""
    cfg = dsa.config_for(wl)
    x = make_inputs(wl, seed, dev, attention=False)
    q_idx, k_idx, w = x["q_idx"], x["k_idx"], x["w"]
    idx = torch.empty((wl.S, wl.K_p), dtype=torch.int32, device=dev)
    ws = dsa.workspace(cfg, dsa.WS_INDEX, dev)
    for _ in range(args.warmup):
        dsa.index_scores_topk(cfg, q_idx, k_idx, w, out=idx, ws=ws)
    torch.cuda.synchronize()
    barrier(dist_on)
    e0, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
    e0.record()
    for _ in range(args.steps):
        dsa.index_scores_topk(cfg, q_idx, k_idx, w, out=idx, ws=ws)
    e1.record()
    torch.cuda.synchronize()
    if dsa.get_device_status(ws):
        raise SystemExit("device status after the indexer calls")
    ms = e0.elapsed_time(e1) / args.steps
    wm = work_model(wl)
    if rank == 0:
        print(json.dumps({
            "metric": "dsa_index_scores_topk ms per call", "value": ms, "unit": "ms",
            "higher_is_better": False, "steps": args.steps, "warmup": args.warmup,
            "config": dict(base_cfg, passes="index"),
            "indexer_tflops_whole_call": wm["indexer_flops"] / (ms / 1e3) / 1e12,
            "memory": {
                "workspace_bytes": dsa.workspace_size(cfg, dsa.WS_INDEX),
                "score_chunk_bytes": min(wl.chunk_q, wl.S) * ((wl.P + 127) // 128 * 128) * 4,
                "unchunked_scores_bytes": wl.S * wl.P * 4,
                "unchunked_per_head_scores_bytes": wl.S * wl.P * wl.H_I * 4,
                "peak_allocated_bytes": torch.cuda.max_memory_allocated(dev),
                "note": "peak_allocated_bytes: torch.cuda.max_memory_allocated over "
                        "the calls (indexer inputs, selection, workspace); the "
                        "unchunked figures are what scoring every query at once "
                        "would hold (one fp32 per (query, pool), and per head)"}}),
            flush=True)
    if dist_on:
        torch.distributed.destroy_process_group()


def settle_host_link(h2d, d2h, limit_s=180.0, target_gbs=120.0):
    """Copy rates of the host step's own largest buffers, polled until two
    polls in a row reach target_gbs both ways or limit_s has passed.

    On the GPU host, right after another process has released a large
    amount of host memory (the GPU test suite does), copies between the
    device and page-locked host memory can run at 13-18 GB/s instead of
    ~210 for minutes, for multi-GB buffers while a 256 MiB buffer still
    copies at full speed.  So the probe copies the step's largest input
    (h2d = (host, device)) and output (d2h = (device, host)) tensors, each
    twice back to back, keeping the second rate (the first copy after an
    idle spell is slow on its own).  The host step is timed once the link
    is back (or the limit is reached); the rates are reported with it."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def rate(src, dst):
        for _ in range(2):
            e0.record()
            dst.copy_(src, non_blocking=True)
            e1.record()
            torch.cuda.synchronize()
        return src.numel() * src.element_size() / 1e9 / (e0.elapsed_time(e1) / 1e3)

    def poll():
        return rate(*h2d), rate(*d2h)

    t0 = time.time()
    first = last = poll()
    ok = 1 if min(last) >= target_gbs else 0
    while ok < 2 and time.time() - t0 < limit_s:
        last = poll()
        ok = ok + 1 if min(last) >= target_gbs else 0
    return {"h2d_gbs_first_poll": round(first[0], 1), "d2h_gbs_first_poll": round(first[1], 1),
            "h2d_gbs_before_timing": round(last[0], 1),
            "d2h_gbs_before_timing": round(last[1], 1),
            "settle_wait_s": round(time.time() - t0, 1), "target_gbs": target_gbs,
            "probe_bytes": [h2d[0].numel() * h2d[0].element_size(),
                            d2h[0].numel() * d2h[0].element_size()]}


def buffer_copy_gbs(hb, scratch):
    """min(host->device, device->host) GB/s of a whole host buffer, copied
    through a device scratch in scratch-sized pieces (one piece first as a
    warm-up: the first copy after an idle spell is slow on its own)."""
    flat = hb.view(-1).view(torch.uint8)
    n, m = flat.numel(), scratch.numel()
    scratch[:min(n, m)].copy_(flat[:min(n, m)], non_blocking=True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    rates = []
    for direction in ("h2d", "d2h"):
        e0.record()
        for i in range(0, n, m):
            j = min(n, i + m)
            if direction == "h2d":
                scratch[:j - i].copy_(flat[i:j], non_blocking=True)
            else:
                flat[i:j].copy_(scratch[:j - i], non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        rates.append(n / 1e9 / (e0.elapsed_time(e1) / 1e3))
    return min(rates)


def checked_host_buffer(shape, dtype, scratch, log, min_gbs=150.0, tries=4):
    """dsa.host_buffer whose copies run at full rate.  On the GPU host some
    freshly allocated page-locked buffers copy at 15-50 GB/s instead of
    ~200 GB/s, and stay that slow for minutes (measured with both
    cudaHostAlloc and 2 MiB-page buffers, most often right after another
    process released a lot of memory; a buffer allocated next to a slow
    one is usually fine; the same host also slows every copy for seconds
    at a time, which no choice of buffer avoids).  A buffer of 256 MiB or more is timed both ways once; below
    min_gbs it is replaced (the slow one is held until a good one is found,
    so that the host does not hand the same pages back), at most tries - 1
    times.  log gets (replacements, rate) per checked buffer."""
    n = 1
    for x in shape:
        n *= int(x)
    if n * torch.empty((), dtype=dtype).element_size() < (256 << 20):
        log.append(None)
        return dsa.host_buffer(shape, dtype)
    held = []
    for attempt in range(tries):
        hb = dsa.host_buffer(shape, dtype)
        r = buffer_copy_gbs(hb, scratch)
        if r >= min_gbs or attempt == tries - 1:
            log.append((attempt, round(r, 1)))
            del held
            return hb
        held.append(hb)


def host_link_probe(dev, seconds, rank):
    """Host<->device copy rates over time, about one sample a second, for 2
    GiB page-locked buffers: cudaHostAlloc (torch's pinned memory),
    dsa.host_buffer (2 MiB pages, cudaHostRegister), and a cudaHostAlloc
    buffer that the CPU rewrites before each sample.  Each sample times one
    copy each way per buffer (host to device first, so the first two
    buffers are read after the previous sample's device-to-host copy wrote
    them), after a second of idle.  Prints one JSON line."""
    n = 2 << 30
    d = torch.empty(n, dtype=torch.uint8, device=dev)
    bufs = {"pinned": torch.empty(n, dtype=torch.uint8, pin_memory=True),
            "host_buffer": dsa.host_buffer((n,), torch.uint8),
            "pinned_cpu_written": torch.empty(n, dtype=torch.uint8, pin_memory=True)}
    for b in bufs.values():
        b.fill_(1)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    samples = []
    t0 = time.time()
    while time.time() - t0 < seconds:
        row = {"t_s": round(time.time() - t0, 1)}
        for name, hb in bufs.items():
            if name == "pinned_cpu_written":
                hb.fill_(len(samples) & 255)  # rewritten by the CPU before each sample
            for direction in ("h2d", "d2h"):
                e0.record()
                if direction == "h2d":
                    d.copy_(hb, non_blocking=True)
                else:
                    hb.copy_(d, non_blocking=True)
                e1.record()
                torch.cuda.synchronize()
                row[f"{name}_{direction}_gbs"] = round(n / 1e9 / (e0.elapsed_time(e1) / 1e3), 1)
        samples.append(row)
        time.sleep(1.0)
    if rank == 0:
        keys = [k for k in samples[0] if k != "t_s"]
        print(json.dumps({"metric": "host<->device copy GB/s over time, 2 GiB buffers",
                          "unit": "GB/s", "buffer_bytes": n,
                          "median": {k: statistics.median(r[k] for r in samples) for k in keys},
                          "min": {k: min(r[k] for r in samples) for k in keys},
                          "samples": samples}), flush=True)


def barrier(dist_on):
    if dist_on:
        torch.distributed.barrier()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="glm_chunked_s128k",
                    choices=sorted(synth.WORKLOADS))
    ap.add_argument("--seq-len", type=int, default=0,
                    help="override S (smaller runs for profiling)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=8,
                    help="query ranges of the host-buffer step (1..64)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--pool", default="mean", choices=["mean", "gated"],
                    help="pool keys by their mean (default) or by gate scores")
    ap.add_argument("--select", default="chunked", choices=["chunked", "streaming"],
                    help="top-k over stored score chunks (default) or fused "
                         "into the indexer")
    ap.add_argument("--kv", default="separate", choices=["separate", "aliased"],
                    help="K and V as two tensors (default) or one (K = V)")
    ap.add_argument("--passes", default="step", choices=["step", "index", "host_link"],
                    help="the whole step (default), or only the chunked indexer "
                         "+ top-k (a small device footprint for counter captures; "
                         "prints its own line, not the step metric), or the host "
                         "link's copy rates over time (its own line)")
    ap.add_argument("--probe-seconds", type=float, default=60.0,
                    help="--passes host_link: how long to sample")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist_on = world > 1
    wl = synth.WORKLOADS[args.workload]
    if args.seq_len:
        wl = synth.scaled(wl, args.seq_len)
    kv = args.kv == "aliased"
    wm = work_model(wl, kv)
    base_cfg = {"workload": wl.name, "S": wl.S, "indexer": f"{wl.H_I}x{wl.D_I}",
                "topk_pools": wl.K_p, "keys": wl.keys_per_query,
                "heads": wl.H, "d_qk": wl.d_qk, "d_v": wl.d_v,
                "chunk_q": wl.chunk_q, "passes": "fwd+bwd" if wl.backward else "fwd",
                "pool": args.pool, "kv": args.kv, "select": args.select,
                "replica_per_gpu": True,
                "l2": "inputs larger than L2 (q 8 GiB, k/v 256 MiB at S=131072)"
                      if wl.S >= 65536 else "working set may fit L2"}

    if args.impl == "reference":
        if rank != 0:
            return
        if args.warmup < 0 or args.steps < 1:
            raise SystemExit("bad steps")
        cores = max(1, os.cpu_count() or 1)
        data = reference_rows_data(wl, 20262, gated=args.pool == "gated", kv=kv)
        per_step = max(2.0, 120.0 / max(1, args.steps + args.warmup))
        vals = []
        for i in range(args.warmup + args.steps):
            v, rows, used, wall = run_oracle_sample(wl, data, per_step, cores)
            if i >= args.warmup:
                vals.append((v, rows, wall))
        value = statistics.median([v for v, _, _ in vals])
        rows_tot = sum(r for _, r, _ in vals)
        line = {"impl": "reference", "metric": METRIC, "value": value,
                "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup,
                "ms_per_step": 1000.0 * sum(w for _, _, w in vals) / len(vals),
                "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": base_cfg,
                "cpu_baseline": {"value": value, "unit": "tokens/s",
                                 "cores": cores, "kind": "oracle",
                                 "sample": f"{rows_tot} late query rows of the "
                                 "workload (index+top-k+fwd+bwd per row, fp64),"
                                 f" about {per_step:.0f} s per step"},
                "e2e": {"value": value, "unit": "tokens/s",
                        "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    if dist_on:
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    seed = 20262 + rank
    if args.passes == "index":
        return index_only(args, wl, dev, seed, base_cfg, rank, dist_on)
    if args.passes == "host_link":
        return host_link_probe(dev, args.probe_seconds, rank)
    inputs = make_inputs(wl, seed, dev, gated=args.pool == "gated")
    step = Step(wl, dev, inputs, kv=kv, streaming=args.select == "streaming")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
           for _ in range(args.steps)]
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    st = step.status()
    if any(st):
        raise SystemExit(f"device status after warm-up: {st}")

    barrier(dist_on)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        start.record()
        for i in range(args.steps):
            step.run(evs[i])
        stop.record()
        torch.cuda.synchronize()
    barrier(dist_on)
    ms = start.elapsed_time(stop) / args.steps
    peak_alloc = torch.cuda.max_memory_allocated(dev)
    if any(step.status()):
        raise SystemExit(f"device status after timed steps: {step.status()}")
    t_idx = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    t_fwd = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    t_bwd = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)

    ms_max = ms
    if dist_on:
        tt = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        ms_max = float(tt.item())
    value = world * wl.S / (ms_max / 1000.0)

    # ---- e2e through the public API with pinned host buffers (up to
    # S = 131072: beyond, the pinned copies of q and o alone would take a
    # large part of the host's memory)
    e2e = None
    if wl.S > 131072 and not args.no_e2e:
        e2e = {"value": None, "unit": "tokens/s", "h2d_bytes_per_step": None,
               "d2h_bytes_per_step": None,
               "skipped": "host-buffer step not run above S = 131072 (q and o "
                          "alone would pin %.0f GB of host memory)"
                          % (2 * wl.S * wl.H * wl.d_qk * 2 / 1e9)}
    if not args.no_e2e and e2e is None:
        # page-locked host buffers on 2 MiB pages (dsa.host_buffer), each
        # checked for full-rate copies and replaced if the host gave it
        # memory that copies crawl from (see checked_host_buffer)
        scratch = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        checks = []
        host_in = {k: checked_host_buffer(t.shape, t.dtype, scratch, checks)
                   for k, t in inputs.items()}
        # the inputs are written into the host buffers by the CPU, as a data
        # loader would (on this host, cudaHostAlloc memory last written by a
        # device-to-host copy was measured copying back to the device at
        # 8-20 GB/s at times; rewritten by the CPU, at 96-170 GB/s in the
        # same run)
        for k in host_in:
            host_in[k].copy_(inputs[k].cpu())
        host_out = [checked_host_buffer(t.shape, t.dtype, scratch, checks)
                    for t in step.outputs()]
        del scratch
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out)
        e_start = torch.cuda.Event(enable_timing=True)
        e_stop = torch.cuda.Event(enable_timing=True)
        n_e2e = max(10, args.steps)
        # dsa_step_host: query ranges whose copies overlap the kernels (the
        # fused streaming selection has no host-step form: serial copies)
        pipelined = args.select == "chunked"
        if pipelined:
            names = ["topk_idx", "o", "lse"] + (
                ["dq", "dk"] + ([] if kv else ["dv"]) if wl.backward else [])
            host_step = dict(host_in, **dict(zip(names, host_out)))
            dev_step = dict(inputs, **dict(zip(names, step.outputs())))
            if kv:  # one tensor as keys and values: v is not an input
                host_step.pop("v", None)
                dev_step.pop("v", None)
            if not wl.backward:  # forward only: no upstream gradient
                host_step.pop("dO", None)
                dev_step.pop("dO", None)
            h2d = sum(t.numel() * t.element_size() for k, t in host_step.items()
                      if k not in names)
            ws_step = dsa.workspace(step.cfg, dsa.WS_STEP, dev)
            copy_streams = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))

            def one():
                dsa.step_host(step.cfg, host_step, dev_step, args.e2e_chunks,
                              ws=ws_step, copy_streams=copy_streams)
        else:
            def one():
                for k in host_in:
                    inputs[k].copy_(host_in[k], non_blocking=True)
                step.run()
                for h, d in zip(host_out, step.outputs()):
                    h.copy_(d, non_blocking=True)

        # the kernels run on a stream of their own, as in a training loop;
        # the events are recorded on it
        e2e_stream = torch.cuda.Stream(dev)
        big_in = max(host_in, key=lambda k: host_in[k].numel() * host_in[k].element_size())
        big_out = max(range(len(host_out)),
                      key=lambda i: host_out[i].numel() * host_out[i].element_size())
        probe = ((host_in[big_in], inputs[big_in]),
                 (step.outputs()[big_out], host_out[big_out]))
        link = settle_host_link(*probe)
        with torch.cuda.stream(e2e_stream):
            one()
            torch.cuda.synchronize()
            barrier(dist_on)
            e_start.record(e2e_stream)
            marks = []
            for _ in range(n_e2e):
                one()
                marks.append(torch.cuda.Event(enable_timing=True))
                marks[-1].record(e2e_stream)
            e_stop.record(e2e_stream)
        torch.cuda.synchronize()
        step_ms = [round(a.elapsed_time(b), 1) for a, b in zip([e_start] + marks[:-1], marks)]
        after = settle_host_link(*probe, limit_s=0.0)
        link["h2d_gbs_after_timing"] = after["h2d_gbs_first_poll"]
        link["d2h_gbs_after_timing"] = after["d2h_gbs_first_poll"]
        e_ms = e_start.elapsed_time(e_stop) / n_e2e
        if dist_on:
            tt = torch.tensor([e_ms], device=dev)
            torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
            e_ms = float(tt.item())
        e2e = {"value": world * wl.S / (e_ms / 1000.0), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms, "step_ms": step_ms, "host_link": link,
               "host_buffers": {
                   "checked": sum(1 for c in checks if c is not None),
                   "replaced": sum(c[0] for c in checks if c is not None),
                   "min_gbs_kept": min((c[1] for c in checks if c is not None),
                                       default=None)},
               "path": (f"dsa_step_host, {args.e2e_chunks} query ranges, "
                        "copies overlapped on two side streams, host buffers "
                        "page-locked on 2 MiB pages") if pipelined
                       else "serial copies around the device calls"}
        del host_in, host_out

    if rank != 0:
        if dist_on:
            torch.distributed.destroy_process_group()
        return

    pk, pk_kind = peaks()
    variant = ",".join(x for x in (
        "gated" if args.pool == "gated" else "", "kv" if kv else "") if x)
    parts = {"index_topk_ms": t_idx, "attn_fwd_ms": t_fwd, "attn_bwd_ms": t_bwd}
    # dominant call and its roofline (algorithmic bytes / flops per launch)
    dom = max(parts, key=parts.get)
    if dom == "index_topk_ms":
        achieved = wm["indexer_flops"] / (t_idx / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved,
                "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s",
                "kernel": "dsa_index_scores_topk (pool + indexer + top-k)"}
    elif dom == "attn_fwd_ms":
        achieved = wm["fwd_gather_bytes"] / (t_fwd / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
                "unit": "GB/s",
                "kernel": "attn_fwd_tc_kernel (gathered K/V bytes)",
                "traffic": measured_traffic("attn_fwd_tc", wl, variant)}
    else:
        achieved = wm["bwd_gather_bytes"] / (t_bwd / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
                "unit": "GB/s",
                "kernel": "attn_bwd_tc_kernel, timed as the whole "
                          "dsa_sparse_attn_bwd call (delta + zero + main + "
                          "finalize launches; gathered K/V bytes)",
                "traffic": measured_traffic("attn_bwd_tc", wl, variant),
                "achieved_with_scatter": (wm["bwd_gather_bytes"] +
                                          wm["bwd_scatter_bytes"]) /
                                         (t_bwd / 1e3) / 1e9}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof.setdefault("traffic", None)
    roof["peak_source"] = pk_kind
    aux = {
        "indexer_tflops": wm["indexer_flops"] / (t_idx / 1e3) / 1e12,
        "fwd_gather_gbs": wm["fwd_gather_bytes"] / (t_fwd / 1e3) / 1e9,
        "fwd_tflops": wm["fwd_flops"] / (t_fwd / 1e3) / 1e12,
    }
    if wl.backward:
        aux["bwd_gather_gbs"] = wm["bwd_gather_bytes"] / (t_bwd / 1e3) / 1e9
        aux["bwd_tflops"] = wm["bwd_flops"] / (t_bwd / 1e3) / 1e12
    # the forward against the ceilings it actually faces: its flops at the
    # sustained tensor peak, and the DRAM bytes it moves (most gathered rows
    # hit L2, so the gathered bytes at HBM speed are not a ceiling)
    fwd_flops_ms = wm["fwd_flops"] / (pk["bf16_tflops_sustained"] * 1e12) * 1e3
    fwd_dram = measured_traffic("attn_fwd_tc", wl, variant)
    fwd_dram_ms = None if fwd_dram is None else fwd_dram / (pk["hbm_gbs"] * 1e9) * 1e3
    fwd_bound = max(fwd_flops_ms, fwd_dram_ms or 0.0)
    aux["fwd_roofline"] = {
        "flops_at_sustained_peak_ms": fwd_flops_ms,
        "dram_bytes_at_hbm_ms": fwd_dram_ms,
        "bound_ms": fwd_bound, "measured_ms": t_fwd, "frac": fwd_bound / t_fwd,
        "note": "max(flops / sustained bf16 peak, measured DRAM bytes / HBM "
                "peak); the DRAM term is null when no capture matches the "
                "kernel's sources"}

    mem = {"workspace_bytes": {
               "index": dsa.workspace_size(step.cfg, dsa.WS_STREAM if
                                           args.select == "streaming" else dsa.WS_INDEX),
               "fwd": dsa.workspace_size(step.cfg, dsa.WS_FWD),
               "bwd": dsa.workspace_size(step.cfg, dsa.WS_BWD) if wl.backward else 0},
           "score_chunk_bytes": (0 if args.select == "streaming" else
                                 min(wl.chunk_q, wl.S) * ((wl.P + 127) // 128 * 128) * 4),
           "unchunked_scores_bytes": wl.S * wl.P * 4,
           "peak_allocated_bytes": peak_alloc,
           "note": "peak_allocated_bytes: torch.cuda.max_memory_allocated over "
                   "the device-resident steps (inputs, outputs, workspaces); "
                   "unchunked_scores_bytes: one fp32 score per (query, pool), "
                   "what scoring every query at once would hold"}
    line = {"metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": base_cfg,
            "parallelism": f"replicas{world}",
            "breakdown_ms": parts, "rates": aux,
            "roofline": roof,
            "memory": mem,
            "clocks": clk.summary(),
            "gpu_launches": launches_per_step(
                wl, args.select == "streaming", kv) * args.steps,
            "e2e": e2e}

    if not args.no_cpu:
        cores = max(1, os.cpu_count() or 1)
        v, rows, used, wall = run_oracle_sample(
            wl, oracle_rows_data(wl, inputs, kv=kv), args.cpu_seconds, cores)
        line["cpu_baseline"] = {
            "value": v, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": f"{rows} late query rows (last S/8) of the same workload, "
                      "each through index+top-k+fwd" + ("+bwd" if wl.backward else "") +
                      f" in fp64, {wall:.1f} s wall"}
    print(json.dumps(line), flush=True)
    if dist_on:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

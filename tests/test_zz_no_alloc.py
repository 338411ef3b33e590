"""The allocation-free indexer entry point (dsa_index_scores_topk_static).

It serves callers that cannot allocate device memory (a plugin whose host
application owns all device memory, a service with a fixed footprint): its
scratch is a fixed array inside the library.  This file is collected last so
that a run stopping at the first failure has run every other test first; it
also passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

import long_context_sparse_gb300 as dsa
from long_context_sparse_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _call(lib, cfg, q_idx, k_idx, w, out):
    cc = cfg.c()
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    return lib.dsa_index_scores_topk_static(
        ctypes.byref(cc), ctypes.c_void_p(q_idx.data_ptr()),
        ctypes.c_void_p(k_idx.data_ptr()), ctypes.c_void_p(w.data_ptr()),
        ctypes.c_void_p(out.data_ptr()), stream)


def test_static_scratch_matches_workspace_entry_point_twice():
    lib = dsa._load()
    # two problems, each called through the C ABI twice in a row: the shared
    # array keeps the previous call's contents, results must not depend on it
    for S, seed in ((4099, 3), (9000, 4)):
        wl = synth.scaled(synth.WORKLOADS["glm_s16k"], S)
        cfg = dsa.config_for(wl)
        q_idx, k_idx, w = (x.to(DEV) for x in synth.indexer_inputs(wl, seed, "cpu"))
        ref = dsa.index_scores_topk(cfg, q_idx, k_idx, w)   # with a workspace
        for _ in range(2):
            out = torch.full_like(ref, -7)
            assert _call(lib, cfg, q_idx, k_idx, w, out) == 0
            torch.cuda.synchronize()
            assert torch.equal(out, ref)    # indices: bit-exact
            st = ctypes.c_uint32(99)        # nothing latched by the kernels
            assert lib.dsa_static_device_status(
                ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream),
                ctypes.byref(st)) == 0
            assert st.value == 0


def test_static_scratch_rejects_problems_beyond_its_size():
    lib = dsa._load()
    wl = synth.scaled(synth.WORKLOADS["glm_s16k"], 1 << 20)
    cfg = dsa.config_for(wl)
    assert dsa.workspace_size(cfg, dsa.WS_INDEX) > (32 << 20)
    dummy = torch.empty(16, dtype=torch.uint8, device=DEV)
    assert _call(lib, cfg, dummy, dummy, dummy, dummy) == 3  # too small
